"""CPU oracle of the Layer-Aware Prefetch Planner -- TEST INFRASTRUCTURE.

Only ``tests/`` and the benchmark's CPU legs may import this module; the
library's planner (``spx_plan_prefetch`` in libspx) is written separately and
shares no code with it.

Source (page title + section): ai.info summary "Specter: Fast MoE Inference
via Quantization-Enabled Multi-Step Speculative Offloading", Key
Contributions 3 (the Expert Lookahead Buffer's layer-indexed activation
counters feed a Layer-Aware Prefetch Planner that organises transfers into
Cold Start, Prefetch Overlap and Final Cleanup phases with adaptively sized
draft chunks) and "Methodology in Plain English" (snapshots of the counters
drive host-to-device prefetches; draft work is cut into chunks sized so that
computation roughly matches transfer time on a parallel stream); richland.au
"Specter previews expert routing with an INT4 copy of the model itself",
"What shipped" (a compact prefetch plan formed at chunk boundaries).

The pages name the phases and the sizing goal only; the steps below are the
plainest reading that the rest supports, one call per chunk boundary:

  phase        cold start before any draft step of the cycle, prefetch
               overlap between steps, final cleanup after the last one;
  demand       the experts a layer's counters have seen (count > 0) that are
               not cached yet, most counted first, ties to the lower expert;
  order        layers ascending, the order the verify pass needs them in;
  capacity     a layer caches at most `capacity` experts: a demanded expert
               takes the place of a cached one the counters have not seen
               (lowest index first); when every cached expert is demanded,
               the layer's remaining demand waits for the verify pass;
  next chunk   the draft steps whose compute covers the loads just issued,
               ceil(loads * copy_us / step_us), at least min_chunk and at
               most the steps left (cold start: min_chunk; final cleanup: 0).

Parity status: pinned by hand-made counter tables in ``tests/test_plan.py``
(phase boundaries, order, capacity, chunk sizes, a whole cycle).
"""
from __future__ import annotations

import math

COLD_START, PREFETCH_OVERLAP, FINAL_CLEANUP = 0, 1, 2
EVICT, LOAD = 0, 1


def plan_prefetch(elb, steps_done, cached, K, capacity, step_us, copy_us, min_chunk=1):
    """One planning call at a chunk boundary.

    elb: [L][E] counts after `steps_done` draft steps; cached: [L][E] 0/1,
    updated in place.  Returns (phase, actions, next_chunk) with actions a
    list of (layer, expert, LOAD | EVICT) in issue order."""
    L = len(elb)
    E = len(elb[0]) if L else 0
    if steps_done == 0:
        phase = COLD_START
    elif steps_done < K:
        phase = PREFETCH_OVERLAP
    else:
        phase = FINAL_CLEANUP
    actions = []
    for layer in range(L):
        counts = elb[layer]
        demand = [e for e in range(E) if counts[e] > 0 and not cached[layer][e]]
        demand.sort(key=lambda e: (-int(counts[e]), e))
        for e in demand:
            if sum(1 for v in range(E) if cached[layer][v]) >= capacity:
                victims = [v for v in range(E) if cached[layer][v] and counts[v] == 0]
                if not victims:
                    break
                cached[layer][victims[0]] = 0
                actions.append((layer, victims[0], EVICT))
            cached[layer][e] = 1
            actions.append((layer, e, LOAD))
    loads = sum(1 for a in actions if a[2] == LOAD)
    if phase == FINAL_CLEANUP:
        next_chunk = 0
    else:
        want = math.ceil(loads * copy_us / step_us) if loads else min_chunk
        next_chunk = min(max(want, min_chunk), K - steps_done)
    return phase, actions, next_chunk
