"""The Layer-Aware Prefetch Planner on CPU (host code, no GPU): the oracle
pinned by hand-made counter tables (phase boundaries, load order, capacity,
chunk sizes, a whole cycle), and the library's spx_plan_prefetch equal to the
oracle on seeded cycles of drawn draft routings."""
import numpy as np
import pytest

from oracle import planner as P


def _cached(L, E, on=()):
    c = [[0] * E for _ in range(L)]
    for l, e in on:
        c[l][e] = 1
    return c


def test_cold_start_plans_nothing_and_runs_the_shortest_chunk():
    elb = [[0] * 8 for _ in range(3)]
    phase, acts, chunk = P.plan_prefetch(elb, 0, _cached(3, 8), K=16, capacity=8, step_us=100, copy_us=40,
                                         min_chunk=1)
    assert (phase, acts, chunk) == (P.COLD_START, [], 1)


def test_overlap_loads_layer_by_layer_most_counted_first():
    elb = [[0, 2, 0, 5, 0, 0, 2, 0], [1, 0, 0, 0, 0, 0, 0, 0], [0] * 8]
    cached = _cached(3, 8, on=[(1, 0)])
    phase, acts, chunk = P.plan_prefetch(elb, 1, cached, K=16, capacity=8, step_us=100, copy_us=40)
    assert phase == P.PREFETCH_OVERLAP
    # layer 0: expert 3 (count 5), then experts 1 and 6 (count 2, lower index first); layer 1's expert 0 is cached
    assert acts == [(0, 3, P.LOAD), (0, 1, P.LOAD), (0, 6, P.LOAD)]
    assert chunk == 2  # ceil(3 loads * 40 us / 100 us per step)
    assert cached[0] == [0, 1, 0, 1, 0, 0, 1, 0]
    # the same snapshot again: everything it demands is cached
    assert P.plan_prefetch(elb, 3, cached, K=16, capacity=8, step_us=100, copy_us=40) == (P.PREFETCH_OVERLAP, [], 1)


def test_capacity_evicts_an_unseen_expert_then_leaves_the_rest_to_verify():
    cached = _cached(1, 6, on=[(0, 0), (0, 1)])
    elb = [[0, 3, 0, 1, 0, 4]]
    phase, acts, chunk = P.plan_prefetch(elb, 4, cached, K=8, capacity=2, step_us=50, copy_us=500)
    assert acts == [(0, 0, P.EVICT), (0, 5, P.LOAD)]  # expert 3 waits: both cached experts are counted
    assert cached == [[0, 1, 0, 0, 0, 1]]
    assert chunk == 4  # ceil(1 * 500 / 50) = 10, clamped to the 4 steps left


def test_final_cleanup_loads_the_rest_and_ends_drafting():
    elb = [[0, 1], [2, 0]]
    phase, acts, chunk = P.plan_prefetch(elb, 16, _cached(2, 2), K=16, capacity=2, step_us=10, copy_us=10)
    assert (phase, chunk) == (P.FINAL_CLEANUP, 0)
    assert acts == [(0, 1, P.LOAD), (1, 0, P.LOAD)]


def _draw_cycle(rng, L, E, k, K):
    """Per (step, layer) the k experts of one draft token, Zipf-skewed."""
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    perm = [rng.permutation(E) for _ in range(L)]
    return [[perm[l][rng.choice(E, size=k, replace=False, p=p)] for l in range(L)] for _ in range(K)]


def _run_cycle(plan, L, E, k, K, picks):
    """Drive one cycle: run chunks of draft steps, snapshot, plan.  Returns the
    list of (steps_done, phase, actions, chunk) and the final cached table."""
    elb = np.zeros((L, E), np.uint32)
    cached = np.zeros((L, E), np.uint8)
    done, log = 0, []
    while True:
        phase, acts, chunk = plan(elb.copy(), done, cached)
        log.append((done, phase, [tuple(int(v) for v in a) for a in acts], chunk))
        if phase == P.FINAL_CLEANUP:
            return log, cached
        for st in range(done, done + chunk):
            for l in range(L):
                elb[l, picks[st][l]] += 1
        done += chunk


@pytest.mark.parametrize("seed,L,E,k,K,cap,copy_us", [(0, 26, 64, 6, 16, 64, 38.0), (1, 26, 64, 6, 16, 16, 38.0),
                                                      (2, 24, 60, 4, 8, 20, 38.0), (3, 32, 16, 2, 16, 4, 350.0),
                                                      (4, 4, 8, 2, 5, 3, 0.0)])
def test_oracle_cycle_invariants(seed, L, E, k, K, cap, copy_us):
    rng = np.random.default_rng(seed)
    picks = _draw_cycle(rng, L, E, k, K)
    step_us = 26 * 25.0

    def plan(elb, done, cached):
        c = cached.tolist()
        r = P.plan_prefetch(elb.tolist(), done, c, K=K, capacity=cap, step_us=step_us, copy_us=copy_us)
        cached[:] = np.array(c, np.uint8)
        return r

    log, cached = _run_cycle(plan, L, E, k, K, picks)
    assert [p for _, p, _, _ in log][0] == P.COLD_START and log[-1][1] == P.FINAL_CLEANUP
    assert all(p == P.PREFETCH_OVERLAP for _, p, _, _ in log[1:-1])
    assert sum(c for _, _, _, c in log) == K          # the chunks cover the cycle exactly
    assert all(c >= 1 for _, p, _, c in log if p != P.FINAL_CLEANUP)
    assert (cached.sum(1) <= cap).all()
    final = np.zeros((L, E), np.int64)
    for st in range(K):
        for l in range(L):
            final[l, picks[st][l]] += 1
    if cap == E:  # no eviction: everything the lookahead saw ends up cached, loaded once
        assert np.array_equal(cached.astype(bool), final > 0)
        loads = [a for _, _, acts, _ in log for a in acts if a[2] == P.LOAD]
        assert len(loads) == len(set(loads)) == int((final > 0).sum())


@pytest.mark.parametrize("seed,L,E,k,K,cap,copy_us", [(10, 26, 64, 6, 16, 64, 38.0), (11, 26, 64, 6, 16, 12, 38.0),
                                                      (12, 24, 60, 4, 8, 20, 15.0), (13, 32, 16, 2, 16, 4, 350.0),
                                                      (14, 3, 256, 8, 7, 100, 1.0)])
def test_library_planner_equals_the_oracle(seed, L, E, k, K, cap, copy_us):
    from quantized_expert_gb300 import build, spx
    build.build()
    spx.load()
    rng = np.random.default_rng(seed)
    picks = _draw_cycle(rng, L, E, k, K)
    step_us = 26 * 25.0
    cfg = spx.PlanCfg(L, E, K, cap, 1, step_us, copy_us)

    def lib_plan(elb, done, cached):
        return spx.spx_plan_prefetch(cfg, elb, done, cached)

    def orc_plan(elb, done, cached):
        c = cached.tolist()
        ph, acts, ch = P.plan_prefetch(elb.tolist(), done, c, K=K, capacity=cap, step_us=step_us, copy_us=copy_us)
        cached[:] = np.array(c, np.uint8)
        return ph, np.array(acts, np.int32).reshape(-1, 3), ch

    log_l, cached_l = _run_cycle(lib_plan, L, E, k, K, picks)
    log_o, cached_o = _run_cycle(orc_plan, L, E, k, K, picks)
    assert log_l == log_o
    assert np.array_equal(cached_l, cached_o)


def test_library_planner_rejects_bad_arguments_without_side_effects():
    from quantized_expert_gb300 import build, spx
    build.build()
    spx.load()
    cfg = spx.PlanCfg(2, 4, 8, 4, 1, 100.0, 10.0)
    elb = np.ones((2, 4), np.uint32)
    cached = np.zeros((2, 4), np.uint8)
    with pytest.raises(spx.SpxError):
        spx.spx_plan_prefetch(cfg, elb, 9, cached)   # steps_done beyond K
    bad = spx.PlanCfg(2, 4, 8, 5, 1, 100.0, 10.0)     # capacity above E
    with pytest.raises(spx.SpxError):
        spx.spx_plan_prefetch(bad, elb, 1, cached)
    assert not cached.any()
    lib = spx.load()
    import ctypes as C
    n, ch, ph = C.c_int(), C.c_int(), C.c_int()
    acts = np.zeros((4, 3), np.int32)   # room for 4 actions; 8 demanded experts need 16
    assert lib.spx_plan_prefetch(C.byref(cfg), elb.ctypes.data, 1, cached.ctypes.data, acts.ctypes.data, 4,
                                 C.byref(n), C.byref(ch), C.byref(ph)) == spx.SPX_ERR_INVALID_ARG
    assert not cached.any()
    # the executor checks every action before enqueueing anything (no CUDA call here)
    bad_acts = np.array([[0, 1, spx.SPX_PLAN_LOAD], [5, 0, spx.SPX_PLAN_LOAD]], np.int32)
    ptrs = (C.c_void_p * 2)(256, 256)
    flags = np.array([1, 0, 0, 0, 0, 0, 0, 0], np.uint8)
    assert lib.spx_prefetch_issue(bad_acts.ctypes.data, 2, ptrs, ptrs, 1024, C.c_void_p(256), None,
                                  flags.ctypes.data, 2, 4, None) == spx.SPX_ERR_INVALID_ARG
    assert lib.spx_prefetch_issue(bad_acts.ctypes.data, 1, ptrs, ptrs, 1024, C.c_void_p(256), None, None, 2, 4,
                                  None) == spx.SPX_ERR_INVALID_ARG
