// spx_plan.cu -- the Layer-Aware Prefetch Planner and its copy executor
// (host code only).
//
// Method (ai.info summary of the Specter paper, Key Contributions 3 and
// "Methodology in Plain English"; richland.au post, "What shipped"): the
// Expert Lookahead Buffer's per-layer activation counters are snapshotted at
// draft-chunk boundaries; each snapshot becomes a compact plan of host-to-
// device expert copies, organised in three phases (Cold Start before the first
// draft step, Prefetch Overlap between chunks, Final Cleanup after the last
// step), and the next draft chunk is sized so that its compute roughly covers
// the copies just issued on a parallel stream.  During verification the
// expert launch computes cached experts first and waits (bounded) on the ready
// flag of each expert still in flight.
//
// GB300: the pages' host link is PCIe on an A100; here it is NVLink-C2C between
// Grace memory and HBM.  The planner is link-agnostic: the caller gives the
// measured time of one expert's copy and of one draft step.
#include "spx_internal.cuh"

#include <math.h>

#include <algorithm>
#include <vector>

using namespace spx;

extern "C" int spx_plan_prefetch(const spx_plan_cfg *cfg, const uint32_t *elb, int steps_done, uint8_t *cached,
                                 int32_t *actions, int max_actions, int *n_actions, int *next_chunk, int *phase) {
    if (!cfg || !elb || !cached || !n_actions || !next_chunk || !phase) return SPX_ERR_INVALID_ARG;
    const int L = cfg->L, E = cfg->E, K = cfg->K;
    if (L < 1 || E < 1 || E > kMaxE || K < 1 || cfg->capacity < 1 || cfg->capacity > E) return SPX_ERR_INVALID_ARG;
    if (cfg->min_chunk < 1 || !(cfg->step_us > 0.0) || !(cfg->copy_us >= 0.0)) return SPX_ERR_INVALID_ARG;
    if (steps_done < 0 || steps_done > K) return SPX_ERR_INVALID_ARG;
    if (max_actions < 0 || (max_actions > 0 && !actions)) return SPX_ERR_INVALID_ARG;
    const int ph = steps_done == 0 ? SPX_PLAN_COLD_START : steps_done < K ? SPX_PLAN_PREFETCH_OVERLAP
                                                                          : SPX_PLAN_FINAL_CLEANUP;
    // Check the room first, so that a rejected call leaves `cached` untouched:
    // every demanded expert costs at most one eviction and one load.
    int need = 0;
    for (int l = 0; l < L; ++l)
        for (int e = 0; e < E; ++e) need += (elb[(size_t)l * E + e] > 0 && !cached[(size_t)l * E + e]) ? 2 : 0;
    if (need > max_actions) return SPX_ERR_INVALID_ARG;

    int n = 0, loads = 0;
    std::vector<int> order;
    order.reserve(E);
    for (int l = 0; l < L; ++l) {  // layers in the order the verify pass needs them
        const uint32_t *cnt = elb + (size_t)l * E;
        uint8_t *cch = cached + (size_t)l * E;
        order.clear();
        for (int e = 0; e < E; ++e)
            if (cnt[e] > 0 && !cch[e]) order.push_back(e);
        // most counted first; equal counts in expert order (stable sort of an ascending list)
        std::stable_sort(order.begin(), order.end(), [cnt](int a, int b) { return cnt[a] > cnt[b]; });
        int held = 0;
        for (int e = 0; e < E; ++e) held += cch[e] ? 1 : 0;
        for (int e : order) {
            if (held >= cfg->capacity) {
                int victim = -1;  // a cached expert the counters have not seen, lowest index
                for (int v = 0; v < E && victim < 0; ++v)
                    if (cch[v] && cnt[v] == 0) victim = v;
                if (victim < 0) break;  // the cache holds only demanded experts
                cch[victim] = 0;
                --held;
                actions[3 * n] = l;
                actions[3 * n + 1] = victim;
                actions[3 * n + 2] = SPX_PLAN_EVICT;
                ++n;
            }
            cch[e] = 1;
            ++held;
            actions[3 * n] = l;
            actions[3 * n + 1] = e;
            actions[3 * n + 2] = SPX_PLAN_LOAD;
            ++n;
            ++loads;
        }
    }
    int chunk = 0;
    if (ph != SPX_PLAN_FINAL_CLEANUP) {
        const double cover = loads ? ceil((double)loads * cfg->copy_us / cfg->step_us) : (double)cfg->min_chunk;
        const double c = std::min(std::max(cover, (double)cfg->min_chunk), (double)(K - steps_done));
        chunk = (int)c;
    }
    *n_actions = n;
    *next_chunk = chunk;
    *phase = ph;
    return SPX_OK;
}

extern "C" int spx_prefetch_issue(const int32_t *actions, int n_actions, const void *const *host_experts,
                                  void *const *dev_experts, size_t expert_bytes, uint32_t *ready, uint8_t *resident,
                                  const uint8_t *host_flags, int L, int E, spx_stream_t stream) {
    if (n_actions < 0 || (n_actions > 0 && (!actions || !host_experts || !dev_experts || !ready || !host_flags)))
        return SPX_ERR_INVALID_ARG;
    if (L < 1 || E < 1 || expert_bytes == 0) return SPX_ERR_INVALID_ARG;
    for (int i = 0; i < n_actions; ++i) {  // every action checked before anything is enqueued
        const int l = actions[3 * i], e = actions[3 * i + 1], kind = actions[3 * i + 2];
        if (l < 0 || l >= L || e < 0 || e >= E || (kind != SPX_PLAN_LOAD && kind != SPX_PLAN_EVICT))
            return SPX_ERR_INVALID_ARG;
        if (kind == SPX_PLAN_LOAD && (!host_experts[l] || !dev_experts[l])) return SPX_ERR_INVALID_ARG;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int i = 0; i < n_actions; ++i) {
        const int l = actions[3 * i], e = actions[3 * i + 1];
        const size_t f = (size_t)l * E + e;
        cudaError_t err;
        // Flags are host-to-device copies of the caller's page-locked constants
        // (bytes 0-3 nonzero, 4-7 zero): the copy engines write them, so no SM
        // is needed while an expert launch that waits for them holds every SM.
        const uint8_t *val = host_flags + (actions[3 * i + 2] == SPX_PLAN_LOAD ? 0 : 4);
        if (actions[3 * i + 2] == SPX_PLAN_LOAD) {
            // one copy per expert (its packed bytes are contiguous), then its
            // flags, in stream order behind the copy
            err = cudaMemcpyAsync(static_cast<uint8_t *>(dev_experts[l]) + (size_t)e * expert_bytes,
                                  static_cast<const uint8_t *>(host_experts[l]) + (size_t)e * expert_bytes,
                                  expert_bytes, cudaMemcpyHostToDevice, s);
            if (err == cudaSuccess && resident) err = cudaMemcpyAsync(resident + f, val, 1, cudaMemcpyHostToDevice, s);
            if (err == cudaSuccess) err = cudaMemcpyAsync(ready + f, val, sizeof(uint32_t), cudaMemcpyHostToDevice, s);
        } else {
            err = cudaMemcpyAsync(ready + f, val, sizeof(uint32_t), cudaMemcpyHostToDevice, s);
            if (err == cudaSuccess && resident) err = cudaMemcpyAsync(resident + f, val, 1, cudaMemcpyHostToDevice, s);
        }
        if (err != cudaSuccess) return record_launch(err);
    }
    return SPX_OK;
}
