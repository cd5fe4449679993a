// ledger.cpp -- host-side byte ledgers (no CUDA calls).
//
// [K4] §① traffic(): a cut plan splits the K stages into consecutive kernels.  A kernel reads
// the output of the kernel before it (the `writes` of the stage just before its first stage,
// if any) plus the external reads of all its stages, and writes the output of its last stage.
// [K4] §② also needs the register peak of a plan: the largest sum of live_regs in one kernel.
#include <stdint.h>

#include "fusechain.h"

extern "C" int fuse_ledger(const fuse_stage* st, int K, uint32_t cut_mask, int elem_bytes,
                           fuse_ledger_t* out) {
    if (!st || !out || K < 1 || K > FUSE_MAX_STAGES || elem_bytes <= 0) return FUSE_EINVAL;
    if ((static_cast<uint64_t>(cut_mask) >> (K - 1)) != 0) return FUSE_EINVAL;  // past the last boundary
    for (int s = 0; s < K; ++s)
        if (st[s].writes < 0 || st[s].ext_reads < 0 || st[s].flops < 0 || st[s].live_regs < 0)
            return FUSE_EINVAL;
    int64_t elems = 0, launches = 0, reg_peak = 0, flops = 0;
    int first = 0;
    while (first < K) {
        int last = first;  // the kernel covers stages first..last
        while (last < K - 1 && !((cut_mask >> last) & 1u)) ++last;
        int64_t reads = first > 0 ? st[first - 1].writes : 0;
        int64_t regs = 0;
        for (int s = first; s <= last; ++s) {
            reads += st[s].ext_reads;
            regs += st[s].live_regs;
            flops += st[s].flops;
        }
        elems += reads + st[last].writes;
        if (regs > reg_peak) reg_peak = regs;
        ++launches;
        first = last + 1;
    }
    out->bytes = elems * elem_bytes;
    out->launches = launches;
    out->reg_peak = reg_peak;
    out->flops = flops;
    return FUSE_OK;
}

// [K4] §② time_estimate: each kernel of the plan costs max(memory time, compute time) + launch;
// a kernel whose live registers exceed the limit has its memory time multiplied by the spill
// penalty (§③).  §② best_plan: enumerate the 2^(K-1) cut masks and keep the cheapest.
extern "C" int fuse_plan_time(const fuse_stage* st, int K, uint32_t cut_mask, int elem_bytes,
                              const fuse_cost_model* m, double* seconds) {
    if (!st || !m || !seconds || K < 1 || K > FUSE_MAX_STAGES || elem_bytes <= 0) return FUSE_EINVAL;
    if ((static_cast<uint64_t>(cut_mask) >> (K - 1)) != 0) return FUSE_EINVAL;
    if (!(m->hbm_bytes_per_s > 0) || !(m->flops_per_s > 0) || !(m->launch_s >= 0) ||
        !(m->spill_penalty >= 1))
        return FUSE_EINVAL;
    double total = 0.0;
    int first = 0;
    while (first < K) {
        int last = first;
        while (last < K - 1 && !((cut_mask >> last) & 1u)) ++last;
        int64_t elems = first > 0 ? st[first - 1].writes : 0;
        int64_t regs = 0, flops = 0;
        for (int s = first; s <= last; ++s) {
            if (st[s].writes < 0 || st[s].ext_reads < 0 || st[s].flops < 0 || st[s].live_regs < 0)
                return FUSE_EINVAL;
            elems += st[s].ext_reads;
            regs += st[s].live_regs;
            flops += st[s].flops;
        }
        elems += st[last].writes;
        double mem = static_cast<double>(elems) * elem_bytes / m->hbm_bytes_per_s;
        if (regs > m->reg_limit) mem *= m->spill_penalty;
        const double comp = static_cast<double>(flops) / m->flops_per_s;
        total += (mem > comp ? mem : comp) + m->launch_s;
        first = last + 1;
    }
    *seconds = total;
    return FUSE_OK;
}

extern "C" int fuse_best_plan(const fuse_stage* st, int K, int elem_bytes, const fuse_cost_model* m,
                              uint32_t* best_mask, double* best_seconds) {
    if (!best_mask || !best_seconds || K < 1 || K > 20) return FUSE_EINVAL;  // 2^19 plans at most
    double best = 0.0;
    uint32_t arg = 0;
    for (uint32_t mask = 0; mask < (1u << (K - 1)); ++mask) {
        double t = 0.0;
        const int rc = fuse_plan_time(st, K, mask, elem_bytes, m, &t);
        if (rc != FUSE_OK) return rc;
        if (mask == 0 || t < best) {
            best = t;
            arg = mask;
        }
    }
    *best_mask = arg;
    *best_seconds = best;
    return FUSE_OK;
}

// "AIGC fundamentals | operator fusion and CUDA Graph" §3.4: single-stream timeline of N kernels.
// Eager: kernel i starts at max(end of kernel i-1, (i+1) t_launch), which solves to
// t_launch + N t_exec when the host keeps ahead (t_launch <= t_exec) and N t_launch + t_exec when
// it does not.  Graph: one submission, then t_exec + t_dispatch per node.
extern "C" int fuse_launch_model(int64_t n_kernels, double t_launch, double t_exec,
                                 double t_dispatch, double* eager, double* eager_idle,
                                 double* graph) {
    if (n_kernels < 0 || !(t_launch >= 0) || !(t_exec >= 0) || !(t_dispatch >= 0) || !eager ||
        !eager_idle || !graph)
        return FUSE_EINVAL;
    const double n = static_cast<double>(n_kernels);
    double total = 0.0;
    if (n_kernels > 0) total = t_launch <= t_exec ? t_launch + n * t_exec : n * t_launch + t_exec;
    *eager = total;
    *eager_idle = total - n * t_exec;
    *graph = t_launch + n * (t_exec + t_dispatch);
    return FUSE_OK;
}
