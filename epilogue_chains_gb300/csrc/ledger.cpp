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
