#!/usr/bin/env python3
"""Benchmark of the fused-chain hot path on one GB300 (or N, one process per GPU, weak scaling).

Metric: fused-chain HBM GB/s (and % of the GB300 peak) with the fused/unfused speedup as a
function of K, on the pointwise chain x, y fp32 [16,777,216], K in {2, 3, 4, 6, 8}, stage
y = a_s y + b_s (a_s ~ U[0.9,1.1], b_s ~ U[-0.1,0.1]), ReLU on even s.

One step = one pass over every row of the hot path on its own synthetic batch:
  chain fused (K = 2,3,4,6,8) | chain unfused (same K) | fat probe (K = 4) |
  RMSNorm [2048,4096] fused + unfused | residual add + RMSNorm | SiLU*up |
  causal softmax [8,16,2048,2048] fused (skip 0/64/128) + unfused | attention [128,2048,256] |
  GEMM + bias + GELU + residual 4096^3 and 16x4096x4096, every cut plan.
Each group is one kind of call: one untimed call first, then its timed calls back to back over
rotating buffers (4 input/output pairs, 512 MiB for the chain: larger than the 126 MiB L2), so
every timed call pays for the dirty lines its predecessor left in L2, as in a steady stream.  One
pair of CUDA events on the launching stream brackets the group's timed calls, so a call's time is
the group's time over its calls: the work of a stream of such calls, without an event between
every two of them.  A separate pass after the timed region brackets single calls (rows.per_call).

``value`` = fused-chain algorithmic bytes (2 N b per call, N b read + N b written) / the fused
chain groups' device time.  ``e2e`` = the same bytes / the time of the same chains run through
the C ABI's host-buffer entry point (fuse_chain_run_host) from pinned host memory: each call
copies its x in and its y out in slices whose copies overlap the kernels.

``--impl reference`` times the plain CPU oracle (the only other place this script runs it) on
the same workload on the host cores, rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 7900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--rows", choices=["all", "chain"], default="all",
                    help="'chain' restricts a step to the metric's own row (the chain sweep)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", default=None,
                    choices=["chain_fused", "chain_unfused", "chain_fat", "rmsnorm_fused",
                             "rmsnorm_unfused", "softmax_fused", "softmax_unfused", "gemm",
                             "add_rmsnorm_fused", "add_rmsnorm_unfused", "silu_mul_fused",
                             "silu_mul_unfused", "attention"],
                    help="run only `--launches` calls of one row (for ncu), print a short line")
    ap.add_argument("--size", type=int, default=None,
                    help="profile size: chain elements, RMSNorm rows or softmax batch*heads")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--K", type=int, default=8, help="chain stages for --profile")
    ap.add_argument("--tile", type=int, default=64, help="softmax skip tile for --profile")
    ap.add_argument("--mask", type=int, default=0, help="GEMM cut mask for --profile gemm")
    ap.add_argument("--no-static-b", action="store_true",
                    help="--profile gemm at M <= 64: leave FUSE_GEMM_STATIC_B off")
    return ap.parse_args()


def max_over_ranks(values, world, device):
    """Each value's maximum over all ranks (one all_reduce of the vector), or the values as they
    are with a single rank.  The timed region of every rank is bracketed by a barrier, so the
    slowest rank's time is the job's time."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def weak_scaling_gbs(bytes_per_rank, world, elapsed_s):
    """Whole-job throughput of a weak-scaling run: every rank moved `bytes_per_rank`, the job took
    the slowest rank's `elapsed_s`."""
    return bytes_per_rank * world / elapsed_s / 1e9


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append({"t": _smi_time(f[0]), "sm": float(f[2]), "sm_max": float(f[3]),
                             "power": f[4], "active": f[5], "hw": f[6], "hw_thermal": f[7],
                             "sw_thermal": f[8], "sw_power": f[9]})
            except ValueError:
                continue
        return rows


def _smi_time(stamp: str) -> float:
    """nvidia-smi timestamp 'YYYY/MM/DD HH:MM:SS.mmm' (local time) -> seconds since the epoch."""
    whole, _, frac = stamp.partition(".")
    return time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S")) + (float("0." + frac) if frac else 0.0)


def summarize_clocks(rows, t0, t1):
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
    inside = [r for r in rows if t0 - 0.05 <= r["t"] <= t1 + 0.05] or rows
    reasons = set()
    for r in inside:
        for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
            if r[key].lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(r["sm"] for r in inside),
            "sm_max_mhz": max(r["sm_max"] for r in inside), "reasons": sorted(reasons),
            "samples": len(inside)}


# ------------------------------------------------------------------------------ traffic
def committed_traffic(group: str, src_name: str):
    """DRAM bytes per launch of a kernel from its committed ncu summary (profiles/<group>.txt),
    if that summary was captured from the current kernel source (sha256 recorded in it)."""
    path = os.path.join(ROOT, "profiles", f"{group}.txt")
    src = os.path.join(ROOT, "epilogue_chains_gb300", "csrc", src_name)
    if not src_name or not os.path.exists(path) or not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_sha256") != sha:
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------------------ our arm
class Group:
    """One kind of call in a step: an untimed leading call, then `n` timed calls back to back.

    fn(): one call (rotating its buffers); units: the call's algorithmic bytes (bound "hbm") or
    flops (bound "tensor"); kernel: the single kernel a call launches (None if it launches
    several); launches: kernels of ours per call; family: groups of the same kernel that add up
    to one roofline row."""

    def __init__(self, name, fn, units, n, bound, kernel, launches, family=None):
        self.name, self.fn, self.units, self.n = name, fn, units, n
        self.bound, self.kernel, self.launches = bound, kernel, launches
        self.family = family or name


def run_ours(args, rank, world, local):
    import torch
    import epilogue_chains_gb300 as fc
    from epilogue_chains_gb300 import workloads as wl

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    lib = fc._load()
    peaks, peak_src = load_peaks()
    counter = {"launches": 0}

    def check(rc, where):
        if rc != 0:
            raise fc.FuseError(rc, where)

    def rotating(n):
        state = {"i": 0}

        def nxt():
            state["i"] += 1
            return (state["i"] - 1) % n
        return nxt

    # ------------------------------------------------------------------ pointwise chain
    N, KS, R = wl.CHAIN_N, wl.CHAIN_KS, 4
    with torch.cuda.stream(stream):
        xs = [wl.chain_input(N, device=dev, salt=r + 100 * rank) for r in range(R)]
        ys = [torch.empty_like(xs[0]) for _ in range(R)]
    stage_sets = {}
    for K in KS:
        relu, a, b = wl.chain_stages(K)
        stage_sets[K] = fc._stages([(fc.FUSE_OP_AFFINE_RELU if r_ else fc.FUSE_OP_AFFINE, p, q)
                                    for r_, p, q in zip(relu, a, b)])
    chain_bytes = fc.fuse_chain_bytes(1, N, fc.FUSE_F32, fc.FUSE_FUSED)  # 2 N b, any K
    crot = rotating(R)

    def chain(K, mode):
        def fn():
            i = crot()
            check(lib.fuse_chain_run(stage_sets[K], K, xs[i].data_ptr(), ys[i].data_ptr(), N,
                                     fc.FUSE_F32, mode, sh), "fuse_chain_run")
            counter["launches"] += K if mode == fc.FUSE_UNFUSED else 1
        return fn

    # Calls of one kind run back to back between one event pair.  The first call after an event
    # record cannot start under the preceding call's tail (measured per call for the K = 4 chain:
    # 21.5 / 20.2 / 19.5 / 19.1 us for 2 / 4 / 8 / 16 calls; SiLU*up 28.6 / 27.4 / 26.7 / 26.3 us;
    # RMSNorm 13.3 / 12.5 / 12.0 / 11.6 us), so calls under ~100 us are timed 8 to a group, fused
    # and unfused alike, and longer ones 2 to 4 (4 where that start, ~7 us for attention, would
    # otherwise cost more than 1 %).
    groups = [Group(f"chain_fused_K{K}", chain(K, fc.FUSE_FUSED), chain_bytes, 8, "hbm",
                    "chain_fused_kernel<f32>", 1, "chain_fused") for K in KS]
    groups += [Group(f"chain_unfused_K{K}", chain(K, fc.FUSE_UNFUSED),
                     fc.fuse_chain_bytes(K, N, fc.FUSE_F32, fc.FUSE_UNFUSED), 8, "hbm", None, K,
                     "chain_unfused") for K in KS]
    # The same sweep at N = 2^26 (256 MiB per operand, twice the L2): an unfused stage's 256 MiB
    # intermediate cannot stay in L2, so every stage moves its 2 N b through DRAM as the ledger
    # prices it, where at N = 2^24 the 64 MiB intermediate is partly served from L2.
    NB, RB = 4 * N, 2
    with torch.cuda.stream(stream):
        xbs = [wl.chain_input(NB, device=dev, salt=r + 7 + 100 * rank) for r in range(RB)]
        ybs = [torch.empty_like(xbs[0]) for _ in range(RB)]
    brot = rotating(RB)
    chain_bytes_big = fc.fuse_chain_bytes(1, NB, fc.FUSE_F32, fc.FUSE_FUSED)

    def chain_big(K, mode):
        def fn():
            i = brot()
            check(lib.fuse_chain_run(stage_sets[K], K, xbs[i].data_ptr(), ybs[i].data_ptr(), NB,
                                     fc.FUSE_F32, mode, sh), "fuse_chain_run")
            counter["launches"] += K if mode == fc.FUSE_UNFUSED else 1
        return fn

    groups += [Group(f"chain26_fused_K{K}", chain_big(K, fc.FUSE_FUSED), chain_bytes_big, 4, "hbm",
                     "chain_fused_kernel<f32>", 1, "chain26_fused") for K in KS]
    groups += [Group(f"chain26_unfused_K{K}", chain_big(K, fc.FUSE_UNFUSED),
                     fc.fuse_chain_bytes(K, NB, fc.FUSE_F32, fc.FUSE_UNFUSED), 2, "hbm", None, K,
                     "chain26_unfused") for K in KS]
    # the fat probe is a fixed-point probe at K = 4 ([C05] §5: not part of the sweep)
    groups += [Group("chain_fat", chain(4, fc.FUSE_FAT), chain_bytes, 2, "hbm", "chain_fat_kernel<f32>", 1)]

    plans = {"[4]": 0, "[1,3]": 1, "[2,2]": 2, "[1,1,1,1]": 7}
    gemm_bufs = {}
    if args.rows == "all":
        # -------------------------------------------------------------- RMSNorm
        with torch.cuda.stream(stream):
            rx, rw = wl.rmsnorm_input(device=dev, salt=rank)
            rxs = [rx] + [rx.clone() for _ in range(7)]   # 8 x/y pairs: 512 MiB, four times the L2
            rys = [torch.empty_like(rx) for _ in range(8)]
            rws = torch.empty(fc.fuse_rmsnorm_workspace_bytes(wl.RMS_ROWS, wl.RMS_HIDDEN, fc.FUSE_UNFUSED),
                              dtype=torch.uint8, device=dev)
        rrot = rotating(8)

        def rms(mode):
            def fn():
                i = rrot()
                check(lib.fuse_rmsnorm(rxs[i].data_ptr(), rw.data_ptr(), rys[i].data_ptr(), wl.RMS_ROWS,
                                       wl.RMS_HIDDEN, wl.RMS_EPS, mode, rws.data_ptr(), rws.numel(), sh),
                      "fuse_rmsnorm")
                counter["launches"] += 1 if mode == fc.FUSE_FUSED else 4
            return fn
        rb = {m: fc.fuse_rmsnorm_bytes(wl.RMS_ROWS, wl.RMS_HIDDEN, m) for m in (fc.FUSE_FUSED, fc.FUSE_UNFUSED)}
        groups += [
            # one call per x/y pair of the rotation: the group's leading launch latency is spread over
            # as many ~13 us calls as the rotation holds
            Group("rmsnorm_fused", rms(fc.FUSE_FUSED), rb[fc.FUSE_FUSED], 8, "hbm", "rmsnorm_row_kernel", 1),
            Group("rmsnorm_unfused", rms(fc.FUSE_UNFUSED), rb[fc.FUSE_UNFUSED], 8, "hbm", None, 4),
        ]
        # -------------------------------------------------------------- residual add + RMSNorm
        with torch.cuda.stream(stream):
            ax, ar, aw = wl.add_rmsnorm_input(device=dev, salt=rank)
            axs, ars = [ax] + [ax.clone() for _ in range(3)], [ar] + [ar.clone() for _ in range(3)]
            ahs = [torch.empty_like(ax) for _ in range(4)]   # 4 sets of x, r, h, y: 512 MiB
            ays = [torch.empty_like(ax) for _ in range(4)]
        arot = rotating(4)
        AR, AH = wl.ADDRMS_ROWS, wl.ADDRMS_HIDDEN

        def addrms(mode):
            def fn():
                i = arot()
                check(lib.fuse_add_rmsnorm(axs[i].data_ptr(), ars[i].data_ptr(), aw.data_ptr(),
                                           ahs[i].data_ptr(), ays[i].data_ptr(), AR, AH, wl.RMS_EPS, mode,
                                           rws.data_ptr(), rws.numel(), sh), "fuse_add_rmsnorm")
                counter["launches"] += 1 if mode == fc.FUSE_FUSED else 5
            return fn
        ab = {m: fc.fuse_add_rmsnorm_bytes(AR, AH, m) for m in (fc.FUSE_FUSED, fc.FUSE_UNFUSED)}
        # -------------------------------------------------------------- SiLU(gate) * up
        SR, SC = wl.SILU_ROWS, wl.SILU_COLS
        with torch.cuda.stream(stream):
            gu0 = wl.silu_input(device=dev, salt=rank)
            gus = [gu0, gu0.clone()]
            sys_ = [torch.empty(SR, SC, dtype=gu0.dtype, device=dev) for _ in range(2)]
        grot = rotating(2)

        def silu(mode):
            def fn():
                i = grot()
                base = gus[i].data_ptr()
                check(lib.fuse_silu_mul(base, base + SC * 2, 2 * SC, sys_[i].data_ptr(), SR, SC,
                                        fc.FUSE_BF16, mode, sh), "fuse_silu_mul")
                counter["launches"] += 1 if mode == fc.FUSE_FUSED else 2
            return fn
        sb = {m: fc.fuse_silu_mul_bytes(SR, SC, fc.FUSE_BF16, m) for m in (fc.FUSE_FUSED, fc.FUSE_UNFUSED)}
        groups += [
            Group("add_rmsnorm_fused", addrms(fc.FUSE_FUSED), ab[fc.FUSE_FUSED], 8, "hbm",
                  "rmsnorm_row_kernel<+residual>", 1),
            Group("add_rmsnorm_unfused", addrms(fc.FUSE_UNFUSED), ab[fc.FUSE_UNFUSED], 8, "hbm", None, 5),
            Group("silu_mul_fused", silu(fc.FUSE_FUSED), sb[fc.FUSE_FUSED], 8, "hbm", "silu_mul_vec_kernel<bf16>", 1),
            Group("silu_mul_unfused", silu(fc.FUSE_UNFUSED), sb[fc.FUSE_UNFUSED], 8, "hbm", None, 2),
        ]
        # -------------------------------------------------------------- causal softmax
        bh, S = wl.SM_B * wl.SM_H, wl.SM_S
        with torch.cuda.stream(stream):
            ss = [wl.softmax_input(bh, S, device=dev, salt=rank), None]
            ss[1] = ss[0].clone()
            sps = [torch.empty_like(ss[0]) for _ in range(2)]
            sws = torch.empty(fc.fuse_causal_softmax_workspace_bytes(bh, S, fc.FUSE_UNFUSED),
                              dtype=torch.uint8, device=dev)
        srot = rotating(2)

        def sm(tile, mode):
            def fn():
                i = srot()
                check(lib.fuse_causal_softmax(ss[i].data_ptr(), sps[i].data_ptr(), bh, S, wl.SM_SCALE,
                                              tile, fc.FUSE_BF16, mode, sws.data_ptr(), sws.numel(), sh),
                      "fuse_causal_softmax")
                counter["launches"] += 1 if mode == fc.FUSE_FUSED else 5
            return fn
        groups += [Group(f"softmax_fused_T{t}", sm(t, fc.FUSE_FUSED),
                         fc.fuse_causal_softmax_bytes(bh, S, t, fc.FUSE_BF16, fc.FUSE_FUSED), 2, "hbm",
                         "softmax_fused_kernel<bf16>", 1, "softmax_fused") for t in (0, 64, 128)]
        groups += [Group("softmax_unfused", sm(0, fc.FUSE_UNFUSED),
                         fc.fuse_causal_softmax_bytes(bh, S, 0, fc.FUSE_BF16, fc.FUSE_UNFUSED), 1, "hbm", None, 5)]
        # -------------------------------------------------------------- attention, no score matrix
        with torch.cuda.stream(stream):
            aq, ak, av = wl.attention_input(device=dev, salt=rank)
            aos = [torch.empty_like(aq) for _ in range(2)]
        orot = rotating(2)
        ABH, AS, AD = wl.ATT_BH, wl.ATT_S, wl.ATT_D

        def attn():
            check(lib.fuse_attention(aq.data_ptr(), ak.data_ptr(), av.data_ptr(), aos[orot()].data_ptr(),
                                     ABH, AS, AD, wl.ATT_SCALE, sh), "fuse_attention")
            counter["launches"] += 1
        att_flops = fc.fuse_attention_flops(ABH, AS, AD)
        groups += [Group("attention_fused", attn, att_flops, 4, "tensor", "attn_persist_kernel<D=256>", 1)]
        # -------------------------------------------------------------- GEMM epilogue chain
        gN, gK = wl.GEMM_N, wl.GEMM_K
        with torch.cuda.stream(stream):
            for M in wl.GEMM_MS:
                A, B, bias, Rr = wl.gemm_input(M, device=dev, salt=rank)
                nb = 6 if M < 128 else 1   # decode: rotate 6 weight copies (192 MiB, beyond L2)
                Bs = [B] + [B.clone() for _ in range(nb - 1)]
                Ys = [torch.empty(M, gN, dtype=torch.float16, device=dev) for _ in range(2)]
                # split-K workspace for the last wave of tiles (zero-filled once, reused)
                gws = torch.zeros(max(1, fc.fuse_gemm_workspace_bytes(M, gN, gK)), dtype=torch.uint8, device=dev)
                gemm_bufs[M] = (A, Bs, bias, Rr, Ys, rotating(nb), rotating(2), gws)

        def gemm(M, mask, flags=0):
            A, Bs, bias, Rr, Ys, brot, yrot, gws = gemm_bufs[M]

            def fn():
                b, y = Bs[brot()], Ys[yrot()]
                check(lib.fuse_gemm_epilogue_ws(A.data_ptr(), b.data_ptr(), bias.data_ptr(), Rr.data_ptr(),
                                                y.data_ptr(), M, gN, gK, mask | flags, gws.data_ptr(), gws.numel(),
                                                sh), "fuse_gemm_epilogue_ws")
                counter["launches"] += 1 + bin(mask).count("1")
            return fn
        flops = {M: 2 * M * gN * gK for M in wl.GEMM_MS}
        for p_, m_ in plans.items():
            groups.append(Group(f"gemm_M4096_{p_}", gemm(4096, m_), flops[4096], 4 if m_ == 0 else 2, "tensor",
                                "gemm_tc_kernel" if m_ == 0 else None, 1 + bin(m_).count("1"),
                                "gemm_M4096_fused" if m_ == 0 else "gemm_M4096_unfused"))
        # decode calls are ~10 us: 16 (8) back-to-back calls per group, as a decode loop issues
        # them, so the group's leading launch latency is spread over enough calls
        # the decode loop's weights are never written by the kernels before them, so its calls
        # carry FUSE_GEMM_STATIC_B (the first weight boxes load while the preceding call finishes);
        # one group without it shows the plain stream-ordered call
        for p_, m_ in plans.items():
            groups.append(Group(f"gemm_M16_{p_}", gemm(16, m_, fc.FUSE_GEMM_STATIC_B), fc.fuse_gemm_bytes(16, gN, gK, m_),
                                16 if m_ == 0 else 8, "hbm", "gemm_decode_kernel<16>" if m_ == 0 else None,
                                1 + bin(m_).count("1"), "gemm_M16_fused" if m_ == 0 else "gemm_M16_unfused"))
        groups.append(Group("gemm_M16_[4]_nostatic", gemm(16, 0), fc.fuse_gemm_bytes(16, gN, gK, 0), 16, "hbm", None,
                            1, "gemm_M16_nostatic"))

    def make_events():
        # per group: the untimed leading call's pair, then one pair around the timed calls
        return {g.name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                         for _ in range(2)] for g in groups}

    def step(evs):
        with torch.cuda.stream(stream):
            for g in groups:
                (l0, l1), (e0, e1) = evs[g.name]
                l0.record(stream)
                g.fn()
                l1.record(stream)
                e0.record(stream)
                for _ in range(g.n):
                    g.fn()
                e1.record(stream)

    for _ in range(max(3, args.warmup)):      # warm-up steps (untimed)
        step(make_events())
    torch.cuda.synchronize()

    all_evs = [make_events() for _ in range(args.steps)]
    sampler = ClockSampler(local)
    time.sleep(0.3)  # let nvidia-smi start sampling
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    counter["launches"] = 0
    t0 = time.time()
    for s_ in range(args.steps):
        step(all_evs[s_])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t1 = time.time()
    clocks = summarize_clocks(sampler.stop(), t0, t1)
    # every kernel of ours launched inside the timed region, the untimed leading calls included
    timed_launches = counter["launches"]

    gmap = {g.name: g for g in groups}
    # ms of a group's timed calls per step, and of its leading call
    gms = {g.name: [evs[g.name][1][0].elapsed_time(evs[g.name][1][1]) for evs in all_evs] for g in groups}
    lead = {g.name: [evs[g.name][0][0].elapsed_time(evs[g.name][0][1]) for evs in all_evs] for g in groups}

    def call_ms(name):       # mean ms per call of a group
        return float(np.mean(gms[name])) / gmap[name].n

    step_ms = float(np.mean([sum(gms[g][s_] for g in gms) for s_ in range(args.steps)]))
    fused_groups = [g for g in groups if g.family == "chain_fused"]
    elapsed_s = sum(sum(gms[g.name]) for g in fused_groups) / 1e3
    n_fused = args.steps * sum(g.n for g in fused_groups)
    elapsed_s, step_ms = max_over_ranks([elapsed_s, step_ms], world, dev)
    value = weak_scaling_gbs(n_fused * chain_bytes, world, elapsed_s)

    kernel_src = {"softmax_fused": "softmax.cu", "chain_fused": "chain.cu", "gemm_M4096_fused": "gemm.cu",
                  "chain_fat": "chain.cu", "rmsnorm_fused": "rmsnorm.cu", "gemm_M16_fused": "gemm_decode.cu",
                  "add_rmsnorm_fused": "rmsnorm.cu", "silu_mul_fused": "silu_mul.cu",
                  "attention_fused": "attention.cu", "chain26_fused": "chain.cu"}
    families = {}
    for g in groups:
        families.setdefault(g.family, []).append(g)

    def family_ms(fam):      # mean ms per step of a family's timed calls
        return sum(float(np.mean(gms[g.name])) for g in families[fam])

    def roofline_of(fam):
        gs = families[fam]
        calls = sum(g.n for g in gs)
        tot_units = sum(g.units * g.n for g in gs)
        tot_ms = family_ms(fam)
        if gs[0].bound == "hbm":
            achieved, peak, unit = tot_units / tot_ms / 1e6, peaks["hbm_gbs"], "GB/s"
        else:
            achieved, peak, unit = tot_units / tot_ms / 1e9, peaks["bf16_tflops"], "TFLOP/s"
        out = {"bound": gs[0].bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
               "frac": round(achieved / peak, 4), "kernel": gs[0].kernel,
               "units_per_launch": int(tot_units / calls),
               "avg_launch_us": round(tot_ms / calls * 1e3, 2),
               "step_share": round(tot_ms / step_ms, 4)}
        if gs[0].bound == "tensor":
            out["frac_of_sustained"] = round(achieved / peaks["bf16_tflops_sustained"], 4)
        else:
            out["frac_of_nominal"] = round(achieved / NOMINAL_HBM_GBS, 4)
        # DRAM bytes per launch from the committed ncu summary of this kernel source, else None
        out["traffic"] = committed_traffic(fam, kernel_src.get(fam, ""))
        return out

    # dominant kernel: the single-kernel family with the largest share of the step
    single = [f for f, gs in families.items() if gs[0].kernel is not None]
    dominant = max(single, key=family_ms)
    roofline = roofline_of(dominant)
    roofline["peak_source"] = peak_src

    rows = {"timing": "per group: one untimed call, then its timed calls back to back between one "
                      "CUDA event pair; per-call figures are the group time over its calls",
            "step_share": {f: round(family_ms(f) / step_ms, 4) for f in families}}
    # the same shares over every launch of the step, the untimed lead calls included: the figure an
    # ncu launch list of this command (all launches, serialised) can be compared with
    all_ms = {f: sum(float(np.mean(gms[g.name])) + float(np.mean(lead[g.name])) for g in gs)
              for f, gs in families.items()}
    rows["step_share_all_launches"] = {k: round(v / sum(all_ms.values()), 4) for k, v in all_ms.items()}
    per_k = {}
    for K in KS:
        f = call_ms(f"chain_fused_K{K}")
        u = call_ms(f"chain_unfused_K{K}")
        per_k[str(K)] = {"fused_us": round(f * 1e3, 2), "unfused_us": round(u * 1e3, 2),
                         "speedup_fused_vs_unfused": round(u / f, 3),
                         "fused_GBs": round(chain_bytes / (f / 1e3) / 1e9, 1),
                         "unfused_ledger_GBs": round(fc.fuse_chain_bytes(K, N, fc.FUSE_F32, fc.FUSE_UNFUSED)
                                                     / (u / 1e3) / 1e9, 1)}
    per_k26 = {}
    for K in KS:
        f = call_ms(f"chain26_fused_K{K}")
        u = call_ms(f"chain26_unfused_K{K}")
        per_k26[str(K)] = {"fused_us": round(f * 1e3, 2), "unfused_us": round(u * 1e3, 2),
                           "speedup_fused_vs_unfused": round(u / f, 3),
                           "fused_GBs": round(chain_bytes_big / (f / 1e3) / 1e9, 1),
                           "unfused_ledger_GBs": round(fc.fuse_chain_bytes(K, NB, fc.FUSE_F32, fc.FUSE_UNFUSED)
                                                       / (u / 1e3) / 1e9, 1)}
    fat = call_ms("chain_fat")
    rows["chain"] = {"per_K": per_k, "roofline_fused": roofline_of("chain_fused"),
                     "per_K_N2^26": per_k26, "roofline_fused_N2^26": roofline_of("chain26_fused"),
                     "note_N2^26": "operands of 256 MiB, twice the L2: every unfused stage's "
                                   "intermediate goes through DRAM, as the 2KNb ledger prices it",
                     "fat_K4": {"us": round(fat * 1e3, 2), "fat_over_fused": round(fat / call_ms("chain_fused_K4"), 3)}}
    if args.rows == "all":
        rf, ru = call_ms("rmsnorm_fused"), call_ms("rmsnorm_unfused")
        rows["rmsnorm"] = {"fused_us": round(rf * 1e3, 2), "unfused_us": round(ru * 1e3, 2),
                           "speedup": round(ru / rf, 3), "roofline_fused": roofline_of("rmsnorm_fused")}
        af, au = call_ms("add_rmsnorm_fused"), call_ms("add_rmsnorm_unfused")
        rows["add_rmsnorm"] = {"fused_us": round(af * 1e3, 2), "unfused_us": round(au * 1e3, 2),
                               "speedup": round(au / af, 3),
                               "unfused_ledger_GBs": round(ab[fc.FUSE_UNFUSED] / au / 1e6, 1),
                               "roofline_fused": roofline_of("add_rmsnorm_fused")}
        sf, su = call_ms("silu_mul_fused"), call_ms("silu_mul_unfused")
        rows["silu_mul"] = {"fused_us": round(sf * 1e3, 2), "unfused_us": round(su * 1e3, 2),
                            "speedup": round(su / sf, 3),
                            "unfused_ledger_GBs": round(sb[fc.FUSE_UNFUSED] / su / 1e6, 1),
                            "roofline_fused": roofline_of("silu_mul_fused")}
        at = call_ms("attention_fused")
        rows["attention"] = {"us": round(at * 1e3, 1), "flops": att_flops,
                             "TFLOPs": round(att_flops / at / 1e9, 1),
                             "bytes": fc.fuse_attention_bytes(ABH, AS, AD),
                             "roofline": roofline_of("attention_fused"),
                             "softmax_alone_T0_us": round(call_ms("softmax_fused_T0") * 1e3, 1),
                             "vs_softmax_alone": round(call_ms("softmax_fused_T0") / at, 3),
                             "note": "the materialised path needs Q K^T and P V GEMMs besides the "
                                     "softmax over the 1 GiB score tensor; the softmax alone is its "
                                     "lower bound"}
        smr = {}
        for t in (0, 64, 128):
            ms_ = call_ms(f"softmax_fused_T{t}")
            b_ = gmap[f"softmax_fused_T{t}"].units
            smr[f"fused_T{t}"] = {"us": round(ms_ * 1e3, 1), "bytes": b_, "GBs": round(b_ / ms_ / 1e6, 1),
                                  "frac_hbm": round(b_ / ms_ / 1e6 / peaks["hbm_gbs"], 4)}
        mu = call_ms("softmax_unfused")
        bu = gmap["softmax_unfused"].units
        smr["unfused"] = {"us": round(mu * 1e3, 1), "bytes": bu, "GBs": round(bu / mu / 1e6, 1)}
        smr["speedup_fused_T0"] = round(mu / call_ms("softmax_fused_T0"), 3)
        smr["speedup_fused_T64"] = round(mu / call_ms("softmax_fused_T64"), 3)
        rows["causal_softmax"] = smr
        gm = {}
        for M in wl.GEMM_MS:
            fus = call_ms(f"gemm_M{M}_[4]")
            ent = {"[4]_us": round(fus * 1e3, 2), "[4]_TFLOPs": round(flops[M] / fus / 1e9, 1),
                   "[4]_ledger_GBs": round(fc.fuse_gemm_bytes(M, gN, gK, 0) / fus / 1e6, 1)}
            for p_, m_ in plans.items():
                if m_ == 0:
                    continue
                u = call_ms(f"gemm_M{M}_{p_}")
                ent[f"{p_}_us"] = round(u * 1e3, 2)
                ent[f"speedup_[4]_vs_{p_}"] = round(u / fus, 3)
            gm[f"M{M}"] = ent
        gm["M4096"]["roofline"] = roofline_of("gemm_M4096_fused")
        gm["M16"]["roofline"] = roofline_of("gemm_M16_fused")
        gm["M16"]["static_weight_flag"] = "FUSE_GEMM_STATIC_B on every M = 16 group but one"
        gm["M16"]["[4]_no_static_flag_us"] = round(call_ms("gemm_M16_[4]_nostatic") * 1e3, 2)
        rows["gemm_epilogue"] = gm
        rows["launch_graph"] = launch_graph_rows(fc, lib, wl, torch, dev, gemm_bufs[16], check)
        rows["planner"] = planner_rows(fc, wl, peaks, rows["launch_graph"]["t_exec_queued_us"],
                                       {M: {p_: call_ms(f"gemm_M{M}_{p_}") for p_ in plans} for M in wl.GEMM_MS},
                                       plans)
    rows["per_call"] = per_call_rows(torch, stream, {K: chain(K, fc.FUSE_FUSED) for K in KS},
                                     {K: chain(K, fc.FUSE_UNFUSED) for K in KS})

    # same-size copy reference: cudaMemcpy D2D of one chain operand (64 MiB) -- the practical roof
    # for a 2 x 64 MiB streaming kernel at this size (the measured peak is a 2 GiB copy), timed
    # like the groups (back to back between one event pair)
    with torch.cuda.stream(stream):
        for i in range(5):
            ys[i % R].copy_(xs[(i + 1) % R])
        cts = []
        for rep in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(4):
                ys[i % R].copy_(xs[(i + 1) % R])
            e1.record(stream)
            cts.append((e0, e1))
    torch.cuda.synchronize()
    copy_us = float(np.median([e0.elapsed_time(e1) for e0, e1 in cts])) / 4 * 1e3
    rows["chain"]["copy_reference"] = {"us": round(copy_us, 2),
                                       "GBs": round(chain_bytes / copy_us / 1e3, 1),
                                       "what": "cudaMemcpy D2D of 64 MiB, same rotation, back to back"}

    # dense fp16 and bf16 tensor peaks measured in this run the way the pool's bf16 figure was
    # (cuBLAS through torch.matmul, 8192^3, best of 10): the GEMM chain computes in fp16
    if args.rows == "all":
        tp = tensor_peaks(torch, dev, stream)
        rows["tensor_peaks_in_run"] = tp
        for key in ("M4096",):
            r4 = rows["gemm_epilogue"][key]["roofline"]
            r4["frac_of_fp16_in_run"] = round(r4["achieved"] / tp["fp16_tflops"], 4)
            r4["fp16_peak_in_run"] = tp["fp16_tflops"]

    # register / occupancy report of every kernel variant ([K4] §③, [C05] §6.2)
    report_rows = []
    for i in range(fc.fuse_kernel_count()):
        r_ = fc.fuse_kernel_report(i)
        report_rows.append({k: r_[k] for k in ("name", "regs_per_thread", "local_bytes_per_thread",
                                               "dynamic_smem_bytes", "block_threads", "blocks_per_sm",
                                               "cluster_size", "max_active_clusters", "blocks_per_sm_api",
                                               "tmem_cols", "ptxas_registers",
                                               "stack_bytes", "spill_store_bytes", "spill_load_bytes")})
    rows["kernel_report"] = report_rows

    # ---------------------------------------------------------------- e2e through host buffers
    e2e = run_e2e(args, fc, lib, wl, stage_sets, N, KS, chain_bytes, dev, stream, world)
    e2e["_elapsed"] = max_over_ranks([e2e["_elapsed"]], world, dev)[0]
    e2e_value = weak_scaling_gbs(e2e["_bytes"], world, e2e["_elapsed"])

    report = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(wl, seconds=10.0)
            if args.rows == "all":
                rows["cpu_baselines"] = cpu_baselines_per_config(wl)
        report = {
            "metric": "fused-chain HBM GB/s and % of GB300 peak; fused/unfused speedup vs K",
            "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "pointwise chain fp32 N=16,777,216, K in {2,3,4,6,8}, "
                                   "a_s~U[0.9,1.1], b_s~U[-0.1,0.1], ReLU on even s",
                       "N": N, "K": list(KS),
                       "step": "all rows" if args.rows == "all" else "chain rows",
                       "l2": "inputs larger than L2 or rotated (chain: 4 x/y pairs = 512 MiB; RMSNorm: "
                             "8 pairs = 512 MiB; residual add + RMSNorm: 4 sets = 512 MiB; decode GEMM: "
                             "4 weight copies); each group led by an untimed same-kind call; timed calls "
                             "back to back between one CUDA event pair",
                       "parallelism": f"replicas x{world}"},
            "frac_of_peak": round(value / world / peaks["hbm_gbs"], 4),
            "frac_of_nominal": round(value / world / NOMINAL_HBM_GBS, 4),
            "nominal_hbm_gbs": NOMINAL_HBM_GBS,
            "roofline": roofline,
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                    "path": f"fuse_chain_run_host (C ABI, pinned host x and y, {e2e['slices']} slices per call)"},
            "gpu_launches": timed_launches,
            "clocks": clocks,
            "rows": rows,
            "cpu_baseline": cpu,
        }
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return report


def tensor_peaks(torch, dev, stream, n=8192, reps=10):
    """Dense fp16 and bf16 GEMM throughput of cuBLAS (torch.matmul, n^3, best of `reps`)."""
    out = {"what": f"torch.matmul {n}^3 (cuBLAS), best of {reps}, CUDA events on the launching stream"}
    with torch.cuda.stream(stream):
        for name, dt in (("fp16", torch.float16), ("bf16", torch.bfloat16)):
            a = torch.randn(n, n, device=dev, dtype=dt)
            b = torch.randn(n, n, device=dev, dtype=dt)
            for _ in range(3):
                torch.matmul(a, b)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for e0, e1 in ev:
                e0.record(stream)
                torch.matmul(a, b)
                e1.record(stream)
            torch.cuda.synchronize()
            best = min(e0.elapsed_time(e1) for e0, e1 in ev) / 1e3
            out[f"{name}_tflops"] = round(2 * n ** 3 / best / 1e12, 1)
            del a, b
    out["fp16_over_bf16"] = round(out["fp16_tflops"] / out["bf16_tflops"], 4)
    return out


def per_call_rows(torch, stream, fused, unfused, reps=10):
    """The chain sweep with one CUDA event pair around every single call (after the timed region):
    per K the median call time fused and unfused and their ratio.  An event between every two
    calls adds the event's own cost to each call, so these times sit a little above the groups'."""
    def med_us(fn):
        with torch.cuda.stream(stream):
            fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for e0, e1 in ev:
                e0.record(stream)
                fn()
                e1.record(stream)
        torch.cuda.synchronize()
        return float(np.median([e0.elapsed_time(e1) for e0, e1 in ev])) * 1e3
    out = {}
    for K in fused:
        f, u = med_us(fused[K]), med_us(unfused[K])
        out[str(K)] = {"fused_us": round(f, 2), "unfused_us": round(u, 2), "speedup": round(u / f, 3)}
    return {"what": "chain sweep, one event pair per call, median of %d calls" % reps, "per_K": out}


def launch_graph_rows(fc, lib, wl, torch, dev, gemm16, check):
    """Eager vs CUDA-graph replay of the launch-bound cases ("AIGC fundamentals | operator fusion
    and CUDA Graph" §3.4): the 8-stage affine chain on 4096 elements and the M = 16 GEMM plans.
    Each case starts on an idle GPU (synchronize, then events around the submission), so host
    submission cost shows as it does for a lone call.  Measured outside the timed step."""
    import ctypes
    s = torch.cuda.Stream(device=dev)
    sh = s.cuda_stream
    relu, a, b, x0 = wl.affine_chain()
    st = fc._stages([(fc.FUSE_OP_AFFINE_RELU if r_ else fc.FUSE_OP_AFFINE, p, q)
                     for r_, p, q in zip(relu, a, b)])
    K, n = len(a), x0.size
    x = torch.from_numpy(x0).to(dev)
    y = torch.empty_like(x)
    A, Bs, bias, Rr, Ys, _, _, _ = gemm16

    def chain(mode, xx=x, yy=y):
        return lambda: check(lib.fuse_chain_run(st, K, xx.data_ptr(), yy.data_ptr(), n, fc.FUSE_F32,
                                                mode, sh), "fuse_chain_run")

    def gemm(mask):
        return lambda: check(lib.fuse_gemm_epilogue_plan(A.data_ptr(), Bs[0].data_ptr(), bias.data_ptr(),
                                                         Rr.data_ptr(), Ys[0].data_ptr(), 16, wl.GEMM_N,
                                                         wl.GEMM_K, mask, sh), "fuse_gemm_epilogue_plan")

    def capture(fn):
        check(lib.fuse_graph_begin(sh), "fuse_graph_begin")
        try:
            fn()
        finally:
            g = ctypes.c_void_p()
            rc = lib.fuse_graph_end(sh, ctypes.byref(g))
        check(rc, "fuse_graph_end")
        return g.value

    def idle_start_us(fn, reps=60):
        e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for _ in range(5):
            fn()
        s.synchronize()
        for e0, e1 in e:
            s.synchronize()
            e0.record(s)
            fn()
            e1.record(s)
        s.synchronize()
        return float(np.median([e0.elapsed_time(e1) for e0, e1 in e])) * 1e3

    graphs = []
    try:
        cases = {"affine_K8_N4096": {"fused": chain(fc.FUSE_FUSED), "unfused": chain(fc.FUSE_UNFUSED)},
                 "gemm_M16": {"[4]": gemm(0), "[1,1,1,1]": gemm(7)}}
        out = {}
        for cname, plans in cases.items():
            ent = {}
            for pname, fn in plans.items():
                g = capture(fn)
                graphs.append(g)
                ent[f"{pname}_eager_us"] = round(idle_start_us(fn), 2)
                ent[f"{pname}_graph_us"] = round(idle_start_us(
                    lambda g=g: check(lib.fuse_graph_launch(g, sh), "fuse_graph_launch")), 2)
                ent[f"{pname}_kernels"] = lib.fuse_graph_kernel_count(g)
                ent[f"{pname}_graph_speedup"] = round(ent[f"{pname}_eager_us"] / ent[f"{pname}_graph_us"], 3)
            out[cname] = ent
        # the model's inputs, measured: the host cost of one submission through the C ABI (ctypes
        # call included) for a kernel and for a graph, and the GPU's cost per kernel when kernels
        # are queued behind other work, eager and as graph nodes
        small = chain(fc.FUSE_FUSED)
        nq = 64
        g64 = capture(lambda: [small() for _ in range(nq)])
        graphs.append(g64)
        g1 = capture(small)
        graphs.append(g1)

        def host_us(fn, reps=2000):
            s.synchronize()
            t0 = time.perf_counter()
            for _ in range(reps):
                fn()
            t = (time.perf_counter() - t0) / reps * 1e6
            s.synchronize()
            return t

        t_launch = host_us(small)
        t_launch_graph = host_us(lambda: check(lib.fuse_graph_launch(g1, sh), "fuse_graph_launch"))
        big = torch.empty(1 << 26, dtype=torch.float32, device=dev)

        def queued_us(fn_many):
            ts = []
            for _ in range(10):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(s):
                    for _ in range(6):
                        big.mul_(1.0)      # ~0.5 ms of HBM work, so the submissions get ahead
                e0.record(s)
                fn_many()
                e1.record(s)
                s.synchronize()
                ts.append(e0.elapsed_time(e1))
            return float(np.median(ts)) * 1e3

        t_exec = queued_us(lambda: [small() for _ in range(nq)]) / nq
        t_node = queued_us(lambda: check(lib.fuse_graph_launch(g64, sh), "fuse_graph_launch")) / nq
        ach = out["affine_K8_N4096"]
        eager = fc.fuse_launch_model(K, t_launch, t_exec, 0.0)["eager"]
        graph = fc.fuse_launch_model(K, t_launch_graph, t_node, 0.0)["graph"]
        out.update({"t_launch_us": round(t_launch, 3), "t_launch_graph_us": round(t_launch_graph, 3),
                    "t_exec_queued_us": round(t_exec, 3), "t_node_queued_us": round(t_node, 3),
                    "t_dispatch_us": round(t_node - t_exec, 3),
                    "model_unfused_K8": {"eager_us": round(eager, 2), "graph_us": round(graph, 2),
                                         "measured_eager_us": ach["unfused_eager_us"],
                                         "measured_graph_us": ach["unfused_graph_us"]}})
        del big
        return out
    finally:
        for g in graphs:
            lib.fuse_graph_destroy(g)


def planner_rows(fc, wl, peaks, launch_us, measured_ms, plans):
    """The [K4] cost model with this GPU's constants (measured HBM copy bandwidth and bf16 dense
    peak, the measured back-to-back kernel cost as the launch term) against the measured time of
    every GEMM plan: does it pick the plan that is fastest?"""
    model = dict(hbm_bytes_per_s=peaks["hbm_gbs"] * 1e9, flops_per_s=peaks["bf16_tflops"] * 1e12,
                 launch_s=launch_us * 1e-6, spill_penalty=3.0, reg_limit=255)
    out = {"model": {k: (round(v, 9) if isinstance(v, float) else v) for k, v in model.items()}}
    N, Kd = wl.GEMM_N, wl.GEMM_K
    for M in wl.GEMM_MS:
        st = [dict(op=0, a=0, b=0, writes=M * N, ext_reads=M * Kd + Kd * N, flops=2 * M * N * Kd, live_regs=128),
              dict(op=0, a=0, b=0, writes=M * N, ext_reads=N, flops=M * N, live_regs=8),
              dict(op=0, a=0, b=0, writes=M * N, ext_reads=0, flops=8 * M * N, live_regs=0),
              dict(op=0, a=0, b=0, writes=M * N, ext_reads=M * N, flops=M * N, live_regs=24)]
        pred = {p_: fc.fuse_plan_time(st, m_, 2, model) * 1e6 for p_, m_ in plans.items()}
        meas = {p_: measured_ms[M][p_] * 1e3 for p_ in plans}
        best_mask, _ = fc.fuse_best_plan(st, 2, model)
        best_pred = [p_ for p_, m_ in plans.items() if m_ == best_mask]
        out[f"M{M}"] = {"predicted_us": {k: round(v, 2) for k, v in pred.items()},
                        "measured_us": {k: round(v, 2) for k, v in meas.items()},
                        "best_plan_predicted": best_pred[0] if best_pred else f"mask {best_mask}",
                        "best_plan_measured": min(meas, key=meas.get),
                        "order_predicted": sorted(pred, key=pred.get),
                        "order_measured": sorted(meas, key=meas.get)}
    return out


def run_e2e(args, fc, lib, wl, stage_sets, N, KS, chain_bytes, dev, stream, world, slices=8):
    """Per K: the fused chain through the C ABI's host-buffer entry point, fuse_chain_run_host():
    x from pinned host memory, y back to pinned host memory, through device scratch the caller
    owns.  The library cuts each call into `slices` pieces whose copies in (one helper stream),
    kernels (the caller's stream) and copies out (a second helper stream) overlap.  Bytes moved
    per step: x in and y out once per K."""
    import torch
    hx = torch.from_numpy(wl.chain_input(N, salt=7)).pin_memory()
    hy = torch.empty(N, dtype=torch.float32).pin_memory()
    dx = torch.empty(N, dtype=torch.float32, device=dev)
    dy = torch.empty(N, dtype=torch.float32, device=dev)
    sh = stream.cuda_stream

    def one_step():
        for K in KS:
            rc = lib.fuse_chain_run_host(stage_sets[K], K, hx.data_ptr(), hy.data_ptr(), N, fc.FUSE_F32,
                                         fc.FUSE_FUSED, dx.data_ptr(), dy.data_ptr(), slices, sh)
            if rc != 0:
                raise fc.FuseError(rc, "fuse_chain_run_host")

    for _ in range(2):
        one_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(3, min(args.steps, 10))
    e0.record(stream)
    for _ in range(steps):
        one_step()
    e1.record(stream)
    torch.cuda.synchronize()
    # the sliced, pipelined call must give what one device call on the whole vector gives
    with torch.cuda.stream(stream):
        rc = lib.fuse_chain_run(stage_sets[KS[-1]], KS[-1], dx.data_ptr(), dy.data_ptr(), N, fc.FUSE_F32,
                                fc.FUSE_FUSED, sh)
        if rc != 0:
            raise fc.FuseError(rc, "fuse_chain_run")
    torch.cuda.synchronize()
    if not torch.equal(hy.to(dev), dy):
        raise RuntimeError("e2e: the host-buffer call differs from the whole-vector device call")
    elapsed = e0.elapsed_time(e1) / 1e3
    return {"_elapsed": elapsed, "_bytes": steps * len(KS) * chain_bytes,
            "h2d": len(KS) * N * 4, "d2h": len(KS) * N * 4, "slices": slices}


# ------------------------------------------------------------------------------ oracle arms
def cpu_baseline(wl, seconds=10.0):
    """The plain CPU oracle (single thread), as it stands, on the same chain workload: whole K
    sweeps over the full N = 16,777,216 elements, repeated until ~`seconds` of CPU time."""
    import oracle
    x = wl.chain_input(wl.CHAIN_N, salt=0)
    stages = {K: wl.chain_stages(K) for K in wl.CHAIN_KS}
    nbytes, t_total, sweeps = 0, 0.0, 0
    while t_total < seconds or sweeps == 0:
        for K in wl.CHAIN_KS:
            relu, a, b = stages[K]
            t0 = time.perf_counter()
            oracle.chain(relu, a, b, x)
            t_total += time.perf_counter() - t0
            nbytes += 2 * wl.CHAIN_N * 4
        sweeps += 1
    return {"value": round(nbytes / t_total / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "host_cores_available": _host_cores(),
            "sample": f"{sweeps} full K-sweeps (K=2,3,4,6,8) over N=16,777,216 fp32, single thread, "
                      f"{t_total:.1f} s"}


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baselines_per_config(wl, seconds=2.0):
    """Every other config's oracle, as it stands (single thread), on a bounded sample of its
    workload, each rate in its row's own unit.  A baseline, not a target."""
    import oracle

    def timed(fn):
        n, t = 0, 0.0
        while t < seconds or n == 0:
            t0 = time.perf_counter()
            fn()
            t += time.perf_counter() - t0
            n += 1
        return n, t

    def row(value, unit, sample):
        return {"value": value, "unit": unit, "cores": 1, "kind": "oracle", "sample": sample}

    out = {"host_cores_available": _host_cores(), "threads_used": 1}
    x, w = wl.rmsnorm_input()
    n, t = timed(lambda: oracle.rmsnorm(x, w, wl.RMS_EPS))
    b = 2 * x.size * 4 + x.shape[1] * 4
    out["rmsnorm"] = row(round(b * n / t / 1e9, 3), "GB/s",
                         f"{n} calls on the full [{x.shape[0]}, {x.shape[1]}] fp32, {t:.1f} s")
    sl, S = 2, wl.SM_S
    s_ = wl.softmax_input(sl, S)
    n, t = timed(lambda: oracle.causal_softmax(s_, wl.SM_SCALE))
    b = sl * 2 * S * S * 2
    out["causal_softmax"] = row(round(b * n / t / 1e9, 3), "GB/s",
                                f"{n} calls on {sl} of the 128 [{S}, {S}] bf16 slices (fused ledger "
                                f"2 N b, no skip), {t:.1f} s")
    A, B, bias, R = wl.gemm_input(16)
    n, t = timed(lambda: oracle.gemm_epilogue(A, B, bias, R, 0))
    out["gemm_M16"] = row(round(2 * 16 * wl.GEMM_N * wl.GEMM_K * n / t / 1e12, 6), "TFLOP/s",
                          f"{n} calls of the full 16 x 4096 x 4096 plan [4], {t:.1f} s")
    A, B, bias, R = wl.gemm_input(4096)
    rows_ = np.arange(0, 4096, 512)
    n, t = timed(lambda: oracle.gemm_epilogue(A, B, bias, R, 0, rows=rows_))
    per_row = t / n / rows_.size
    out["gemm_M4096"] = row(round(2 * rows_.size * wl.GEMM_N * wl.GEMM_K * n / t / 1e12, 6), "TFLOP/s",
                            f"{n} calls on {rows_.size} of the 4096 rows of 4096^3 plan [4], {t:.1f} s; "
                            f"the whole problem would take {per_row * 4096:.0f} s")
    q, k, v = wl.attention_input(1, wl.ATT_S, wl.ATT_D)
    arows = np.arange(0, wl.ATT_S, 128) + 127
    n, t = timed(lambda: oracle.attention(q, k, v, wl.ATT_SCALE, rows=arows))
    fl = int(sum(4 * wl.ATT_D * (int(i) + 1) for i in arows))
    out["attention"] = row(round(fl * n / t / 1e12, 6), "TFLOP/s",
                           f"{n} calls on {arows.size} query rows of one [{wl.ATT_S}, {wl.ATT_D}] slice, "
                           f"{t:.1f} s")
    return out


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle timed on the host cores, rank 0 only."""
    if rank != 0:
        return None
    from epilogue_chains_gb300 import workloads as wl
    import oracle
    N = wl.CHAIN_N
    x = wl.chain_input(N, salt=0)
    stages = {K: wl.chain_stages(K) for K in wl.CHAIN_KS}

    def sweep():
        for K in wl.CHAIN_KS:
            relu, a, b = stages[K]
            oracle.chain(relu, a, b, x)

    for _ in range(args.warmup):
        sweep()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sweep()
    dt = time.perf_counter() - t0
    nbytes = args.steps * len(wl.CHAIN_KS) * 2 * N * 4
    value = nbytes / dt / 1e9
    return {"impl": "reference",
            "metric": "fused-chain HBM GB/s and % of GB300 peak; fused/unfused speedup vs K",
            "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": "pointwise chain fp32 N=16,777,216, K in {2,3,4,6,8}, "
                                   "a_s~U[0.9,1.1], b_s~U[-0.1,0.1], ReLU on even s",
                       "N": N, "K": list(wl.CHAIN_KS), "step": "one K sweep"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} full K-sweeps over N=16,777,216, single thread"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_profile(args):
    """A fixed number of calls of one row on cuda:0 and nothing else, for ncu captures."""
    import torch
    import epilogue_chains_gb300 as fc
    from epilogue_chains_gb300 import workloads as wl
    dev = torch.device("cuda:0")
    lib = fc._load()
    stream = torch.cuda.current_stream().cuda_stream
    name, L = args.profile, args.launches
    if name.startswith("chain"):
        n = args.size or wl.CHAIN_N
        relu, a, b = wl.chain_stages(args.K)
        st = fc._stages([(int(r_), float(p_), float(q_)) for r_, p_, q_ in zip(relu, a, b)])
        mode = {"chain_fused": fc.FUSE_FUSED, "chain_unfused": fc.FUSE_UNFUSED,
                "chain_fat": fc.FUSE_FAT}[name]
        xs = [wl.chain_input(n, device=dev, salt=r) for r in range(2)]
        ys = [torch.empty_like(xs[0]) for _ in range(2)]
        for i in range(L):
            rc = lib.fuse_chain_run(st, args.K, xs[i % 2].data_ptr(), ys[i % 2].data_ptr(), n,
                                    fc.FUSE_F32, mode, stream)
            assert rc == 0, fc.fuse_strerror(rc)
        nbytes = fc.fuse_chain_bytes(args.K, n, fc.FUSE_F32, mode)
    elif name.startswith("rmsnorm"):
        rows = args.size or wl.RMS_ROWS
        mode = fc.FUSE_FUSED if name == "rmsnorm_fused" else fc.FUSE_UNFUSED
        x0, w = wl.rmsnorm_input(rows, wl.RMS_HIDDEN, device=dev)
        npairs = 8 if rows <= 4096 else 2     # large sizes: 2 pairs already exceed L2
        xs = [x0] + [x0.clone() for _ in range(npairs - 1)]
        ys = [torch.empty_like(x0) for _ in range(npairs)]
        ws = torch.empty(max(1, fc.fuse_rmsnorm_workspace_bytes(rows, wl.RMS_HIDDEN, mode)),
                         dtype=torch.uint8, device=dev)
        for i in range(L):
            rc = lib.fuse_rmsnorm(xs[i % npairs].data_ptr(), w.data_ptr(), ys[i % npairs].data_ptr(), rows,
                                  wl.RMS_HIDDEN, wl.RMS_EPS, mode, ws.data_ptr(), ws.numel(), stream)
            assert rc == 0, fc.fuse_strerror(rc)
        nbytes = fc.fuse_rmsnorm_bytes(rows, wl.RMS_HIDDEN, mode)
    elif name.startswith("add_rmsnorm"):
        rows = args.size or wl.ADDRMS_ROWS
        mode = fc.FUSE_FUSED if name == "add_rmsnorm_fused" else fc.FUSE_UNFUSED
        x, r, w = wl.add_rmsnorm_input(rows, wl.ADDRMS_HIDDEN, device=dev)
        ns = 4 if rows <= 4096 else 2
        xs, rs = [x] + [x.clone() for _ in range(ns - 1)], [r] + [r.clone() for _ in range(ns - 1)]
        hs, ys = [torch.empty_like(x) for _ in range(ns)], [torch.empty_like(x) for _ in range(ns)]
        ws = torch.empty(max(1, fc.fuse_rmsnorm_workspace_bytes(rows, wl.ADDRMS_HIDDEN, mode)),
                         dtype=torch.uint8, device=dev)
        for i in range(L):
            rc = lib.fuse_add_rmsnorm(xs[i % ns].data_ptr(), rs[i % ns].data_ptr(), w.data_ptr(),
                                      hs[i % ns].data_ptr(), ys[i % ns].data_ptr(), rows, wl.ADDRMS_HIDDEN,
                                      wl.RMS_EPS, mode, ws.data_ptr(), ws.numel(), stream)
            assert rc == 0, fc.fuse_strerror(rc)
        nbytes = fc.fuse_add_rmsnorm_bytes(rows, wl.ADDRMS_HIDDEN, mode)
    elif name.startswith("silu_mul"):
        rows = args.size or wl.SILU_ROWS
        mode = fc.FUSE_FUSED if name == "silu_mul_fused" else fc.FUSE_UNFUSED
        gus = [wl.silu_input(rows, wl.SILU_COLS, device=dev, salt=r_) for r_ in range(2)]
        ys = [torch.empty(rows, wl.SILU_COLS, dtype=gus[0].dtype, device=dev) for _ in range(2)]
        C = wl.SILU_COLS
        for i in range(L):
            base = gus[i % 2].data_ptr()
            rc = lib.fuse_silu_mul(base, base + 2 * C, 2 * C, ys[i % 2].data_ptr(), rows, C,
                                   fc.FUSE_BF16, mode, stream)
            assert rc == 0, fc.fuse_strerror(rc)
        nbytes = fc.fuse_silu_mul_bytes(rows, C, fc.FUSE_BF16, mode)
    elif name == "attention":
        bh = args.size or wl.ATT_BH
        q, k, v = wl.attention_input(bh, wl.ATT_S, wl.ATT_D, device=dev)
        os_ = [torch.empty_like(q) for _ in range(2)]
        for i in range(L):
            rc = lib.fuse_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), os_[i % 2].data_ptr(), bh,
                                    wl.ATT_S, wl.ATT_D, wl.ATT_SCALE, stream)
            assert rc == 0, fc.fuse_strerror(rc)
        nbytes = fc.fuse_attention_bytes(bh, wl.ATT_S, wl.ATT_D)
    elif name == "gemm":
        M = args.size or 4096
        A, B, bias, Rr = wl.gemm_input(M, device=dev)
        # decode shapes rotate six weight copies (192 MiB, beyond L2), as the bench does, and carry
        # FUSE_GEMM_STATIC_B as the bench's decode loop does unless --no-static-b is given
        Bs = [B] + [B.clone() for _ in range(5)] if M <= 64 else [B]
        flags = fc.FUSE_GEMM_STATIC_B if M <= 64 and not args.no_static_b else 0
        Ys = [torch.empty(M, wl.GEMM_N, dtype=torch.float16, device=dev) for _ in range(2)]
        gws = torch.zeros(max(1, fc.fuse_gemm_workspace_bytes(M, wl.GEMM_N, wl.GEMM_K)), dtype=torch.uint8,
                          device=dev)
        for i in range(L):
            rc = lib.fuse_gemm_epilogue_ws(A.data_ptr(), Bs[i % len(Bs)].data_ptr(), bias.data_ptr(), Rr.data_ptr(),
                                           Ys[i % 2].data_ptr(), M, wl.GEMM_N, wl.GEMM_K, args.mask | flags,
                                           gws.data_ptr(), gws.numel(), stream)
            assert rc == 0, fc.fuse_strerror(rc)
        nbytes = fc.fuse_gemm_bytes(M, wl.GEMM_N, wl.GEMM_K, args.mask)
    else:
        bh = args.size or wl.SM_B * wl.SM_H
        S = wl.SM_S
        mode = fc.FUSE_FUSED if name == "softmax_fused" else fc.FUSE_UNFUSED
        tile = args.tile if mode == fc.FUSE_FUSED else 0
        s_ = wl.softmax_input(bh, S, device=dev)
        ps = [torch.empty_like(s_) for _ in range(2)]
        ws = torch.empty(max(1, fc.fuse_causal_softmax_workspace_bytes(bh, S, mode)),
                         dtype=torch.uint8, device=dev)
        for i in range(L):
            rc = lib.fuse_causal_softmax(s_.data_ptr(), ps[i % 2].data_ptr(), bh, S, wl.SM_SCALE,
                                         tile, fc.FUSE_BF16, mode, ws.data_ptr(), ws.numel(), stream)
            assert rc == 0, fc.fuse_strerror(rc)
        nbytes = fc.fuse_causal_softmax_bytes(bh, S, tile, fc.FUSE_BF16, mode)
    torch.cuda.synchronize()
    assert fc.fuse_check() == fc.FUSE_OK
    print(json.dumps({"profile": name, "launches": L, "algorithmic_bytes_per_call": nbytes}))


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.profile:
        run_profile(args)
        return
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
