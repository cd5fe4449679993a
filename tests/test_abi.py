"""C-ABI checks that need no GPU: the library builds and loads, exports every symbol the header
declares, validates arguments on the host, and its byte ledgers reproduce the pages' numbers."""
import ctypes
import os
import re

import pytest

import epilogue_chains_gb300 as fc
from conftest import ROOT, read_golden

HEADER = os.path.join(ROOT, "include", "fusechain.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fuse_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fuse_chain_run", "fuse_rmsnorm", "fuse_causal_softmax", "fuse_ledger",
                     "fuse_kernel_report", "fuse_check", "fuse_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol():
    fc._load()  # builds the library if needed
    lib = ctypes.CDLL(fc.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    assert set(declared_functions()) == set(fc.SIGNATURES)


def test_host_side_validation_needs_no_gpu():
    lib = fc._load()
    st = (fc.fuse_stage * 1)(fc.fuse_stage(0, 1.0, 0.0, 0, 0, 0, 0))
    assert lib.fuse_chain_run(st, 0, None, None, 16, fc.FUSE_F32, fc.FUSE_FUSED, None) == fc.FUSE_EINVAL
    assert lib.fuse_chain_run(st, 33, None, None, 16, fc.FUSE_F32, fc.FUSE_FUSED, None) == fc.FUSE_EINVAL
    assert lib.fuse_chain_run(st, 1, None, None, 0, fc.FUSE_F32, fc.FUSE_FUSED, None) == fc.FUSE_OK
    assert lib.fuse_chain_run(st, 1, None, None, 16, 7, fc.FUSE_FUSED, None) == fc.FUSE_EINVAL
    assert lib.fuse_chain_run(st, 1, None, None, 16, fc.FUSE_F32, 9, None) == fc.FUSE_EINVAL
    assert lib.fuse_chain_run(st, 1, None, None, 16, fc.FUSE_F32, fc.FUSE_FUSED, None) == fc.FUSE_EINVAL
    # partial overlap of x and y is rejected before any launch
    assert lib.fuse_chain_run(st, 1, 0x10000, 0x10004, 16, fc.FUSE_F32, fc.FUSE_FUSED, None) == fc.FUSE_EINVAL
    assert lib.fuse_chain_run(st, 1, 0x10002, 0x20000, 16, fc.FUSE_F32, fc.FUSE_FUSED, None) == fc.FUSE_EALIGN
    assert lib.fuse_rmsnorm(None, None, None, 4, 0, 1e-6, 0, None, 0, None) == fc.FUSE_EINVAL
    assert lib.fuse_rmsnorm(0x1000, 0x2000, 0x3000, 4, 20000, 1e-6, fc.FUSE_FUSED, None, 0,
                            None) == fc.FUSE_EUNSUPPORTED
    assert lib.fuse_rmsnorm(0x1000, 0x2000, 0x3000, 4, 64, 1e-6, fc.FUSE_UNFUSED, None, 0,
                            None) == fc.FUSE_EWORKSPACE
    assert lib.fuse_causal_softmax(0x1000, 0x100000, 1, 16, 0.5, 12, fc.FUSE_BF16, 0, None, 0,
                                   None) == fc.FUSE_EINVAL           # tile not a multiple of 16
    assert lib.fuse_causal_softmax(0x1000, 0x100000, 1, 16, 0.5, 64, fc.FUSE_BF16,
                                   fc.FUSE_UNFUSED, None, 0, None) == fc.FUSE_EUNSUPPORTED
    assert lib.fuse_causal_softmax(0x1000, 0x1000, 1, 16, 0.5, 0, fc.FUSE_BF16, fc.FUSE_FUSED,
                                   None, 0, None) == fc.FUSE_EINVAL  # s and p overlap
    assert fc.fuse_strerror(fc.FUSE_ETIMEOUT).startswith("bounded device wait")


# ------------------------------------------------------------------------------ ptxas table
def _entries(table, stem):
    return [r for r in table if stem in r["symbol"]]


def test_ptxas_table_covers_every_kernel_family_without_spills():
    """[K4] §③ / [C05] §6.2: spill bytes are the signal that a fused kernel has outgrown the
    register file.  The table is the build's own ptxas -v output, read without a GPU."""
    table = fc.fuse_ptxas_table()
    assert len(table) == fc._load().fuse_ptxas_count() > 0
    for stem in ("chain_fused_kernel", "chain_stage_kernel", "chain_fat_kernel", "rmsnorm_row_kernel",
                 "rms_square_kernel", "rms_rowmean_kernel", "rms_scale_kernel", "rms_weight_kernel",
                 "softmax_fused_kernel", "sm_rowmax_kernel", "sm_sub_kernel", "sm_exp_kernel",
                 "sm_rowsum_kernel", "sm_div_kernel", "gemm_tc_kernel", "gemm_decode_kernel",
                 "epi_tail_kernel", "attn_persist_kernel", "silu_mul_vec_kernel", "residual_add_kernel"):
        rows = _entries(table, stem)
        assert rows, stem
        for r in rows:
            assert r["registers"] > 0, r
            assert r["spill_store_bytes"] == 0 and r["spill_load_bytes"] == 0, r
            assert r["stack_bytes"] == 0, r
    with pytest.raises(fc.FuseError):
        fc._check(fc._load().fuse_ptxas_entry(len(table), ctypes.byref(fc.fuse_ptxas_record())), "entry")
    assert fc._load().fuse_ptxas_entry(0, None) == fc.FUSE_EINVAL


def _blocks_per_sm_by_registers(regs, threads=256):
    # registers are granted per warp in units of 256 (a per-thread count rounded up to 8); 64 Ki
    # registers, 2048 threads and 32 blocks per SM
    per_warp = -(-regs * 32 // 256) * 256
    return min(65536 // (per_warp * (threads // 32)), 2048 // threads, 32)


def test_fat_probe_collapses_occupancy_in_the_ptxas_figures():
    """[C05] §6.2: 48 live temporaries per element push the fat kernel's registers so high that
    one 256-thread block fits an SM, where the thin fused kernel keeps the SM full."""
    table = fc.fuse_ptxas_table()
    fat = [r for r in _entries(table, "chain_fat_kernel") if "kernelIf" in r["symbol"]]
    fused = [r for r in _entries(table, "chain_fused_kernel") if "kernelIf" in r["symbol"]]
    assert len(fat) == 1 and len(fused) == 1
    assert fat[0]["registers"] >= 192
    assert _blocks_per_sm_by_registers(fat[0]["registers"]) == 1
    assert _blocks_per_sm_by_registers(fused[0]["registers"]) == 8


# ------------------------------------------------------------------------------ ledgers
def mlp_epilogue_stages(M, N, K):
    """[K4] §① chain_mlp_epilogue: mm -> +bias -> GELU -> +residual."""
    return [
        dict(op=0, a=0, b=0, writes=M * N, ext_reads=M * K + K * N, flops=2 * M * N * K, live_regs=128),
        dict(op=0, a=0, b=0, writes=M * N, ext_reads=N, flops=M * N, live_regs=8),
        dict(op=0, a=0, b=0, writes=M * N, ext_reads=0, flops=8 * M * N, live_regs=0),
        dict(op=0, a=0, b=0, writes=M * N, ext_reads=M * N, flops=M * N, live_regs=24),
    ]


def test_gemm_chain_ledger_matches_printed_bytes_and_launches():
    st = mlp_epilogue_stages(4096, 4096, 4096)
    for plan, mask, nbytes, launches in read_golden("k4_ledger_bytes.txt"):
        led = fc.fuse_ledger(st, int(mask), 2)
        assert led["bytes"] == int(nbytes), plan
        assert led["launches"] == int(launches), plan


def test_gemm_chain_register_peaks_follow_the_table():
    """[K4] §① table prints register peaks 128 / 128 / 136 / 160 for the four plans; the
    per-stage live_regs are not printed, mm=128, bias=8, gelu=0, res=24 reproduce all four."""
    st = mlp_epilogue_stages(4096, 4096, 4096)
    peaks = {7: 128, 1: 128, 2: 136, 0: 160}
    for mask, peak in peaks.items():
        assert fc.fuse_ledger(st, mask, 2)["reg_peak"] == peak


def test_equal_bytes_of_the_two_single_cut_plans():
    """[K4] self-check: [1,3] and [2,2] both round-trip exactly one MN intermediate."""
    for M in (16, 128, 4096):
        st = mlp_epilogue_stages(M, 4096, 4096)
        assert fc.fuse_ledger(st, 1, 2)["bytes"] == fc.fuse_ledger(st, 2, 2)["bytes"]
        diff = fc.fuse_ledger(st, 1, 2)["bytes"] - fc.fuse_ledger(st, 0, 2)["bytes"]
        assert diff == 2 * M * 4096 * 2


def test_decode_shape_ledger():
    st = mlp_epilogue_stages(16, 4096, 4096)
    assert fc.fuse_ledger(st, 0, 2)["bytes"] == 33_955_840
    assert fc.fuse_ledger(st, 7, 2)["bytes"] == 34_742_272


def test_heavy_counterexample_bytes():
    """[K4] §③: a(live 200) + b(live 100) at n = 2^26: [1,1] moves 4n*2 B, [2] moves 2n*2 B but
    its register sum 300 exceeds 255."""
    n = 1 << 26
    heavy = [dict(op=0, a=0, b=0, writes=n, ext_reads=n, flops=n, live_regs=200),
             dict(op=0, a=0, b=0, writes=n, ext_reads=0, flops=n, live_regs=100)]
    split, fused = fc.fuse_ledger(heavy, 1, 2), fc.fuse_ledger(heavy, 0, 2)
    assert split["bytes"] == 4 * n * 2 and fused["bytes"] == 2 * n * 2
    assert split["reg_peak"] == 200 and fused["reg_peak"] == 300


def test_ledger_rejects_mask_bits_past_the_last_boundary():
    st = mlp_epilogue_stages(16, 16, 16)
    out = fc.fuse_ledger_t()
    arr = fc._stages(st)
    assert fc._load().fuse_ledger(arr, 4, 8, 2, ctypes.byref(out)) == fc.FUSE_EINVAL


def test_byte_ledgers_match_printed_mib_and_gib():
    g = {k: float(v) for k, v in read_golden("ofcg_byte_ledger.txt")}
    MiB, GiB = 2.0 ** 20, 2.0 ** 30
    n = 4_000_000
    assert f"{fc.fuse_chain_bytes(8, n, fc.FUSE_F32, fc.FUSE_UNFUSED) / MiB:.1f}" == f"{g['chain_unfused_MiB']:.1f}"
    assert f"{fc.fuse_chain_bytes(8, n, fc.FUSE_F32, fc.FUSE_FUSED) / MiB:.1f}" == f"{g['chain_fused_MiB']:.1f}"
    # chain ledger through the generic stage ledger: x read by stage 0, every stage writes n
    st = [dict(op=0, a=1, b=0, writes=n, ext_reads=n if s == 0 else 0, flops=2 * n, live_regs=0)
          for s in range(8)]
    assert fc.fuse_ledger(st, 0x7F, 4)["bytes"] == fc.fuse_chain_bytes(8, n, fc.FUSE_F32, fc.FUSE_UNFUSED)
    assert fc.fuse_ledger(st, 0, 4)["bytes"] == fc.fuse_chain_bytes(8, n, fc.FUSE_F32, fc.FUSE_FUSED)
    # RMSNorm fused: one read + one write of the tensor (+ the weight row)
    assert f"{fc.fuse_rmsnorm_bytes(1000, 4000, fc.FUSE_FUSED) / MiB:.1f}" == f"{g['rmsnorm_fused_MiB']:.1f}"
    # softmax over [8,16,2048,2048] bf16: 8 copies unfused, 2 fused (row statistics are extra)
    bh, S = 8 * 16, 2048
    unf = fc.fuse_causal_softmax_bytes(bh, S, 0, fc.FUSE_BF16, fc.FUSE_UNFUSED)
    fus = fc.fuse_causal_softmax_bytes(bh, S, 0, fc.FUSE_BF16, fc.FUSE_FUSED)
    assert f"{fus / GiB:.3f}" == f"{g['softmax_fused_GiB']:.3f}"
    assert f"{(unf - 4 * bh * S * 4) / GiB:.3f}" == f"{g['softmax_unfused_GiB']:.3f}"
    assert f"{bh * S * S * 2 / GiB:.3f}" == f"{g['softmax_mask_GiB']:.3f}"


def test_causal_block_skip_reads_the_kept_fraction():
    """§3.5: with tile T the read volume is (n_b + 1)/(2 n_b) of the scores, n_b = S/T."""
    g = {k: float(v) for k, v in read_golden("ofcg_byte_ledger.txt")}
    bh, S = 8 * 16, 2048
    write = bh * S * S * 2
    for T, key in ((64, "kept_block64_pct"), (128, "kept_block128_pct"), (256, "kept_block256_pct")):
        read = fc.fuse_causal_softmax_bytes(bh, S, T, fc.FUSE_BF16, fc.FUSE_FUSED) - write
        frac = read / (bh * S * S * 2)
        nb = S // T
        assert frac == (nb + 1) / (2 * nb)
        assert f"{100 * frac:.1f}" == f"{g[key]:.1f}"
    assert f"{100 * (S + 1) / (2 * S):.1f}" == f"{g['kept_exact_pct']:.1f}"
    assert fc.fuse_causal_softmax_bytes(bh, S, 64, fc.FUSE_BF16, fc.FUSE_FUSED) == 1_627_389_952
    assert fc.fuse_causal_softmax_bytes(bh, S, 128, fc.FUSE_BF16, fc.FUSE_FUSED) == 1_644_167_168


def test_gemm_bytes_match_printed_plan_ledger():
    """fuse_gemm_bytes() (the kernels' DRAM traffic) equals [K4] §①'s four printed integers."""
    for plan, mask, nbytes, launches in read_golden("k4_ledger_bytes.txt"):
        assert fc.fuse_gemm_bytes(4096, 4096, 4096, int(mask)) == int(nbytes), plan
    st = mlp_epilogue_stages(16, 4096, 4096)
    for mask in range(8):
        assert fc.fuse_gemm_bytes(16, 4096, 4096, mask) == fc.fuse_ledger(st, mask, 2)["bytes"]


def test_gemm_host_validation():
    lib = fc._load()
    assert lib.fuse_gemm_epilogue_plan(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 64, 60, 64, 0,
                                       None) == fc.FUSE_EALIGN      # N % 8
    assert lib.fuse_gemm_epilogue_plan(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 64, 64, 60, 0,
                                       None) == fc.FUSE_EALIGN      # K % 8
    assert lib.fuse_gemm_epilogue_plan(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 64, 64, 64, 8,
                                       None) == fc.FUSE_EINVAL      # mask beyond 3 cuts
    assert lib.fuse_gemm_epilogue_plan(0x1000, 0x2000, 0x3000, 0x4000, 0x4000, 64, 64, 64, 0,
                                       None) == fc.FUSE_EINVAL      # Y overlaps R
    assert lib.fuse_gemm_epilogue_plan(0x1008, 0x2000, 0x3000, 0x4000, 0x9000, 64, 64, 64, 0,
                                       None) == fc.FUSE_EALIGN      # A not 16-byte aligned
    assert lib.fuse_gemm_epilogue_plan(None, None, None, None, None, 0, 64, 64, 0, None) == fc.FUSE_OK
    # the static-weight flag is the only bit accepted beside the plan's three
    assert lib.fuse_gemm_epilogue_plan(None, None, None, None, None, 0, 64, 64,
                                       fc.FUSE_GEMM_STATIC_B | 7, None) == fc.FUSE_OK
    assert lib.fuse_gemm_epilogue_plan(0x1000, 0x2000, 0x3000, 0x4000, 0x9000, 16, 64, 64,
                                       0x200, None) == fc.FUSE_EINVAL
    hdr = open(HEADER).read()
    assert re.search(r"#define FUSE_GEMM_STATIC_B 0x100u", hdr) and fc.FUSE_GEMM_STATIC_B == 0x100


def test_gemm_workspace_bytes_is_host_arithmetic():
    """The split-K workspace size needs no GPU: a 2 KB header of ticket and full words plus one
    512 KB fp32 partial tile per CTA pair tile (two K halves x two CTAs x 128 x 256), for at most
    64 tiles; none for the decode shapes."""
    assert fc.fuse_gemm_workspace_bytes(16, 4096, 4096) == 0
    assert fc.fuse_gemm_workspace_bytes(64, 4096, 4096) == 0
    assert fc.fuse_gemm_workspace_bytes(256, 256, 64) == 2048 + 1 * 4 * 128 * 256 * 4
    assert fc.fuse_gemm_workspace_bytes(2560, 2048, 128) == 2048 + 64 * 4 * 128 * 256 * 4
    assert fc.fuse_gemm_workspace_bytes(4096, 4096, 4096) == 2048 + 64 * 4 * 128 * 256 * 4
