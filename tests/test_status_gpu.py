"""Watchdog and kernel report on the GPU.

The watchdog test makes a bounded wait run out on purpose: one thread waits on an mbarrier that
nothing arrives on, gives up after a short budget, records the timeout and returns.  Nothing
faults or traps; the context stays usable, which the follow-up chain call checks."""
import numpy as np
import pytest

import epilogue_chains_gb300 as fc
import oracle
from epilogue_chains_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_device):
    import torch
    assert fc.fuse_check() == fc.FUSE_OK
    fc.fuse_debug_expire_wait(2_000_000)          # ~1 ms of SM clocks
    assert fc.fuse_check() == fc.FUSE_ETIMEOUT
    assert fc.fuse_check() == fc.FUSE_OK          # the flag is cleared once reported
    relu, a, b = wl.chain_stages(4)
    x = wl.chain_input(4096, salt=1)
    y = torch.empty(4096, device="cuda")
    fc.fuse_chain_run([(int(r), float(p), float(q)) for r, p, q in zip(relu, a, b)],
                      torch.from_numpy(x).cuda(), y)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), oracle.chain(relu, a, b, x))


def test_kernel_report_covers_every_variant(cuda_device):
    n = fc.fuse_kernel_count()
    assert n >= 10
    for i in range(n):
        r = fc.fuse_kernel_report(i)
        assert r["regs_per_thread"] > 0 and r["blocks_per_sm"] >= 1, r
        assert r["blocks_per_sm_api"] >= 1, r
    with pytest.raises(fc.FuseError):
        fc.fuse_kernel_report(n)


def test_decode_gemm_grid_is_resident_in_one_wave(cuda_device):
    """The decode GEMM's 83 KB of shared memory and 32 tensor-memory columns let two CTAs share an
    SM, so the 256 CTAs of N = 4096 (32 clusters of 8) fit the 152 SMs at once; the tcgen05 GEMM
    and attention kernels hold one CTA per SM."""
    recs = {fc.fuse_kernel_report(i)["name"].split(" ")[0]: fc.fuse_kernel_report(i)
            for i in range(fc.fuse_kernel_count())}
    dec = recs["gemm_decode_kernel<16>"]
    assert dec["tmem_cols"] == 32 and dec["blocks_per_sm"] == 2, dec
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert dec["blocks_per_sm"] * sms >= 256
    for name in ("gemm_tc_kernel", "attn_persist_kernel<D=256>"):
        assert recs[name]["blocks_per_sm"] == 1 and recs[name]["tmem_cols"] == 512, recs[name]


def test_kernel_report_carries_the_ptxas_figures_of_its_build(cuda_device):
    """Every reported kernel is found, by its device symbol, in the ptxas -v table the build
    linked in; ptxas's register count is the one the runtime reports; no kernel spills."""
    table = {r["symbol"]: r for r in fc.fuse_ptxas_table()}
    for i in range(fc.fuse_kernel_count()):
        r = fc.fuse_kernel_report(i)
        assert r["symbol"] in table, r["name"]
        t = table[r["symbol"]]
        assert r["ptxas_registers"] == t["registers"] == r["regs_per_thread"], r["name"]
        assert r["spill_store_bytes"] == 0 and r["spill_load_bytes"] == 0, r["name"]
        assert r["stack_bytes"] == 0 and r["local_bytes_per_thread"] == 0, r["name"]


def test_kernel_report_needs_no_prior_launch():
    """The report's occupancy figures do not depend on which kernels ran before: in a fresh
    process, before any launch, every record already gives at least one resident block."""
    import subprocess, sys, os
    code = ("import epilogue_chains_gb300 as fc\n"
            "bad = [r['name'] for r in (fc.fuse_kernel_report(i) for i in range(fc.fuse_kernel_count()))"
            " if r['blocks_per_sm_api'] < 1 or r['blocks_per_sm'] < 1]\n"
            "assert not bad, bad\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
