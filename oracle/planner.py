"""Cut-plan cost model of the K4 walkthrough, written out plainly -- TEST INFRASTRUCTURE ONLY.

"K4 walkthrough: the three ledgers of fusion -- bytes, launches, registers", §② (time_estimate,
best_plan) and §③ (spill penalty): a plan is a split of the stages into consecutive kernels; a
kernel reads the previous kernel's output and its stages' external inputs, writes its last stage's
output, and costs max(bytes / bandwidth, flops / peak) + one launch, with the memory part multiplied
by the spill penalty when the live registers of its stages add up to more than the limit.
best_plan enumerates every way to cut the n stages (2^(n-1) of them) and keeps the cheapest; ties go
to the plan with the lower cut mask (bit i = a cut after stage i).

Parity status: pinned (tests/test_planner.py) against the estimates the page prints.
"""
from __future__ import annotations


def segments(n_stages: int, cut_mask: int):
    """The kernels of a plan as (first, last) stage index pairs."""
    out, start = [], 0
    for i in range(n_stages):
        if i == n_stages - 1 or (cut_mask >> i) & 1:
            out.append((start, i))
            start = i + 1
    return out


def plan_time(stages, cut_mask, elem_bytes, bw, peak, launch, penalty, reg_limit):
    """stages: list of dicts with writes, ext_reads, flops, live_regs."""
    total = 0.0
    for first, last in segments(len(stages), cut_mask):
        elems = stages[first - 1]["writes"] if first > 0 else 0
        elems += sum(stages[s]["ext_reads"] for s in range(first, last + 1))
        elems += stages[last]["writes"]
        mem = elems * elem_bytes / bw
        if sum(stages[s]["live_regs"] for s in range(first, last + 1)) > reg_limit:
            mem *= penalty
        comp = sum(stages[s]["flops"] for s in range(first, last + 1)) / peak
        total += max(mem, comp) + launch
    return total


def best_plan(stages, elem_bytes, bw, peak, launch, penalty, reg_limit):
    best = None
    for mask in range(2 ** (len(stages) - 1)):
        t = plan_time(stages, mask, elem_bytes, bw, peak, launch, penalty, reg_limit)
        if best is None or t < best[1]:
            best = (mask, t)
    return best
