"""Launch timeline model of "AIGC fundamentals | operator fusion and CUDA Graph" §3.4 (and its
appendix script launch_model, sections [F1]/[F2]) -- TEST INFRASTRUCTURE ONLY.

One stream, N kernels.  Eager: the host spends t_launch submitting each kernel and goes straight on
to the next; kernel i may start once kernel i-1 has finished and its own submission is done.
Graph: one submission (t_launch) for the whole graph, after which the GPU front end still spends
t_dispatch per node.  The eager side is simulated event by event, as the section describes it.

Parity status: pinned (tests/test_launch_model.py) against the page's printed [F2] speed-ups and
the §6.4 large-kernel figure.
"""
from __future__ import annotations


def simulate_eager(n_kernels: int, t_launch: float, t_exec: float):
    """Returns (total time, GPU idle time)."""
    gpu_free, idle = 0.0, 0.0
    for i in range(n_kernels):
        submitted = (i + 1) * t_launch
        start = gpu_free if gpu_free > submitted else submitted
        idle += start - gpu_free
        gpu_free = start + t_exec
    return gpu_free, idle


def simulate_graph(n_kernels: int, t_launch: float, t_exec: float, t_dispatch: float):
    """Returns (total time, GPU idle time): one submission, then every node pays t_dispatch."""
    return t_launch + n_kernels * (t_exec + t_dispatch), t_launch
