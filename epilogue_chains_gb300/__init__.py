"""epilogue_chains_gb300 -- vertical fusion of dependent operator chains on one GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/fusechain.h`` (``libfusechain.so``): the functions
below have the C names and only marshal arguments (torch tensors -> device pointers, the current
torch stream -> ``cudaStream_t``, status codes -> ``FuseError``).  Every step of every chain runs
in the library's CUDA kernels; there is no fallback: if the library cannot be built or loaded, the
first call raises.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import threading

FUSE_OK, FUSE_EINVAL, FUSE_EALIGN, FUSE_EUNSUPPORTED = 0, -1, -2, -3
FUSE_ECUDA, FUSE_ETIMEOUT, FUSE_EWORKSPACE = -4, -5, -6
FUSE_F32, FUSE_F16, FUSE_BF16 = 0, 1, 2
FUSE_FUSED, FUSE_UNFUSED, FUSE_FAT = 0, 1, 2
FUSE_OP_AFFINE, FUSE_OP_AFFINE_RELU = 0, 1
FUSE_MAX_STAGES = 32
FUSE_FAT_TEMPS = 48


class FuseError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _load()
        msg = lib.fuse_strerror(status).decode()
        extra = lib.fuse_last_cuda_error().decode() if status == FUSE_ECUDA else ""
        super().__init__(f"{where}: {msg} ({status}) {extra}".strip())
        self.status = status


class fuse_stage(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("a", ctypes.c_float), ("b", ctypes.c_float),
                ("writes", ctypes.c_int64), ("ext_reads", ctypes.c_int64),
                ("flops", ctypes.c_int64), ("live_regs", ctypes.c_int32)]


class fuse_ledger_t(ctypes.Structure):
    _fields_ = [("bytes", ctypes.c_int64), ("launches", ctypes.c_int64),
                ("reg_peak", ctypes.c_int64), ("flops", ctypes.c_int64)]


class fuse_cost_model(ctypes.Structure):
    _fields_ = [("hbm_bytes_per_s", ctypes.c_double), ("flops_per_s", ctypes.c_double),
                ("launch_s", ctypes.c_double), ("spill_penalty", ctypes.c_double),
                ("reg_limit", ctypes.c_int32)]


class fuse_kernel_record(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 64), ("regs_per_thread", ctypes.c_int32),
                ("local_bytes_per_thread", ctypes.c_int32), ("static_smem_bytes", ctypes.c_int32),
                ("dynamic_smem_bytes", ctypes.c_int32), ("block_threads", ctypes.c_int32),
                ("blocks_per_sm", ctypes.c_int32), ("max_threads_per_block", ctypes.c_int32),
                ("cluster_size", ctypes.c_int32), ("max_active_clusters", ctypes.c_int32),
                ("blocks_per_sm_api", ctypes.c_int32), ("tmem_cols", ctypes.c_int32),
                ("ptxas_registers", ctypes.c_int32), ("stack_bytes", ctypes.c_int32),
                ("spill_store_bytes", ctypes.c_int32), ("spill_load_bytes", ctypes.c_int32),
                ("symbol", ctypes.c_char * 256)]


class fuse_ptxas_record(ctypes.Structure):
    _fields_ = [("symbol", ctypes.c_char * 256), ("registers", ctypes.c_int32),
                ("stack_bytes", ctypes.c_int32), ("spill_store_bytes", ctypes.c_int32),
                ("spill_load_bytes", ctypes.c_int32)]


_P, _I32, _I64, _U32, _F32, _SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32,
                                   ctypes.c_float, ctypes.c_size_t)
# every symbol the header declares, with its C signature
SIGNATURES = {
    "fuse_chain_run": ([ctypes.POINTER(fuse_stage), _I32, _P, _P, _I64, _I32, _I32, _P], _I32),
    "fuse_chain_run_host": ([ctypes.POINTER(fuse_stage), _I32, _P, _P, _I64, _I32, _I32, _P, _P, _I32, _P], _I32),
    "fuse_rmsnorm": ([_P, _P, _P, _I64, _I64, _F32, _I32, _P, _SZ, _P], _I32),
    "fuse_rmsnorm_workspace_bytes": ([_I64, _I64, _I32], _SZ),
    "fuse_rmsnorm_unfused_static": ([_P, _P, _P, _I64, _I64, _F32, _P], _I32),
    "fuse_causal_softmax": ([_P, _P, _I64, _I64, _F32, _I32, _I32, _I32, _P, _SZ, _P], _I32),
    "fuse_causal_softmax_workspace_bytes": ([_I64, _I64, _I32], _SZ),
    "fuse_gemm_epilogue": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _P], _I32),
    "fuse_gemm_epilogue_plan": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _U32, _P], _I32),
    "fuse_gemm_epilogue_ws": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _U32, _P, _SZ, _P], _I32),
    "fuse_gemm_workspace_bytes": ([_I64, _I64, _I64], _SZ),
    "fuse_gemm_bytes": ([_I64, _I64, _I64, _U32], _I64),
    "fuse_attention_schedule": ([_I64, _I64, _I32, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)], _I64),
    "fuse_ledger": ([ctypes.POINTER(fuse_stage), _I32, _U32, _I32, ctypes.POINTER(fuse_ledger_t)], _I32),
    "fuse_plan_time": ([ctypes.POINTER(fuse_stage), _I32, _U32, _I32, ctypes.POINTER(fuse_cost_model),
                        ctypes.POINTER(ctypes.c_double)], _I32),
    "fuse_best_plan": ([ctypes.POINTER(fuse_stage), _I32, _I32, ctypes.POINTER(fuse_cost_model),
                        ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_double)], _I32),
    "fuse_launch_model": ([_I64, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                           ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                           ctypes.POINTER(ctypes.c_double)], _I32),
    "fuse_add_rmsnorm": ([_P, _P, _P, _P, _P, _I64, _I64, _F32, _I32, _P, _SZ, _P], _I32),
    "fuse_silu_mul": ([_P, _P, _I64, _P, _I64, _I64, _I32, _I32, _P], _I32),
    "fuse_add_rmsnorm_bytes": ([_I64, _I64, _I32], _I64),
    "fuse_attention": ([_P, _P, _P, _P, _I64, _I64, _I64, _F32, _P], _I32),
    "fuse_attention_bytes": ([_I64, _I64, _I64], _I64),
    "fuse_attention_flops": ([_I64, _I64, _I64], _I64),
    "fuse_silu_mul_bytes": ([_I64, _I64, _I32, _I32], _I64),
    "fuse_chain_bytes": ([_I32, _I64, _I32, _I32], _I64),
    "fuse_rmsnorm_bytes": ([_I64, _I64, _I32], _I64),
    "fuse_causal_softmax_bytes": ([_I64, _I64, _I32, _I32, _I32], _I64),
    "fuse_kernel_count": ([], _I32),
    "fuse_kernel_report": ([_I32, ctypes.POINTER(fuse_kernel_record)], _I32),
    "fuse_ptxas_count": ([], _I32),
    "fuse_ptxas_entry": ([_I32, ctypes.POINTER(fuse_ptxas_record)], _I32),
    "fuse_strerror": ([_I32], ctypes.c_char_p),
    "fuse_last_cuda_error": ([], ctypes.c_char_p),
    "fuse_check": ([_P], _I32),
    "fuse_debug_expire_wait": ([_I64, _P], _I32),
    "fuse_debug_split_window": ([_I64], _I32),
    "fuse_graph_begin": ([_P], _I32),
    "fuse_graph_end": ([_P, ctypes.POINTER(ctypes.c_void_p)], _I32),
    "fuse_graph_launch": ([_P, _P], _I32),
    "fuse_graph_kernel_count": ([_P], _I32),
    "fuse_graph_destroy": ([_P], None),
    "fuse_version": ([], _I32),
}

_lock = threading.Lock()
_lib = None


def _load():
    """Build (if needed) and load libfusechain.so; raises if either fails."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            from . import _build
            path = _build.build()
            lib = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def library_path() -> str:
    from . import _build
    return _build.LIB


def _check(status: int, where: str) -> None:
    if status != FUSE_OK:
        raise FuseError(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    return {torch.float32: FUSE_F32, torch.float16: FUSE_F16, torch.bfloat16: FUSE_BF16}[t.dtype]


def _stages(stages) -> ctypes.Array:
    """Accept fuse_stage objects, (op, a, b) tuples or dicts with the struct's field names."""
    arr = (fuse_stage * len(stages))()
    for i, s in enumerate(stages):
        if isinstance(s, fuse_stage):
            arr[i] = s
        elif isinstance(s, dict):
            arr[i] = fuse_stage(**s)
        else:
            op, a, b = s
            arr[i] = fuse_stage(int(op), float(a), float(b), 0, 0, 0, 0)
    return arr


def _need_device(*ts):
    for t in ts:
        if t is not None and not isinstance(t, int):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError("tensors must be contiguous CUDA tensors")


# ------------------------------------------------------------------------------- chains
def fuse_chain_run(stages, x, y, mode: int = FUSE_FUSED, stream=None) -> None:
    """y <- f_{K-1}(...f_0(x)) with f_s(v) = [ReLU](a_s v + b_s); see fusechain.h."""
    _need_device(x, y)
    if x.dtype != y.dtype or x.numel() != y.numel():
        raise ValueError("x and y must have the same dtype and element count")
    st = _stages(stages)
    _check(_load().fuse_chain_run(st, len(st), _ptr(x), _ptr(y), x.numel(), _dtype_code(x), mode,
                                  _stream(stream)), "fuse_chain_run")


def fuse_chain_run_host(stages, x_host, y_host, x_dev, y_dev, mode: int = FUSE_FUSED, slices: int = 8,
                        stream=None) -> None:
    """The chain on host tensors (x_host in, y_host out; pinned for asynchronous copies) through
    the caller's device scratch x_dev, y_dev (same dtype and element count); see fusechain.h.
    y_host is valid after the stream is synchronized."""
    _need_device(x_dev, y_dev)
    for t in (x_host, y_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("x_host and y_host must be contiguous host tensors")
    n = x_host.numel()
    if any(t.numel() != n or t.dtype != x_host.dtype for t in (y_host, x_dev, y_dev)):
        raise ValueError("all four tensors must have the same dtype and element count")
    st = _stages(stages)
    _check(_load().fuse_chain_run_host(st, len(st), _ptr(x_host), _ptr(y_host), n, _dtype_code(x_host),
                                       mode, _ptr(x_dev), _ptr(y_dev), int(slices), _stream(stream)),
           "fuse_chain_run_host")


def fuse_rmsnorm(x, w, y, eps: float, mode: int = FUSE_FUSED, workspace=None, stream=None) -> None:
    """y = x * rsqrt(mean(x^2, -1) + eps) * w over rows of a [rows, hidden] fp32 tensor."""
    import torch
    _need_device(x, w, y)
    rows, hidden = x.shape
    lib = _load()
    ws_bytes = lib.fuse_rmsnorm_workspace_bytes(rows, hidden, mode)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    ws_size = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.fuse_rmsnorm(_ptr(x), _ptr(w), _ptr(y), rows, hidden, float(eps), mode,
                            _ptr(workspace), ws_size, _stream(stream)), "fuse_rmsnorm")


def fuse_add_rmsnorm(x, r, w, h, y, eps: float, mode: int = FUSE_FUSED, workspace=None,
                     stream=None) -> None:
    """h = x + r; y = h * rsqrt(mean(h^2, -1) + eps) * w over rows of [rows, hidden] fp32."""
    import torch
    _need_device(x, r, w, h, y)
    rows, hidden = x.shape
    lib = _load()
    ws_bytes = lib.fuse_rmsnorm_workspace_bytes(rows, hidden, mode)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    ws_size = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.fuse_add_rmsnorm(_ptr(x), _ptr(r), _ptr(w), _ptr(h), _ptr(y), rows, hidden,
                                float(eps), mode, _ptr(workspace), ws_size, _stream(stream)),
           "fuse_add_rmsnorm")


def fuse_silu_mul(g, u, y, mode: int = FUSE_FUSED, stream=None) -> None:
    """y = SiLU(g) * u.  g and u: [rows, cols] tensors (possibly the two column halves of one
    merged [rows, 2 cols] tensor: same row stride); y: contiguous [rows, cols]."""
    for t in (g, u, y):
        if not t.is_cuda or t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("g, u, y must be 2-D CUDA tensors with unit column stride")
    if g.shape != u.shape or g.shape != y.shape or g.stride(0) != u.stride(0):
        raise ValueError("g, u, y must have one shape and g, u one row stride")
    if not y.is_contiguous() or g.dtype != u.dtype or g.dtype != y.dtype:
        raise ValueError("y must be contiguous and all three of one dtype")
    rows, cols = g.shape
    _check(_load().fuse_silu_mul(_ptr(g), _ptr(u), g.stride(0), _ptr(y), rows, cols,
                                 _dtype_code(g), mode, _stream(stream)), "fuse_silu_mul")


def fuse_attention(q, k, v, o, scale: float, stream=None) -> None:
    """o = causal softmax(scale q k^T) v over bf16 [bh, S, D] tensors, no score matrix."""
    _need_device(q, k, v, o)
    if q.shape != k.shape or q.shape != v.shape or q.shape != o.shape or q.dim() != 3:
        raise ValueError("q, k, v, o must be [bh, S, D] tensors of one shape")
    bh, S, D = q.shape
    _check(_load().fuse_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(o), bh, S, D, float(scale),
                                  _stream(stream)), "fuse_attention")


def fuse_rmsnorm_unfused_static(x, w, y, eps: float, stream=None) -> None:
    """Unfused RMSNorm with its row statistics in the library's own fixed device array (no
    workspace, no allocation; rows <= FUSE_RMSNORM_STATIC_MAX_ROWS)."""
    _need_device(x, w, y)
    rows, hidden = x.shape
    _check(_load().fuse_rmsnorm_unfused_static(_ptr(x), _ptr(w), _ptr(y), rows, hidden, float(eps),
                                               _stream(stream)), "fuse_rmsnorm_unfused_static")


FUSE_RMSNORM_STATIC_MAX_ROWS = 65536
FUSE_GEMM_STATIC_B = 0x100


def fuse_causal_softmax(s, p, scale: float, skip_tile: int = 0, mode: int = FUSE_FUSED,
                        workspace=None, stream=None) -> None:
    """p = causal softmax(scale * s) over the last axis of a bf16 [..., S, S] tensor."""
    import torch
    _need_device(s, p)
    S = s.shape[-1]
    bh = s.numel() // (S * S)
    lib = _load()
    ws_bytes = lib.fuse_causal_softmax_workspace_bytes(bh, S, mode)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=s.device)
    ws_size = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.fuse_causal_softmax(_ptr(s), _ptr(p), bh, S, float(scale), int(skip_tile),
                                   _dtype_code(p), mode, _ptr(workspace), ws_size,
                                   _stream(stream)), "fuse_causal_softmax")


# split-K workspaces handed out by fuse_gemm_epilogue(workspace=None): one zero-filled buffer per
# (device, stream), reused (every completed call leaves it zero-filled), never freed
_GEMM_WS = {}


def _gemm_workspace(M: int, N: int, K: int, dev, stream_handle):
    import torch
    need = fuse_gemm_workspace_bytes(M, N, K)
    if need == 0:
        return None
    key = (dev.index, stream_handle)
    ws = _GEMM_WS.get(key)
    if ws is not None and ws.numel() >= need:
        return ws
    # allocate only on torch's current stream and outside graph capture; otherwise the call
    # runs unsplit
    if torch.cuda.is_current_stream_capturing() or stream_handle != torch.cuda.current_stream(dev).cuda_stream:
        return None
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    torch.cuda.current_stream(dev).synchronize()   # zero-filled before any stream uses it
    _GEMM_WS[key] = ws
    return ws


def fuse_gemm_epilogue(A, B, bias, R, Y, cut_mask: int = 0, workspace=None, stream=None) -> None:
    """Y = fp16(GELU(A @ B + bias) + R) for fp16 A [M,K], B [K,N], bias [N], R, Y [M,N]; cut_mask
    selects the plan (0 = fully fused [4]; 7 = [1,1,1,1]).  workspace: a zero-filled device tensor
    of fuse_gemm_workspace_bytes(M, N, K) bytes (see fuse_gemm_epilogue_ws in the header), reused
    across calls on one stream; None: a buffer of that kind kept by this module per device and
    stream; False: none (the last wave of tiles is not split over K)."""
    _need_device(A, B, bias, R, Y)
    M, K = A.shape
    K2, N = B.shape
    if K != K2 or tuple(R.shape) != (M, N) or tuple(Y.shape) != (M, N) or bias.numel() != N:
        raise ValueError("shape mismatch")
    sh = _stream(stream)
    if workspace is None:
        workspace = _gemm_workspace(M, N, K, A.device, sh)
    elif workspace is False:
        workspace = None
    ws_size = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_load().fuse_gemm_epilogue_ws(_ptr(A), _ptr(B), _ptr(bias), _ptr(R), _ptr(Y), M, N, K,
                                         int(cut_mask), _ptr(workspace), ws_size, sh),
           "fuse_gemm_epilogue")


def fuse_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return _load().fuse_gemm_workspace_bytes(M, N, K)


def fuse_attention_schedule(bh: int, S: int, clusters: int):
    """Per-cluster item lists of the persistent attention kernel: (first [clusters + 1], items)."""
    n = bh * S // 256
    first = (ctypes.c_int32 * (clusters + 1))()
    items = (ctypes.c_int32 * max(1, n))()
    rc = _load().fuse_attention_schedule(bh, S, clusters, first, items)
    _check(rc if rc < 0 else 0, "fuse_attention_schedule")
    return list(first), list(items[:rc])


def fuse_gemm_bytes(M: int, N: int, K: int, cut_mask: int) -> int:
    return _load().fuse_gemm_bytes(M, N, K, cut_mask)


# ------------------------------------------------------------------------------- ledgers
def fuse_ledger(stages, cut_mask: int, elem_bytes: int) -> dict:
    st = _stages(stages)
    out = fuse_ledger_t()
    _check(_load().fuse_ledger(st, len(st), cut_mask, elem_bytes, ctypes.byref(out)), "fuse_ledger")
    return {"bytes": out.bytes, "launches": out.launches, "reg_peak": out.reg_peak,
            "flops": out.flops}


def _model(model) -> fuse_cost_model:
    if isinstance(model, fuse_cost_model):
        return model
    return fuse_cost_model(**model)


def fuse_plan_time(stages, cut_mask: int, elem_bytes: int, model) -> float:
    """[K4] time_estimate of one cut plan, seconds."""
    st = _stages(stages)
    out = ctypes.c_double()
    _check(_load().fuse_plan_time(st, len(st), cut_mask, elem_bytes, ctypes.byref(_model(model)),
                                  ctypes.byref(out)), "fuse_plan_time")
    return out.value


def fuse_best_plan(stages, elem_bytes: int, model) -> tuple:
    """[K4] best_plan: (cut_mask, seconds) of the cheapest of the 2^(K-1) plans."""
    st = _stages(stages)
    mask, sec = ctypes.c_uint32(), ctypes.c_double()
    _check(_load().fuse_best_plan(st, len(st), elem_bytes, ctypes.byref(_model(model)),
                                  ctypes.byref(mask), ctypes.byref(sec)), "fuse_best_plan")
    return mask.value, sec.value


def fuse_add_rmsnorm_bytes(rows: int, hidden: int, mode: int) -> int:
    return _load().fuse_add_rmsnorm_bytes(rows, hidden, mode)


def fuse_silu_mul_bytes(rows: int, cols: int, dtype: int, mode: int) -> int:
    return _load().fuse_silu_mul_bytes(rows, cols, dtype, mode)


def fuse_attention_bytes(bh: int, S: int, D: int) -> int:
    return _load().fuse_attention_bytes(bh, S, D)


def fuse_attention_flops(bh: int, S: int, D: int) -> int:
    return _load().fuse_attention_flops(bh, S, D)


def fuse_launch_model(n_kernels: int, t_launch: float, t_exec: float, t_dispatch: float) -> dict:
    """Eager vs CUDA-graph timeline of n_kernels kernels; see fusechain.h."""
    e, i, g = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    _check(_load().fuse_launch_model(n_kernels, t_launch, t_exec, t_dispatch, ctypes.byref(e),
                                     ctypes.byref(i), ctypes.byref(g)), "fuse_launch_model")
    return {"eager": e.value, "eager_idle": i.value, "graph": g.value}


def fuse_chain_bytes(K: int, n: int, dtype: int, mode: int) -> int:
    return _load().fuse_chain_bytes(K, n, dtype, mode)


def fuse_rmsnorm_bytes(rows: int, hidden: int, mode: int) -> int:
    return _load().fuse_rmsnorm_bytes(rows, hidden, mode)


def fuse_causal_softmax_bytes(bh: int, S: int, skip_tile: int, out_dtype: int, mode: int) -> int:
    return _load().fuse_causal_softmax_bytes(bh, S, skip_tile, out_dtype, mode)


def fuse_rmsnorm_workspace_bytes(rows: int, hidden: int, mode: int) -> int:
    return _load().fuse_rmsnorm_workspace_bytes(rows, hidden, mode)


def fuse_causal_softmax_workspace_bytes(bh: int, S: int, mode: int) -> int:
    return _load().fuse_causal_softmax_workspace_bytes(bh, S, mode)


# ------------------------------------------------------------------------------- status
def fuse_kernel_count() -> int:
    return _load().fuse_kernel_count()


def fuse_kernel_report(index: int) -> dict:
    rec = fuse_kernel_record()
    _check(_load().fuse_kernel_report(index, ctypes.byref(rec)), "fuse_kernel_report")
    return {f: (getattr(rec, f).decode() if f in ("name", "symbol") else getattr(rec, f))
            for f, _ in fuse_kernel_record._fields_}


def fuse_ptxas_table() -> list[dict]:
    """The ptxas -v record of every kernel compiled into the library (host only)."""
    lib = _load()
    out = []
    for i in range(lib.fuse_ptxas_count()):
        rec = fuse_ptxas_record()
        _check(lib.fuse_ptxas_entry(i, ctypes.byref(rec)), "fuse_ptxas_entry")
        out.append({f: (getattr(rec, f).decode() if f == "symbol" else getattr(rec, f))
                    for f, _ in fuse_ptxas_record._fields_})
    return out


def fuse_check(stream=None) -> int:
    return _load().fuse_check(_stream(stream))


def fuse_debug_expire_wait(budget_cycles: int, stream=None) -> None:
    _check(_load().fuse_debug_expire_wait(int(budget_cycles), _stream(stream)),
           "fuse_debug_expire_wait")


# ------------------------------------------------------------------------------- graphs
def fuse_graph_begin(stream=None) -> None:
    """Start capturing this library's calls on `stream` (a non-default stream)."""
    _check(_load().fuse_graph_begin(_stream(stream)), "fuse_graph_begin")


def fuse_graph_end(stream=None) -> int:
    """End the capture; returns the executable graph's handle (free with fuse_graph_destroy)."""
    g = ctypes.c_void_p()
    _check(_load().fuse_graph_end(_stream(stream), ctypes.byref(g)), "fuse_graph_end")
    return g.value


def fuse_graph_launch(graph: int, stream=None) -> None:
    _check(_load().fuse_graph_launch(graph, _stream(stream)), "fuse_graph_launch")


def fuse_graph_kernel_count(graph: int) -> int:
    n = _load().fuse_graph_kernel_count(graph)
    _check(min(n, 0), "fuse_graph_kernel_count")
    return n


def fuse_graph_destroy(graph: int) -> None:
    _load().fuse_graph_destroy(graph)


def fuse_strerror(status: int) -> str:
    return _load().fuse_strerror(status).decode()


def fuse_version() -> int:
    return _load().fuse_version()
