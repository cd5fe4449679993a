"""Seeded synthetic inputs for the four chains (shared by the tests, the bench and smoke).

This module holds no arithmetic of the method: it only draws random numbers and rounds them
to the storage types.  Both the CUDA path and the CPU oracle consume the arrays it returns.

Seeds: the pages' fusion_lab script fixes RNG_SEED = 20261002 ("Operator fusion and CUDA Graph",
appendix fusion_lab, section [A]); each workload adds its config index to it, and a ``salt``
separates independent draws inside one config (e.g. one stage-coefficient draw per K).

Workload recipes (the five configurations of the hot path):
  0  8-stage affine chain h <- 1.01 h + 0.01, x fp32 [4096] ~ N(0,1)
  1  pointwise chain, x fp32 [16,777,216] ~ N(0,1), K in {2,3,4,6,8};
     a_s ~ U[0.9, 1.1], b_s ~ U[-0.1, 0.1] (fp32), ReLU on even s (0-based)
  2  RMSNorm x fp32 [2048, 4096] ~ N(0,1), w fp32 [4096] ~ N(1, 0.02), eps 1e-6
  3  causal softmax s bf16 [8, 16, 2048, 2048] ~ N(0,1) rounded to bf16, scale 1/16
  4  GEMM + bias + GELU + residual, fp16: A [M,4096], B [4096,4096] ~ N(0, std 1/64),
     bias [4096] ~ N(0, 0.1), R [M,4096] ~ N(0,1); M in {4096, 16}
  5  residual add + RMSNorm: x, r fp32 [2048, 4096] ~ N(0,1), w fp32 [4096] ~ N(1, 0.02),
     eps 1e-6 (config 2's rows and hidden size, plus the residual input)
  6  SiLU(gate) * up: one merged gate/up output gu bf16 [2048, 2 x 14336] ~ N(0,1) (gate the
     first 14336 columns, up the rest); 14336 is the FFN width of the Llama-3-8B configuration
     the pages count kernels for, 2048 rows as config 2
  7  causal attention without the score matrix: q, k, v bf16 [8 x 16, 2048, 256] ~ N(0,1)
     rounded to bf16 (B=8, H=16, S=2048, d=4096 -> head size 256: the shape whose score tensor
     is config 3), scale 1/16 = 1/sqrt(256)
"""
from __future__ import annotations

import numpy as np

RNG_SEED = 20261002

AFFINE_K, AFFINE_A, AFFINE_B, AFFINE_N = 8, 1.01, 0.01, 4096
CHAIN_N = 16_777_216
CHAIN_KS = (2, 3, 4, 6, 8)
RMS_ROWS, RMS_HIDDEN, RMS_EPS = 2048, 4096, 1e-6
SM_B, SM_H, SM_S = 8, 16, 2048
SM_SCALE = 1.0 / 16.0          # 1/sqrt(256)
GEMM_N, GEMM_K = 4096, 4096
GEMM_MS = (4096, 16)
GEMM_STD = 1.0 / 64.0          # "N(0, 1/sqrt(4096))", second parameter read as the std
ADDRMS_ROWS, ADDRMS_HIDDEN = 2048, 4096
SILU_ROWS, SILU_COLS = 2048, 14336
ATT_BH, ATT_S, ATT_D = SM_B * SM_H, SM_S, 256
ATT_SCALE = 1.0 / 16.0          # 1/sqrt(256)


def rng(config: int, salt: int = 0) -> np.random.Generator:
    return np.random.default_rng([RNG_SEED + config, salt])


def _torch_gen(config: int, salt: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((RNG_SEED + config) * 1_000_003 + salt)
    return g


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (RNE) and return the uint16 bit patterns (input preparation)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f16_bits_from_f64(x: np.ndarray) -> np.ndarray:
    """Round to fp16 (numpy's IEEE conversion) and return the uint16 bit patterns."""
    return np.ascontiguousarray(x).astype(np.float16).view(np.uint16)


# ----------------------------------------------------------------------------- chains
def affine_chain(n: int = AFFINE_N, K: int = AFFINE_K):
    """Config 0: stage coefficients (all a = 1.01, b = 0.01, no ReLU) and x ~ N(0,1) fp32."""
    x = rng(0).standard_normal(n).astype(np.float32)
    a = np.full(K, AFFINE_A, dtype=np.float32)
    b = np.full(K, AFFINE_B, dtype=np.float32)
    relu = np.zeros(K, dtype=np.int32)
    return relu, a, b, x


def chain_stages(K: int, config: int = 1):
    """Config 1 stage coefficients for one K: a_s ~ U[0.9,1.1], b_s ~ U[-0.1,0.1], ReLU on even s."""
    g = rng(config, 1000 + K)
    a = g.uniform(0.9, 1.1, K).astype(np.float32)
    b = g.uniform(-0.1, 0.1, K).astype(np.float32)
    relu = np.array([1 if s % 2 == 0 else 0 for s in range(K)], dtype=np.int32)
    return relu, a, b


def chain_input(n: int, config: int = 1, salt: int = 0, device=None):
    """x ~ N(0,1) fp32 of n elements: numpy on the host, or a torch tensor drawn on ``device``."""
    if device is None:
        return rng(config, salt).standard_normal(n).astype(np.float32)
    import torch
    return torch.randn(n, generator=_torch_gen(config, salt, device), device=device,
                       dtype=torch.float32)


# ----------------------------------------------------------------------------- RMSNorm
def rmsnorm_input(rows: int = RMS_ROWS, hidden: int = RMS_HIDDEN, config: int = 2, salt: int = 0,
                  device=None):
    """x ~ N(0,1) fp32 [rows, hidden], w ~ N(1, 0.02) fp32 [hidden]."""
    if device is None:
        g = rng(config, salt)
        x = g.standard_normal((rows, hidden)).astype(np.float32)
        w = (1.0 + 0.02 * g.standard_normal(hidden)).astype(np.float32)
        return x, w
    import torch
    g = _torch_gen(config, salt, device)
    x = torch.randn(rows, hidden, generator=g, device=device, dtype=torch.float32)
    w = 1.0 + 0.02 * torch.randn(hidden, generator=g, device=device, dtype=torch.float32)
    return x, w


def add_rmsnorm_input(rows: int = ADDRMS_ROWS, hidden: int = ADDRMS_HIDDEN, config: int = 5,
                      salt: int = 0, device=None):
    """x, r ~ N(0,1) fp32 [rows, hidden], w ~ N(1, 0.02) fp32 [hidden]."""
    if device is None:
        g = rng(config, salt)
        x = g.standard_normal((rows, hidden)).astype(np.float32)
        r = g.standard_normal((rows, hidden)).astype(np.float32)
        w = (1.0 + 0.02 * g.standard_normal(hidden)).astype(np.float32)
        return x, r, w
    import torch
    g = _torch_gen(config, salt, device)
    x = torch.randn(rows, hidden, generator=g, device=device, dtype=torch.float32)
    r = torch.randn(rows, hidden, generator=g, device=device, dtype=torch.float32)
    w = 1.0 + 0.02 * torch.randn(hidden, generator=g, device=device, dtype=torch.float32)
    return x, r, w


# ----------------------------------------------------------------------------- SiLU * up
def silu_input(rows: int = SILU_ROWS, cols: int = SILU_COLS, dtype: str = "bf16", config: int = 6,
               salt: int = 0, scale: float = 1.0, device=None):
    """Merged gate/up tensor [rows, 2 cols] ~ N(0, scale^2): float32 for "f32", else uint16 bit
    patterns of fp16/bf16 on the host; a torch tensor of that dtype on ``device``."""
    if device is None:
        x = scale * rng(config, salt).standard_normal((rows, 2 * cols))
        if dtype == "f32":
            return x.astype(np.float32)
        if dtype == "f16":
            return f16_bits_from_f64(x)
        return bf16_bits_from_f32(x.astype(np.float32))
    import torch
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    g = _torch_gen(config, salt, device)
    return (scale * torch.randn(rows, 2 * cols, generator=g, device=device)).to(tdt)


# ----------------------------------------------------------------------------- attention
def attention_input(bh: int = ATT_BH, S: int = ATT_S, D: int = ATT_D, config: int = 7,
                    salt: int = 0, device=None):
    """q, k, v ~ N(0,1) rounded to bf16, [bh, S, D]: uint16 bit patterns on the host, torch
    bfloat16 tensors on ``device``."""
    if device is None:
        g = rng(config, salt)
        return tuple(bf16_bits_from_f32(g.standard_normal((bh, S, D)).astype(np.float32))
                     for _ in range(3))
    import torch
    g = _torch_gen(config, salt, device)
    return tuple(torch.randn(bh, S, D, generator=g, device=device, dtype=torch.float32).to(
        torch.bfloat16) for _ in range(3))


# ----------------------------------------------------------------------------- softmax
def softmax_input(bh: int, S: int, config: int = 3, salt: int = 0, device=None):
    """Scores ~ N(0,1) rounded to bf16: uint16 bit patterns [bh, S, S] on the host, or a torch
    bfloat16 tensor drawn on ``device``."""
    if device is None:
        x = rng(config, salt).standard_normal((bh, S, S)).astype(np.float32)
        return bf16_bits_from_f32(x)
    import torch
    g = _torch_gen(config, salt, device)
    return torch.randn(bh, S, S, generator=g, device=device, dtype=torch.float32).to(
        torch.bfloat16)


# ----------------------------------------------------------------------------- GEMM
def gemm_input(M: int, N: int = GEMM_N, K: int = GEMM_K, config: int = 4, salt: int = 0,
               std: float = GEMM_STD, device=None):
    """A [M,K], B [K,N] ~ N(0, std), bias [N] ~ N(0, 0.1), R [M,N] ~ N(0,1), all fp16.

    Host: uint16 fp16 bit patterns.  Device: torch float16 tensors."""
    if device is None:
        g = rng(config, salt * 16 + (0 if M >= 128 else 1))
        A = f16_bits_from_f64(std * g.standard_normal((M, K)))
        B = f16_bits_from_f64(std * g.standard_normal((K, N)))
        bias = f16_bits_from_f64(0.1 * g.standard_normal(N))
        R = f16_bits_from_f64(g.standard_normal((M, N)))
        return A, B, bias, R
    import torch
    g = _torch_gen(config, salt * 16 + (0 if M >= 128 else 1), device)
    A = (std * torch.randn(M, K, generator=g, device=device)).to(torch.float16)
    B = (std * torch.randn(K, N, generator=g, device=device)).to(torch.float16)
    bias = (0.1 * torch.randn(N, generator=g, device=device)).to(torch.float16)
    R = torch.randn(M, N, generator=g, device=device).to(torch.float16)
    return A, B, bias, R
