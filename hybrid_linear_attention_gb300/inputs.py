"""Seeded synthetic inputs for the KDA token mixer.

This module draws random numbers and nothing else: it holds none of the layer's arithmetic
(no convolution, no normalisation, no decay, no delta rule).  Both the CUDA path and the
oracle are fed from it, so the two always see identical arrays.

Distributions follow the workloads the KDA layer is measured on: q, k, v ~ N(0, 1) in bf16
(or fp32 for the tiny case), per-channel log-retention g ~ U(-5, 0) (the safe forget gate's
range), write strength beta = sigmoid(N(0, 1)) per head-token, initial states ~ N(0, 0.02),
raw convolution inputs ~ N(0, 1), conv weights ~ N(0, 0.5^2), output-gate logits ~ N(0, 1).
The sigmoid applied to beta's normal draw is part of that distribution's recipe, not of the
path (the path's own beta activation lives in the prologue kernel).

Large arrays can be drawn directly on the GPU (``device="cuda"``) with torch's generator;
the same seed on the same device always gives the same arrays.
"""
from __future__ import annotations

import math

import numpy as np
import torch

LOG_ALPHA_LOW = -5.0  # lower end of the log-retention draw
STATE_STD = 0.02
CONV_W_STD = 0.5


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, *, seed, device="cpu", dtype=torch.bfloat16, std=1.0):
    g = _gen(device, seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def uniform(shape, low, high, *, seed, device="cpu"):
    g = _gen(device, seed)
    x = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    return x.mul_(high - low).add_(low)


def beta_draw(shape, *, seed, device="cpu"):
    """beta = sigmoid(N(0, 1)), fp32."""
    return torch.sigmoid(normal(shape, seed=seed, device=device, dtype=torch.float32))


def cu_seqlens_from_lengths(lengths, device="cpu"):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32, device=device)


def varlen_lengths(n_seqs=32, low=512, high=65536, total_lo=450_000, total_hi=550_000, seed=0):
    """Log-uniform sequence lengths in [low, high]; re-draws with seed+1, +2, ... until the
    total lies in [total_lo, total_hi].  Returns (lengths, seed actually used)."""
    s = seed
    while True:
        rng = np.random.default_rng(s)
        u = rng.uniform(math.log(low), math.log(high), size=n_seqs)
        lens = np.clip(np.rint(np.exp(u)).astype(np.int64), low, high)
        if total_lo <= int(lens.sum()) <= total_hi:
            return [int(x) for x in lens], s
        s += 1


def kda_inputs(lengths, H, d, *, seed, device="cpu", io_dtype=torch.bfloat16,
               init_state=None, gate=False, state_dtype=torch.float32):
    """Packed prefill inputs for sequences of the given lengths.

    init_state: None (zeros), "all" (every sequence ~ N(0, 0.02)) or "even" (even-indexed
    sequences ~ N(0, 0.02), the rest zero).  Returns a dict of tensors on ``device``.
    """
    T = int(sum(lengths))
    N = len(lengths)
    out = {
        "q": normal((T, H, d), seed=seed * 32 + 1, device=device, dtype=io_dtype),
        "k": normal((T, H, d), seed=seed * 32 + 2, device=device, dtype=io_dtype),
        "v": normal((T, H, d), seed=seed * 32 + 3, device=device, dtype=io_dtype),
        "g": uniform((T, H, d), LOG_ALPHA_LOW, 0.0, seed=seed * 32 + 4, device=device),
        "beta": beta_draw((T, H), seed=seed * 32 + 5, device=device),
        "cu_seqlens": cu_seqlens_from_lengths(lengths, device=device),
    }
    if init_state is not None:
        s0 = normal((N, H, d, d), seed=seed * 32 + 6, device=device, dtype=torch.float32,
                    std=STATE_STD)
        if init_state == "even":
            s0[1::2] = 0.0
        out["init_state"] = s0.to(state_dtype)
    if gate:
        out["gate"] = normal((T, H, d), seed=seed * 32 + 7, device=device, dtype=io_dtype)
        out["norm_w"] = torch.ones(d, dtype=torch.float32, device=device)
    return out


def prologue_inputs(lengths, H, d, *, seed, device="cpu", io_dtype=torch.bfloat16,
                    conv_state=True):
    """Raw projections x [T, 3*H*d], conv weights [3*H*d, 4], conv state [N, 3, 3*H*d],
    beta logits [T, H] and raw log-retention [T, H, d]."""
    T = int(sum(lengths))
    N = len(lengths)
    C = 3 * H * d
    out = {
        "x": normal((T, C), seed=seed * 32 + 8, device=device, dtype=io_dtype),
        "conv_w": normal((C, 4), seed=seed * 32 + 9, device=device, dtype=io_dtype,
                         std=CONV_W_STD),
        "beta_logit": normal((T, H), seed=seed * 32 + 10, device=device, dtype=torch.float32),
        "g_raw": uniform((T, H, d), LOG_ALPHA_LOW, 0.0, seed=seed * 32 + 11, device=device),
        "cu_seqlens": cu_seqlens_from_lengths(lengths, device=device),
    }
    if conv_state:
        out["conv_state"] = normal((N, 3, C), seed=seed * 32 + 12, device=device,
                                   dtype=io_dtype)
    return out


def decode_inputs(n_seqs, H, d, *, seed, device="cpu", io_dtype=torch.bfloat16, gate=False):
    """One decode step's per-token inputs: raw x [N, 3*H*d], g [N, H, d], beta [N, H]."""
    C = 3 * H * d
    out = {
        "x": normal((n_seqs, C), seed=seed * 32 + 13, device=device, dtype=io_dtype),
        "g": uniform((n_seqs, H, d), LOG_ALPHA_LOW, 0.0, seed=seed * 32 + 14, device=device),
        "beta": beta_draw((n_seqs, H), seed=seed * 32 + 15, device=device),
    }
    if gate:
        out["gate"] = normal((n_seqs, H, d), seed=seed * 32 + 16, device=device, dtype=io_dtype)
    return out
