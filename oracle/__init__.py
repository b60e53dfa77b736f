"""The oracle for the Kimi Delta Attention (KDA) token mixer.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the benchmark's
CPU-baseline leg may import this package; the product path never does.  It shares no code
with the CUDA library and never imports it.

``kda_oracle.c`` holds the KDA arithmetic (plain C, fp64, token by token); this module
builds it with gcc and marshals numpy arrays into it.  The FP8 output quantiser and the
absorbed gated-MLA decode are written here in plain numpy (fp64, position by position).
Every function returns results computed from the exact stored values of its inputs (fp32
arrays, or bf16 given as the ``torch.bfloat16`` / raw uint16 bit patterns).

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py`` (closed forms,
invariants, brute force and library routines); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")

F32, BF16, F64 = 0, 1, 2
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles kda_oracle.c with gcc into oracle/_build/libkda_oracle.so (plain -O2)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _KdaArgs(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
        ("n_seqs", ctypes.c_int), ("cu_seqlens", ctypes.c_void_p),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("qkv_dtype", ctypes.c_int),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("init_state", ctypes.c_void_p), ("state_dtype", ctypes.c_int),
        ("gate", ctypes.c_void_p), ("gate_dtype", ctypes.c_int),
        ("norm_w", ctypes.c_void_p),
        ("scale", ctypes.c_double), ("l2_eps", ctypes.c_double),
        ("norm_eps", ctypes.c_double), ("g_min", ctypes.c_double),
        ("qk_l2norm", ctypes.c_int),
        ("n_units", ctypes.c_int), ("units", ctypes.c_void_p),
        ("out_offset", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("final_state", ctypes.c_void_p), ("state_norm", ctypes.c_void_p),
        ("n_threads", ctypes.c_int),
    ]


class _ProArgs(ctypes.Structure):
    _fields_ = [
        ("n_seqs", ctypes.c_int), ("cu_seqlens", ctypes.c_void_p),
        ("H", ctypes.c_int), ("d", ctypes.c_int),
        ("x", ctypes.c_void_p), ("x_dtype", ctypes.c_int),
        ("w", ctypes.c_void_p), ("w_dtype", ctypes.c_int),
        ("conv_state_in", ctypes.c_void_p), ("conv_state_out", ctypes.c_void_p),
        ("l2norm_qk", ctypes.c_int), ("l2_eps", ctypes.c_double),
        ("y", ctypes.c_void_p),
        ("beta_logit", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("g_raw", ctypes.c_void_p), ("g", ctypes.c_void_p), ("g_min", ctypes.c_double),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_kda_forward.argtypes = [ctypes.POINTER(_KdaArgs)]
            lib.oracle_kda_forward.restype = ctypes.c_int
            lib.oracle_prologue.argtypes = [ctypes.POINTER(_ProArgs)]
            lib.oracle_prologue.restype = ctypes.c_int
            lib.oracle_state_bytes.argtypes = [ctypes.c_int] * 4
            lib.oracle_state_bytes.restype = ctypes.c_int64
            lib.oracle_conv_tail_bytes.argtypes = [ctypes.c_int] * 4
            lib.oracle_conv_tail_bytes.restype = ctypes.c_int64
            _lib = lib
    return _lib


def _as_np(x):
    """Returns (contiguous numpy array, dtype code).  bf16 torch tensors become uint16 bits."""
    if x is None:
        return None, F32
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float32:
                return x.numpy(), F32
            if x.dtype == torch.float64:
                return x.numpy(), F64
            if x.dtype == torch.int32:
                return x.numpy(), F32
            raise TypeError(f"oracle: unsupported tensor dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, BF16
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.int32:
        return x, F32
    raise TypeError(f"oracle: unsupported array dtype {x.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def kda_forward(q, k, v, g, beta, cu_seqlens, *, init_state=None, gate=None, norm_w=None,
                scale=1.0, l2_eps=1e-6, norm_eps=1e-6, g_min=-5.0, qk_l2norm=True,
                units=None, n_threads=None, want_state_norm=False):
    """Token-by-token fp64 KDA over a packed batch.

    q, k: [T_tot, H, dk]; v: [T_tot, H, dv] (fp32 or bf16); g: [T_tot, H, dk] fp32 raw
    log-retention (clamped at g_min here); beta: [T_tot, H] fp32 in (0, 1);
    cu_seqlens: int32 [N + 1]; init_state: [N, H, dk, dv] or None; gate: [T_tot, H, dv]
    output-gate logits or None (no output norm); norm_w: [dv] fp32 or None (ones).
    units: list of (sequence, head) to compute, default all.

    Returns dict(out=[T_tot, H, dv] fp64 when every unit is computed, otherwise
    unit_out=list of [len, dv] arrays), final_state=[n_units, dk, dv] fp64 (in the units'
    order; reshaped to [N, H, dk, dv] when all units are computed), and state_norm when asked.
    """
    lib = _load()
    qn, qdt = _as_np(q)
    kn, kdt = _as_np(k)
    vn, vdt = _as_np(v)
    if not (qdt == kdt == vdt):
        raise TypeError("oracle: q, k, v must share a storage type")
    gn, _ = _as_np(g)
    bn, _ = _as_np(beta)
    cu, _ = _as_np(cu_seqlens)
    cu = cu.astype(np.int32)
    T, H, dk = qn.shape
    dv = vn.shape[2]
    N = cu.shape[0] - 1
    sn, sdt = _as_np(init_state)
    gt, gdt = _as_np(gate)
    wn, _ = _as_np(norm_w)
    full = units is None
    if full:
        units = [(n, h) for n in range(N) for h in range(H)]
    units_arr = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
    lens = np.array([cu[n + 1] - cu[n] for n, _ in units_arr], dtype=np.int64)
    # each unit's [len, dv] block is written contiguously; the full [T, H, dv] view is
    # scattered together afterwards
    offs = np.zeros(len(units_arr), dtype=np.int64)
    if len(units_arr):
        offs[1:] = np.cumsum(lens[:-1] * dv)
    out = np.zeros(int(lens.sum()) * dv, dtype=np.float64)
    fin = np.zeros((len(units_arr), dk, dv), dtype=np.float64)
    snorm = np.zeros(int(lens.sum()), dtype=np.float64) if want_state_norm else None
    args = _KdaArgs(
        H=H, dk=dk, dv=dv, n_seqs=N, cu_seqlens=_ptr(cu),
        q=_ptr(qn), k=_ptr(kn), v=_ptr(vn), qkv_dtype=qdt,
        g=_ptr(gn), beta=_ptr(bn),
        init_state=_ptr(sn), state_dtype=sdt,
        gate=_ptr(gt), gate_dtype=gdt, norm_w=_ptr(wn),
        scale=scale, l2_eps=l2_eps, norm_eps=norm_eps, g_min=g_min,
        qk_l2norm=1 if qk_l2norm else 0,
        n_units=len(units_arr), units=_ptr(units_arr), out_offset=_ptr(offs),
        out=_ptr(out), final_state=_ptr(fin), state_norm=_ptr(snorm),
        n_threads=n_threads or (os.cpu_count() or 1),
    )
    if lib.oracle_kda_forward(ctypes.byref(args)) != 0:
        raise ValueError("oracle_kda_forward rejected its arguments")
    res = {}
    unit_out = [out[o:o + l * dv].reshape(l, dv) for o, l in zip(offs, lens)]
    if full:
        o_full = np.zeros((T, H, dv), dtype=np.float64)
        for (n, h), uo in zip(units_arr, unit_out):
            o_full[cu[n]:cu[n + 1], h, :] = uo
        res["out"] = o_full
        res["final_state"] = fin.reshape(N, H, dk, dv)
    else:
        res["unit_out"] = unit_out
        res["final_state"] = fin
    if want_state_norm:
        res["state_norm"] = [snorm[o // dv:o // dv + l] for o, l in zip(offs, lens)]
    return res


def prologue(x, conv_w, cu_seqlens, H, d, *, conv_state=None, l2norm_qk=False, l2_eps=1e-6,
             beta_logit=None, g_raw=None, g_min=-5.0):
    """Width-4 causal short convolution + SiLU over the concatenated q|k|v streams.

    x: [T_tot, 3*H*d] (fp32 or bf16); conv_w: [3*H*d, 4]; conv_state: [N, 3, 3*H*d] in x's
    storage type or None.  Returns dict(y=[T_tot, 3*H*d] fp64, conv_state=[N, 3, 3*H*d] in
    x's storage type (numpy; uint16 bits for bf16), beta, g when their inputs are given).
    """
    lib = _load()
    xn, xdt = _as_np(x)
    wn, wdt = _as_np(conv_w)
    cu, _ = _as_np(cu_seqlens)
    cu = cu.astype(np.int32)
    N = cu.shape[0] - 1
    C = 3 * H * d
    T = xn.shape[0]
    sn, sdt = _as_np(conv_state)
    if sn is not None and sdt != xdt:
        raise TypeError("oracle: conv state must share x's storage type")
    y = np.zeros((T, C), dtype=np.float64)
    st_out = np.zeros((N, 3, C), dtype=xn.dtype)
    bl, _ = _as_np(beta_logit)
    gr, _ = _as_np(g_raw)
    beta = np.zeros(bl.shape, dtype=np.float64) if bl is not None else None
    g = np.zeros(gr.shape, dtype=np.float64) if gr is not None else None
    args = _ProArgs(
        n_seqs=N, cu_seqlens=_ptr(cu), H=H, d=d, x=_ptr(xn), x_dtype=xdt,
        w=_ptr(wn), w_dtype=wdt, conv_state_in=_ptr(sn), conv_state_out=_ptr(st_out),
        l2norm_qk=1 if l2norm_qk else 0, l2_eps=l2_eps, y=_ptr(y),
        beta_logit=_ptr(bl), beta=_ptr(beta), g_raw=_ptr(gr), g=_ptr(g), g_min=g_min,
    )
    if lib.oracle_prologue(ctypes.byref(args)) != 0:
        raise ValueError("oracle_prologue rejected its arguments")
    res = {"y": y, "conv_state": st_out}
    if beta is not None:
        res["beta"] = beta
    if g is not None:
        res["g"] = g
    return res


def state_bytes(H, dk, dv, elem_bytes):
    """Bytes of one layer's recurrent state for one sequence."""
    return int(_load().oracle_state_bytes(H, dk, dv, elem_bytes))


def conv_tail_bytes(H, d, width, elem_bytes):
    """Bytes of one layer's short-convolution tail for one sequence."""
    return int(_load().oracle_conv_tail_bytes(H, d, width, elem_bytes))


# ---------------------------------------------------------------------------------------
# FP8 output quantisation
# ---------------------------------------------------------------------------------------
# The checkpoint stores block-FP8 E4M3 weights in 128 x 128 scaling blocks and quantises
# activations dynamically ("Ling-3.1-flash: Grouped Routing and Two Different MLA Caches",
# section "Production boundaries"); the serving setup fuses the quantisation of the KDA output
# feeding o_proj into the KDA kernel ("Ling-3.1-flash: What 63 Linear-Attention Layers Do to
# the KV Budget", section "Fitting it on a node").  Reading: the activation-side counterpart
# of the weights' block scaling -- one group per (token, head), the 128 value channels that
# meet one 128-row block of o_proj's weight -- with the dynamic scale s = a / 448,
# a = max(amax, 1e-10), so that the group's largest magnitude lands on E4M3's largest finite
# value; code = E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
# largest finite 448) of x / s, rounded to nearest even and saturated.  Everything in fp64.

FP8_MAX = 448.0
FP8_EPS = 1e-10


def fp8_e4m3_encode(y):
    """E4M3 codes (uint8) of the values y, rounded to the nearest representable value (ties
    to the even code) and saturated at +-448; NaN maps to 0x7F.  Works in the precision of
    y's dtype: the scaling by powers of two below is exact."""
    y = np.asarray(y)
    a = np.abs(y)
    sign = np.signbit(y).astype(np.uint8) << 7
    code = np.zeros(a.shape, dtype=np.int64)
    # subnormals and zero: multiples of 2^-9 below 2^-6 (an exact 2^-6 rounds up into the
    # first normal binade, code 8 = exponent field 1, mantissa 0: the same value)
    sub = a < 2.0 ** -6
    code[sub] = np.round(a[sub] * 2.0 ** 9).astype(np.int64)
    nrm = ~sub & np.isfinite(a)
    e = np.floor(np.log2(np.where(nrm, a, 1.0))).astype(np.int64)
    # guard log2 rounding at binade edges
    e = np.where(nrm & (np.ldexp(np.ones_like(a), e) > a), e - 1, e)
    e = np.where(nrm & (np.ldexp(np.ones_like(a), e + 1) <= a), e + 1, e)
    m = np.round(np.ldexp(np.where(nrm, a, 1.0), -e) * 8.0).astype(np.int64) - 8  # 0 .. 8
    carry = m == 8
    e = np.where(carry, e + 1, e)
    m = np.where(carry, 0, m)
    code = np.where(nrm, ((e + 7) << 3) | m, code)
    code = np.where(nrm & (e + 7 > 15), 0x7F, code)
    code = np.minimum(code, 0x7E)  # above 448 (including the NaN slot 0x7F): saturate
    code = np.where(np.isinf(a), 0x7E, code)
    out = (code.astype(np.uint8) | sign).astype(np.uint8)
    return np.where(np.isnan(y), np.uint8(0x7F), out)


def fp8_e4m3_decode(codes):
    """fp64 values of E4M3 codes (0x7F / 0xFF decode to NaN)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef, m = (c >> 3) & 0xF, c & 0x7
    val = np.where(ef == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(ef.astype(np.float64) - 7))
    val = np.where((ef == 15) & (m == 7), np.nan, val)
    return s * val


def fp8_quantize_groups(x, group=128):
    """Dynamic FP8 quantisation of the last axis of x in groups of `group` channels, in
    fp64: returns (codes uint8 with x's shape, fp64 scales with x.shape[:-1] + (n_groups,)),
    scale = max(amax, 1e-10) / 448 and code = E4M3(x / scale)."""
    x = np.asarray(x, dtype=np.float64)
    shp = x.shape
    xg = x.reshape(shp[:-1] + (shp[-1] // group, group))
    scale = np.maximum(np.abs(xg).max(axis=-1), FP8_EPS) / FP8_MAX
    codes = fp8_e4m3_encode(xg / scale[..., None])
    return codes.reshape(shp), scale


def fp8_dequantize_groups(codes, scales, group=128):
    """fp64 values of grouped codes: code value x the group's scale."""
    c = np.asarray(codes)
    shp = c.shape
    v = fp8_e4m3_decode(c).reshape(shp[:-1] + (shp[-1] // group, group))
    return (v * np.asarray(scales, dtype=np.float64)[..., None]).reshape(shp)


# ---------------------------------------------------------------------------------------
# Absorbed gated-MLA decode (the other token mixer of the hybrid)
# ---------------------------------------------------------------------------------------
# "Ling-3.1-flash: Grouped Routing and Two Different MLA Caches", sections "MLA's expanded
# reference path" and "Why weight absorption keeps the same attention function".  Per head
# i, the cached latent c_t (512) and shared rotated positional key r_t (64) of every cached
# position t; key up-projection W_K,i and value up-projection W_V,i, each 128 x 512; query
# parts q_i^N (128) and q_i^R (64, already rotated); score scale 1/sqrt(192); one sigmoid
# gate per head on the head's 128-wide output.  Plain fp64, position by position.

def _f64(x):
    a, _ = _as_np(x)
    if a is None:
        return None
    if a.dtype == np.uint16:  # bf16 bit patterns
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _softmax(s):
    e = np.exp(s - s.max())
    return e / e.sum()


def mla_decode_expanded(q_nope, q_rope, c, r, lengths, w_uk, w_uv, gate_logit,
                        scale=192 ** -0.5):
    """The expanded reference path: keys [W_K,i c_t ; r_t] (192 wide) and values W_V,i c_t
    (128 wide) for every cached position t < lengths[b]; softmax of scale * q . k; the
    weighted value sum times sigmoid(gate).  q_nope [B,H,128], q_rope [B,H,64], c [B,L,512],
    r [B,L,64], w_uk / w_uv [H,128,512], gate_logit [B,H].  Returns [B,H,128] fp64."""
    qn, qr, cc, rr = _f64(q_nope), _f64(q_rope), _f64(c), _f64(r)
    wk, wv, gl = _f64(w_uk), _f64(w_uv), _f64(gate_logit)
    B, H, dv = qn.shape[0], qn.shape[1], wv.shape[1]
    out = np.zeros((B, H, dv))
    for b in range(B):
        L = int(lengths[b])
        for i in range(H):
            keys = np.concatenate([cc[b, :L] @ wk[i].T, rr[b, :L]], axis=1)   # [L, 192]
            vals = cc[b, :L] @ wv[i].T                                       # [L, 128]
            q = np.concatenate([qn[b, i], qr[b, i]])
            p = _softmax(scale * (keys @ q))
            out[b, i] = (p @ vals) / (1.0 + np.exp(-gl[b, i]))
    return out


def mla_absorb(q_nope, q_rope, w_uk):
    """The absorbed query: [W_K,i^T q_i^N ; q_i^R], 576 wide per head.  Returns [B,H,576]."""
    qn, qr, wk = _f64(q_nope), _f64(q_rope), _f64(w_uk)
    qt = np.einsum("bhn,hnl->bhl", qn, wk)
    return np.concatenate([qt, qr], axis=2)


def mla_latent_attention(q_cat, cache, lengths, scale=192 ** -0.5):
    """The absorbed attention over the shared 576-wide cached key [c_t ; r_t], with the
    latent c_t itself as the value: per head, z = sum_t softmax_t(scale q . [c_t; r_t]) c_t.
    q_cat [B,H,576], cache [B,L,576].  Returns (z [B,H,512], lse [B,H]) in fp64, lse the
    natural log-sum-exp of the scaled scores."""
    q, kv = _f64(q_cat), _f64(cache)
    B, H = q.shape[0], q.shape[1]
    dl = kv.shape[2] - 64
    z = np.zeros((B, H, dl))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        L = int(lengths[b])
        if L == 0:
            continue
        for i in range(H):
            s = scale * (kv[b, :L] @ q[b, i])
            m = s.max()
            e = np.exp(s - m)
            z[b, i] = (e @ kv[b, :L, :dl]) / e.sum()
            lse[b, i] = m + np.log(e.sum())
    return z, lse


def mla_up_gate(z, w_uv, gate_logit):
    """The value up-projection after the latent sum, then the head's sigmoid gate:
    o_i = W_V,i z_i * sigmoid(gate_i).  z [B,H,512], w_uv [H,128,512], gate_logit [B,H]."""
    zz, wv, gl = _f64(z), _f64(w_uv), _f64(gate_logit)
    return np.einsum("bhl,hvl->bhv", zz, wv) / (1.0 + np.exp(-gl))[..., None]


def mla_decode_absorbed(q_nope, q_rope, c, r, lengths, w_uk, w_uv, gate_logit,
                        scale=192 ** -0.5):
    """The absorbed path: absorb the key up-projection into the query, attend over the
    576-wide cache with the latent as the value, project after the sum, gate."""
    cache = np.concatenate([_f64(c), _f64(r)], axis=2)
    z, _ = mla_latent_attention(mla_absorb(q_nope, q_rope, w_uk), cache, lengths, scale)
    return mla_up_gate(z, w_uv, gate_logit)
