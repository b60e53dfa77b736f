"""Python binding of libkda.so (include/kda.h), argument marshalling only.

Each function has the name of the C entry point it calls, takes torch CUDA tensors (or None
for a NULL pointer), checks dtypes/devices/contiguity, passes raw pointers and the current
(or given) CUDA stream, and raises KdaError on a non-OK status.  All arithmetic runs in the
library's CUDA kernels; there is no fallback.  If libkda.so has not been built, loading it
raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_WORKSPACE, \
    KDA_ERR_TIMEOUT, KDA_ERR_BAD_INDEX, KDA_ERR_BAD_SEQLENS = 0, -1, -2, -3, -4, -5, -6, -7
KDA_F32, KDA_BF16 = 0, 1

_TORCH_OF = {KDA_F32: torch.float32, KDA_BF16: torch.bfloat16}

EXPORTS = (
    "kda_params_default", "kda_status_string", "kda_state_bytes", "kda_prefill_workspace_size",
    "kda_prologue", "kda_prefill", "kda_prefill_fp8", "kda_prefill_checkpointed",
    "kda_conv_tail_checkpoints", "kda_prefill_host_workspace_size", "kda_prefill_host",
    "kda_prefill_host_plan",
    "kda_decode_step", "kda_conv_state_update", "kda_decode_step_fused",
    "kda_decode_step_fused_fp8", "kda_decode_multi", "kda_state_accept",
    "kda_check_device_error", "kda_launch_count", "kda_trace_ranges", "kda_wait_probe",
    "mla_decode_workspace_size", "mla_set_split_override", "mla_decode_latent",
    "mla_decode_latent_noalloc", "mla_decode",
)


class KdaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


PREFILL_FORMS = {"auto": 0, "fused": 1, "pair": 2}


class KdaParams(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int), ("d_k", ctypes.c_int), ("d_v", ctypes.c_int),
        ("scale", ctypes.c_float), ("l2_eps", ctypes.c_float), ("norm_eps", ctypes.c_float),
        ("g_min", ctypes.c_float), ("qk_l2norm", ctypes.c_int),
        ("io_dtype", ctypes.c_int), ("state_dtype", ctypes.c_int),
        ("prefill_form", ctypes.c_int),
    ]

    @property
    def io_torch(self):
        return _TORCH_OF[self.io_dtype]

    @property
    def state_torch(self):
        return _TORCH_OF[self.state_dtype]


_lock = threading.Lock()
_lib = None
_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_P = ctypes.POINTER(KdaParams)


def load():
    """Loads libkda.so (built by hybrid_linear_attention_gb300.build.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "hybrid_linear_attention_gb300.build.build() (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        sig = {
            "kda_params_default": (None, [_P]),
            "kda_status_string": (ctypes.c_char_p, [_i32]),
            "kda_state_bytes": (_sz, [_P]),
            "kda_prefill_workspace_size": (_sz, [_P, _i32, _i64]),
            "kda_prologue": (_i32, [_P, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _vp, _vp,
                                    _vp, _vp, _vp, _vp, _vp, _vp]),
            "kda_prefill": (_i32, [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _vp, _vp,
                                   _vp, _vp, _vp, _sz, _vp]),
            "kda_prefill_fp8": (_i32, [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _vp,
                                       _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
            "kda_prefill_checkpointed": (_i32, [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                                _i64, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp,
                                                _vp, _sz, _vp]),
            "kda_conv_tail_checkpoints": (_i32, [_P, _vp, _vp, _vp, _i32, _i64, _vp, _vp, _i32,
                                                 _vp, _vp]),
            "kda_prefill_host_workspace_size": (_sz, [_P, _i32, _i64, _i32]),
            "kda_prefill_host": (_i32, [_P, _vp, _vp, _vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp,
                                        _vp, _vp, _vp, _vp, _sz, _i64, _vp]),
            "kda_prefill_host_plan": (_i64, [_vp, _i32, _i64, _i64, _vp, _i64]),
            "kda_decode_step": (_i32, [_P, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _vp,
                                       _vp, _vp, _vp]),
            "kda_conv_state_update": (_i32, [_P, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _vp,
                                             _vp]),
            "kda_decode_step_fused": (_i32, [_P, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32,
                                             _vp, _vp, _vp, _vp]),
            "kda_decode_step_fused_fp8": (_i32, [_P, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp,
                                                 _i32, _vp, _vp, _vp, _vp, _vp]),
            "kda_decode_multi": (_i32, [_P, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32,
                                        _vp, _vp, _vp, _vp, _i32, _vp]),
            "kda_state_accept": (_i32, [_P, _vp, _i32, _i32, _vp, _vp, _i32, _vp, _vp]),
            "kda_check_device_error": (_i32, [_vp]),
            "kda_launch_count": (ctypes.c_uint64, []),
            "kda_trace_ranges": (_i32, [ctypes.POINTER(ctypes.c_char_p), _i32]),
            "kda_wait_probe": (_i32, [_i64, _vp]),
            "mla_decode_workspace_size": (_sz, [_i32, _i64]),
            "mla_set_split_override": (_i32, [_i32]),
            "mla_decode_latent": (_i32, [_vp, _vp, _i64, _vp, _i32, ctypes.c_float, _vp, _vp,
                                         _sz, _vp]),
            "mla_decode_latent_noalloc": (_i32, [_vp, _vp, _i64, _vp, _i32, ctypes.c_float, _vp,
                                                 _vp]),
            "mla_decode": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _vp, _i32, _vp, ctypes.c_float,
                                  _vp, _vp, _vp, _vp, _sz, _vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status):
    try:
        return load().kda_status_string(int(status)).decode()
    except Exception:  # the library itself failed to load
        return f"status {status}"


def _check(status, where):
    if status != KDA_OK:
        raise KdaError(status, where)


def params(H=64, d=128, *, scale=1.0, l2_eps=1e-6, norm_eps=1e-6, g_min=-5.0, qk_l2norm=True,
           io_dtype=torch.bfloat16, state_dtype=torch.float32, prefill_form="auto"):
    """Builds a kda_params struct (defaults: the pages' configuration).  prefill_form:
    "auto", "fused" or "pair" (the tensor-core prefill's kernel form)."""
    code = {torch.float32: KDA_F32, torch.bfloat16: KDA_BF16}
    return KdaParams(H=H, d_k=d, d_v=d, scale=scale, l2_eps=l2_eps, norm_eps=norm_eps,
                     g_min=g_min, qk_l2norm=1 if qk_l2norm else 0,
                     io_dtype=code[io_dtype], state_dtype=code[state_dtype],
                     prefill_form=PREFILL_FORMS[prefill_form])


def kda_params_default():
    p = KdaParams()
    load().kda_params_default(ctypes.byref(p))
    return p


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor or None")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (device pointer)")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _hptr(t, dtype=None, name="tensor"):
    """Host pointer of a CPU tensor (page-locked memory lets the library overlap its copies)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor or None")
    if t.is_cuda:
        raise ValueError(f"{name}: must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


def kda_state_bytes(p):
    return int(load().kda_state_bytes(ctypes.byref(p)))


def kda_prefill_workspace_size(p, n_seqs, total_tokens):
    return int(load().kda_prefill_workspace_size(ctypes.byref(p), int(n_seqs), int(total_tokens)))


def kda_launch_count():
    return int(load().kda_launch_count())


def kda_wait_probe(probes, stream=None):
    _check(load().kda_wait_probe(int(probes), _stream(stream)), "kda_wait_probe")


def kda_check_device_error(stream=None):
    _check(load().kda_check_device_error(_stream(stream)), "kda_check_device_error")


def kda_prologue(p, x_raw, conv_w, conv_state, cu_seqlens, q, k, v, *, l2norm_qk=False,
                 beta_logit=None, g_raw=None, beta=None, g=None, stream=None):
    io = p.io_torch
    st = load().kda_prologue(
        ctypes.byref(p), _ptr(x_raw, io, "x_raw"), _ptr(conv_w, io, "conv_w"),
        _ptr(conv_state, io, "conv_state"), _ptr(cu_seqlens, torch.int32, "cu_seqlens"),
        cu_seqlens.numel() - 1, x_raw.shape[0], 1 if l2norm_qk else 0,
        _ptr(beta_logit, torch.float32, "beta_logit"), _ptr(g_raw, torch.float32, "g_raw"),
        _ptr(q, io, "q"), _ptr(k, io, "k"), _ptr(v, io, "v"),
        _ptr(beta, torch.float32, "beta"), _ptr(g, torch.float32, "g"), _stream(stream))
    _check(st, "kda_prologue")


def kda_prefill(p, q, k, v, g, beta, cu_seqlens, out, *, init_state=None, final_state=None,
                gate_logit=None, norm_w=None, workspace=None, stream=None):
    io, sd = p.io_torch, p.state_torch
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().kda_prefill(
        ctypes.byref(p), _ptr(q, io, "q"), _ptr(k, io, "k"), _ptr(v, io, "v"),
        _ptr(g, torch.float32, "g"), _ptr(beta, torch.float32, "beta"),
        _ptr(init_state, sd, "init_state"), _ptr(cu_seqlens, torch.int32, "cu_seqlens"),
        cu_seqlens.numel() - 1, q.shape[0], _ptr(gate_logit, io, "gate_logit"),
        _ptr(norm_w, torch.float32, "norm_w"), _ptr(out, io, "out"),
        _ptr(final_state, sd, "final_state"), _ptr(workspace, None, "workspace"), ws_bytes,
        _stream(stream))
    _check(st, "kda_prefill")


def kda_prefill_host_workspace_size(p, n_seqs, segment_tokens, with_gate=False):
    return int(load().kda_prefill_host_workspace_size(ctypes.byref(p), int(n_seqs),
                                                       int(segment_tokens), 1 if with_gate else 0))


def kda_prefill_host_plan(cu_seqlens, segment_tokens):
    """Row boundaries of the segments kda_prefill_host cuts a batch into (cu_seqlens: a CPU
    int32 tensor); a list [0, b_1, ..., total_tokens]."""
    cu = cu_seqlens.to(torch.int32).contiguous()
    n, T = cu.numel() - 1, int(cu[-1])
    k = load().kda_prefill_host_plan(_hptr(cu, torch.int32, "cu_seqlens"), n, T,
                                     int(segment_tokens), None, 0)
    if k < 0:
        raise KdaError(KDA_ERR_INVALID_ARG, "kda_prefill_host_plan")
    bounds = (ctypes.c_int64 * (k + 1))()
    load().kda_prefill_host_plan(_hptr(cu, torch.int32, "cu_seqlens"), n, T,
                                 int(segment_tokens), bounds, k)
    return [int(b) for b in bounds] if k > 0 else [0]


def kda_prefill_host(p, x_raw, conv_w, conv_state, cu_seqlens, beta_logit, g_raw, out, *,
                     workspace, segment_tokens=512, init_state=None, final_state=None,
                     gate_logit=None, norm_w=None, stream=None):
    """Prologue + prefill of a packed batch in host memory, streamed through the GPU in
    segments: x_raw, conv_state (in/out or None), cu_seqlens (int32), beta_logit, g_raw,
    init_state, gate_logit, out and final_state are CPU tensors (pinned for overlap); conv_w,
    norm_w and the uint8 workspace are CUDA tensors.  The outputs are in host memory once
    `stream` (default: the current stream) has been synchronised."""
    io = p.io_torch
    st = load().kda_prefill_host(
        ctypes.byref(p), _hptr(x_raw, io, "x_raw"), _ptr(conv_w, io, "conv_w"),
        _hptr(conv_state, io, "conv_state"), _hptr(cu_seqlens, torch.int32, "cu_seqlens"),
        cu_seqlens.numel() - 1, x_raw.shape[0], _hptr(beta_logit, torch.float32, "beta_logit"),
        _hptr(g_raw, torch.float32, "g_raw"), _hptr(init_state, torch.float32, "init_state"),
        _hptr(gate_logit, io, "gate_logit"), _ptr(norm_w, torch.float32, "norm_w"),
        _hptr(out, io, "out"), _hptr(final_state, torch.float32, "final_state"),
        *_ws(workspace), int(segment_tokens), _stream(stream))
    _check(st, "kda_prefill_host")


def kda_prefill_fp8(p, q, k, v, g, beta, cu_seqlens, out_q, out_scale, *, init_state=None,
                    final_state=None, gate_logit=None, norm_w=None, workspace=None, stream=None):
    """out_q [T, H, d] uint8 E4M3 codes, out_scale [T, H] fp32 (one group per token, head)."""
    io, sd = p.io_torch, p.state_torch
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().kda_prefill_fp8(
        ctypes.byref(p), _ptr(q, io, "q"), _ptr(k, io, "k"), _ptr(v, io, "v"),
        _ptr(g, torch.float32, "g"), _ptr(beta, torch.float32, "beta"),
        _ptr(init_state, sd, "init_state"), _ptr(cu_seqlens, torch.int32, "cu_seqlens"),
        cu_seqlens.numel() - 1, q.shape[0], _ptr(gate_logit, io, "gate_logit"),
        _ptr(norm_w, torch.float32, "norm_w"), _ptr(out_q, torch.uint8, "out_q"),
        _ptr(out_scale, torch.float32, "out_scale"), _ptr(final_state, sd, "final_state"),
        _ptr(workspace, None, "workspace"), ws_bytes, _stream(stream))
    _check(st, "kda_prefill_fp8")


def kda_prefill_checkpointed(p, q, k, v, g, beta, cu_seqlens, out, ckpt_cu, ckpt_pos,
                             ckpt_states, *, init_state=None, final_state=None, gate_logit=None,
                             norm_w=None, workspace=None, stream=None):
    io, sd = p.io_torch, p.state_torch
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().kda_prefill_checkpointed(
        ctypes.byref(p), _ptr(q, io, "q"), _ptr(k, io, "k"), _ptr(v, io, "v"),
        _ptr(g, torch.float32, "g"), _ptr(beta, torch.float32, "beta"),
        _ptr(init_state, sd, "init_state"), _ptr(cu_seqlens, torch.int32, "cu_seqlens"),
        cu_seqlens.numel() - 1, q.shape[0], _ptr(gate_logit, io, "gate_logit"),
        _ptr(norm_w, torch.float32, "norm_w"), _ptr(out, io, "out"),
        _ptr(final_state, sd, "final_state"), _ptr(ckpt_cu, torch.int32, "ckpt_cu"),
        _ptr(ckpt_pos, torch.int32, "ckpt_pos"), ckpt_pos.numel(),
        _ptr(ckpt_states, sd, "ckpt_states"), _ptr(workspace, None, "workspace"), ws_bytes,
        _stream(stream))
    _check(st, "kda_prefill_checkpointed")


def kda_conv_tail_checkpoints(p, x_raw, conv_state, cu_seqlens, ckpt_cu, ckpt_pos, conv_ckpt, *,
                              stream=None):
    io = p.io_torch
    st = load().kda_conv_tail_checkpoints(
        ctypes.byref(p), _ptr(x_raw, io, "x_raw"), _ptr(conv_state, io, "conv_state"),
        _ptr(cu_seqlens, torch.int32, "cu_seqlens"), cu_seqlens.numel() - 1, x_raw.shape[0],
        _ptr(ckpt_cu, torch.int32, "ckpt_cu"), _ptr(ckpt_pos, torch.int32, "ckpt_pos"),
        ckpt_pos.numel(), _ptr(conv_ckpt, io, "conv_ckpt"), _stream(stream))
    _check(st, "kda_conv_tail_checkpoints")


def kda_decode_step(p, q, k, v, g, beta, state, out, *, slot_idx=None, gate_logit=None,
                    norm_w=None, stream=None):
    io, sd = p.io_torch, p.state_torch
    st = load().kda_decode_step(
        ctypes.byref(p), _ptr(q, io, "q"), _ptr(k, io, "k"), _ptr(v, io, "v"),
        _ptr(g, torch.float32, "g"), _ptr(beta, torch.float32, "beta"),
        _ptr(state, sd, "state"), state.shape[0], _ptr(slot_idx, torch.int32, "slot_idx"),
        q.shape[0], _ptr(gate_logit, io, "gate_logit"), _ptr(norm_w, torch.float32, "norm_w"),
        _ptr(out, io, "out"), _stream(stream))
    _check(st, "kda_decode_step")


def kda_decode_step_fused(p, x_raw, conv_w, conv_state, g, beta, state, out, *, slot_idx=None,
                          gate_logit=None, norm_w=None, stream=None):
    io, sd = p.io_torch, p.state_torch
    st = load().kda_decode_step_fused(
        ctypes.byref(p), _ptr(x_raw, io, "x_raw"), _ptr(conv_w, io, "conv_w"),
        _ptr(conv_state, io, "conv_state"), _ptr(g, torch.float32, "g"),
        _ptr(beta, torch.float32, "beta"), _ptr(state, sd, "state"), state.shape[0],
        _ptr(slot_idx, torch.int32, "slot_idx"), x_raw.shape[0],
        _ptr(gate_logit, io, "gate_logit"), _ptr(norm_w, torch.float32, "norm_w"),
        _ptr(out, io, "out"), _stream(stream))
    _check(st, "kda_decode_step_fused")


def kda_decode_step_fused_fp8(p, x_raw, conv_w, conv_state, g, beta, state, out_q, out_scale, *,
                              slot_idx=None, gate_logit=None, norm_w=None, stream=None):
    """out_q [n_seqs, H, d] uint8 E4M3 codes, out_scale [n_seqs, H] fp32."""
    io, sd = p.io_torch, p.state_torch
    st = load().kda_decode_step_fused_fp8(
        ctypes.byref(p), _ptr(x_raw, io, "x_raw"), _ptr(conv_w, io, "conv_w"),
        _ptr(conv_state, io, "conv_state"), _ptr(g, torch.float32, "g"),
        _ptr(beta, torch.float32, "beta"), _ptr(state, sd, "state"), state.shape[0],
        _ptr(slot_idx, torch.int32, "slot_idx"), x_raw.shape[0],
        _ptr(gate_logit, io, "gate_logit"), _ptr(norm_w, torch.float32, "norm_w"),
        _ptr(out_q, torch.uint8, "out_q"), _ptr(out_scale, torch.float32, "out_scale"),
        _stream(stream))
    _check(st, "kda_decode_step_fused_fp8")


def kda_decode_multi(p, q, k, v, g, beta, state, out, K, *, slot_idx=None, gate_logit=None,
                     norm_w=None, step_states=None, commit_final=False, stream=None):
    """K tokens per sequence: q, k, v, g, beta, out, gate_logit have n_seqs * K rows."""
    io, sd = p.io_torch, p.state_torch
    if q.shape[0] % K:
        raise ValueError("rows must be n_seqs * K")
    st = load().kda_decode_multi(
        ctypes.byref(p), _ptr(q, io, "q"), _ptr(k, io, "k"), _ptr(v, io, "v"),
        _ptr(g, torch.float32, "g"), _ptr(beta, torch.float32, "beta"),
        _ptr(state, sd, "state"), state.shape[0], _ptr(slot_idx, torch.int32, "slot_idx"),
        q.shape[0] // K, K, _ptr(gate_logit, io, "gate_logit"),
        _ptr(norm_w, torch.float32, "norm_w"), _ptr(out, io, "out"),
        _ptr(step_states, sd, "step_states"), 1 if commit_final else 0, _stream(stream))
    _check(st, "kda_decode_multi")


def kda_state_accept(p, step_states, accept_len, state, K, *, slot_idx=None, stream=None):
    sd = p.state_torch
    st = load().kda_state_accept(
        ctypes.byref(p), _ptr(step_states, sd, "step_states"), accept_len.shape[0], K,
        _ptr(accept_len, torch.int32, "accept_len"), _ptr(state, sd, "state"), state.shape[0],
        _ptr(slot_idx, torch.int32, "slot_idx"), _stream(stream))
    _check(st, "kda_state_accept")


def kda_conv_state_update(p, x_new, conv_w, conv_state, y, *, slot_idx=None, stream=None):
    io = p.io_torch
    st = load().kda_conv_state_update(
        ctypes.byref(p), _ptr(x_new, io, "x_new"), _ptr(conv_w, io, "conv_w"),
        _ptr(conv_state, io, "conv_state"), conv_state.shape[0],
        _ptr(slot_idx, torch.int32, "slot_idx"), x_new.shape[0], x_new.shape[1],
        _ptr(y, io, "y"), _stream(stream))
    _check(st, "kda_conv_state_update")


# ---- absorbed gated-MLA decode (mla.h) -----------------------------------------------------

MLA_SCALE = 192 ** -0.5


def kda_trace_ranges():
    """Names of the NVTX ranges the library opens around its calls."""
    lib = load()
    n = lib.kda_trace_ranges(None, 0)
    arr = (ctypes.c_char_p * n)()
    lib.kda_trace_ranges(arr, n)
    return [x.decode() for x in arr]


def mla_decode_workspace_size(n_seqs, cache_len):
    return int(load().mla_decode_workspace_size(int(n_seqs), int(cache_len)))


def mla_set_split_override(n_split):
    """Tuning and testing only: force the MLA split count (0 = the automatic rule)."""
    _check(load().mla_set_split_override(int(n_split)), "mla_set_split_override")


class mla_split:
    """Context manager: the MLA split count forced to n inside the block."""

    def __init__(self, n):
        self.n = n

    def __enter__(self):
        mla_set_split_override(self.n)

    def __exit__(self, *exc):
        mla_set_split_override(0)


def _ws(workspace):
    return (_ptr(workspace, None, "workspace"),
            workspace.numel() * workspace.element_size() if workspace is not None else 0)


def mla_decode_latent(q_cat, cache, lengths, z, *, scale=MLA_SCALE, workspace=None, stream=None):
    """q_cat [B,64,576] bf16, cache [B,L,576] bf16, lengths [B] int32, z [B,64,512] fp32."""
    st = load().mla_decode_latent(
        _ptr(q_cat, torch.bfloat16, "q_cat"), _ptr(cache, torch.bfloat16, "cache"),
        cache.shape[1], _ptr(lengths, torch.int32, "lengths"), q_cat.shape[0], float(scale),
        _ptr(z, torch.float32, "z"), *_ws(workspace), _stream(stream))
    _check(st, "mla_decode_latent")


def mla_decode_latent_noalloc(q_cat, cache, lengths, z, *, scale=MLA_SCALE, stream=None):
    """mla_decode_latent with its split scratch in the library's fixed device buffer."""
    st = load().mla_decode_latent_noalloc(
        _ptr(q_cat, torch.bfloat16, "q_cat"), _ptr(cache, torch.bfloat16, "cache"),
        cache.shape[1], _ptr(lengths, torch.int32, "lengths"), q_cat.shape[0], float(scale),
        _ptr(z, torch.float32, "z"), _stream(stream))
    _check(st, "mla_decode_latent_noalloc")


def mla_decode(q_nope, q_rope, w_uk, w_uv, cache, lengths, gate_logit, q_cat, z, out, *,
               scale=MLA_SCALE, workspace=None, stream=None):
    """One absorbed gated-MLA decode step; q_cat and z are caller-owned intermediates."""
    bf = torch.bfloat16
    st = load().mla_decode(
        _ptr(q_nope, bf, "q_nope"), _ptr(q_rope, bf, "q_rope"), _ptr(w_uk, bf, "w_uk"),
        _ptr(w_uv, bf, "w_uv"), _ptr(cache, bf, "cache"), cache.shape[1],
        _ptr(lengths, torch.int32, "lengths"), q_nope.shape[0], _ptr(gate_logit, bf, "gate_logit"),
        float(scale), _ptr(q_cat, bf, "q_cat"), _ptr(z, torch.float32, "z"), _ptr(out, bf, "out"),
        *_ws(workspace), _stream(stream))
    _check(st, "mla_decode")
