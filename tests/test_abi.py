"""The C-ABI library loads, exports every entry point include/*.h declares, and rejects
bad arguments on the host before touching the GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest
import torch

from hybrid_linear_attention_gb300 import build as kbuild
from hybrid_linear_attention_gb300 import kda

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load()


def _declared_functions():
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
            names |= set(re.findall(r"\b((?:kda|mla)_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_contract_calls():
    names = _declared_functions()
    for must in ("kda_prefill", "kda_decode_step", "kda_conv_state_update", "kda_prologue",
                 "kda_prefill_workspace_size", "kda_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libkda.so does not export {name}"
    assert set(_declared_functions()) <= set(kda.EXPORTS)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert kda.status_string(code).startswith("KDA_")


def test_defaults_are_the_pages_configuration(lib):
    p = kda.kda_params_default()
    assert (p.H, p.d_k, p.d_v, p.qk_l2norm) == (64, 128, 128, 1)
    assert p.g_min == -5.0 and p.scale == 1.0
    assert p.io_dtype == kda.KDA_BF16 and p.state_dtype == kda.KDA_F32


def test_state_bytes_is_the_pages_payload(lib):
    p = kda.params()
    assert kda.kda_state_bytes(p) == 64 * 128 * 128 * 4            # 4 MiB per layer
    assert 63 * kda.kda_state_bytes(p) == 252 * 2**20             # 252 MiB per sequence
    pb = kda.params(state_dtype=torch.bfloat16)
    assert 63 * kda.kda_state_bytes(pb) == 126 * 2**20


def _raw_prefill(lib, p, **kw):
    args = dict(q=16, k=16, v=16, g=16, beta=16, init=None, cu=16, n=1, T=4, gate=None,
                w=None, out=16, fin=None, ws=None, wsb=0)
    args.update(kw)
    return lib.kda_prefill(ctypes.byref(p) if p is not None else None, args["q"], args["k"],
                           args["v"], args["g"], args["beta"], args["init"], args["cu"],
                           args["n"], args["T"], args["gate"], args["w"], args["out"],
                           args["fin"], args["ws"], args["wsb"], None)


def test_prefill_rejects_bad_arguments_on_host(lib):
    p = kda.params()
    assert _raw_prefill(lib, None) == kda.KDA_ERR_INVALID_ARG
    assert _raw_prefill(lib, p, q=None) == kda.KDA_ERR_INVALID_ARG
    assert _raw_prefill(lib, p, cu=None) == kda.KDA_ERR_INVALID_ARG
    assert _raw_prefill(lib, p, n=-1) == kda.KDA_ERR_INVALID_ARG
    assert _raw_prefill(lib, p, n=0, T=5) == kda.KDA_ERR_INVALID_ARG
    assert _raw_prefill(lib, p, q=18) == kda.KDA_ERR_INVALID_ARG          # misaligned
    assert _raw_prefill(lib, p, n=0, T=0) == kda.KDA_OK                   # nothing to do
    bad = kda.params(d=64)
    assert _raw_prefill(lib, bad) == kda.KDA_ERR_UNSUPPORTED
    mixed = kda.params()
    mixed.d_v = 16
    assert _raw_prefill(lib, mixed) == kda.KDA_ERR_UNSUPPORTED
    neg = kda.params(H=0)
    assert _raw_prefill(lib, neg) == kda.KDA_ERR_INVALID_ARG
    nan = kda.params(g_min=float("nan"))
    assert _raw_prefill(lib, nan) == kda.KDA_ERR_INVALID_ARG


def test_decode_and_conv_reject_bad_arguments_on_host(lib):
    p = kda.params()
    P = ctypes.byref(p)
    # state NULL
    assert lib.kda_decode_step(P, 16, 16, 16, 16, 16, None, 4, None, 4, None, None, 16,
                               None) == kda.KDA_ERR_INVALID_ARG
    # identity slots but fewer slots than sequences
    assert lib.kda_decode_step(P, 16, 16, 16, 16, 16, 16, 2, None, 4, None, None, 16,
                               None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_step(P, 16, 16, 16, 16, 16, 16, 4, None, 0, None, None, 16,
                               None) == kda.KDA_OK
    assert lib.kda_decode_step_fused(P, None, 16, 16, 16, 16, 16, 4, None, 4, None, None, 16,
                                     None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_conv_state_update(P, 16, 16, 16, 4, None, 4, 0, 16,
                                     None) == kda.KDA_ERR_INVALID_ARG      # zero channels
    assert lib.kda_conv_state_update(P, 16, 16, 24, 4, None, 4, 64, 16,
                                     None) == kda.KDA_ERR_INVALID_ARG      # misaligned
    assert lib.kda_prologue(P, 16, 16, None, 16, 1, 4, 0, 16, None, 16, 16, 16, None, None,
                            None) == kda.KDA_ERR_INVALID_ARG               # beta out missing


def test_workspace_query(lib):
    p = kda.params()
    assert kda.kda_prefill_workspace_size(p, 32, 500_000) == 0
    bad = kda.params(d=64)
    assert kda.kda_prefill_workspace_size(bad, 1, 10) == 0


def test_multi_decode_and_accept_reject_bad_arguments_on_host(lib):
    p = kda.params(H=2, d=128)
    buf = ctypes.c_void_p(16)  # never dereferenced: every call fails validation first
    vp = lambda: buf
    # K outside 1..64
    for K in (0, 65):
        st = lib.kda_decode_multi(ctypes.byref(p), vp(), vp(), vp(), vp(), vp(), vp(), 4, None,
                                  2, K, None, None, vp(), vp(), 1, None)
        assert st == -1
    # neither step states nor a committed final state: nothing would be kept
    st = lib.kda_decode_multi(ctypes.byref(p), vp(), vp(), vp(), vp(), vp(), vp(), 4, None, 2, 3,
                              None, None, vp(), None, 0, None)
    assert st == -1
    # misaligned step states
    st = lib.kda_decode_multi(ctypes.byref(p), vp(), vp(), vp(), vp(), vp(), vp(), 4, None, 2, 3,
                              None, None, vp(), ctypes.c_void_p(24), 1, None)
    assert st == -1
    # accept: too few slots without an index, bad K, null pointers
    assert lib.kda_state_accept(ctypes.byref(p), vp(), 5, 3, vp(), vp(), 4, None, None) == -1
    assert lib.kda_state_accept(ctypes.byref(p), vp(), 2, 0, vp(), vp(), 4, None, None) == -1
    assert lib.kda_state_accept(ctypes.byref(p), None, 2, 3, vp(), vp(), 4, None, None) == -1
    assert lib.kda_state_accept(ctypes.byref(p), vp(), 0, 3, None, None, 0, None, None) == 0
    assert lib.kda_status_string(-6).decode().startswith("KDA_ERR_BAD_INDEX")


def test_checkpoint_calls_reject_bad_arguments_on_host(lib):
    p = kda.params(H=2, d=128)
    P = ctypes.byref(p)
    buf = ctypes.c_void_p(16)  # never dereferenced: every call fails validation first

    def prefill_ck(n_ckpt=2, cu=buf, pos=buf, states=buf):
        return lib.kda_prefill_checkpointed(P, buf, buf, buf, buf, buf, None, buf, 1, 64, None,
                                            None, buf, None, cu, pos, n_ckpt, states, None, 0,
                                            None)
    assert prefill_ck(n_ckpt=0) == kda.KDA_ERR_INVALID_ARG        # at least one checkpoint
    assert prefill_ck(n_ckpt=-3) == kda.KDA_ERR_INVALID_ARG
    assert prefill_ck(cu=None) == kda.KDA_ERR_INVALID_ARG
    assert prefill_ck(pos=None) == kda.KDA_ERR_INVALID_ARG
    assert prefill_ck(states=None) == kda.KDA_ERR_INVALID_ARG
    assert prefill_ck(states=ctypes.c_void_p(24)) == kda.KDA_ERR_INVALID_ARG  # misaligned

    def conv_ck(n_seqs=1, n_ckpt=2, x=buf, out=buf):
        return lib.kda_conv_tail_checkpoints(P, x, None, buf, n_seqs, 64, buf, buf, n_ckpt, out,
                                             None)
    assert conv_ck(n_ckpt=0) == kda.KDA_OK                            # nothing to do
    assert conv_ck(n_seqs=0) == kda.KDA_ERR_INVALID_ARG
    assert conv_ck(n_ckpt=-1) == kda.KDA_ERR_INVALID_ARG
    assert conv_ck(n_ckpt=70000) == kda.KDA_ERR_INVALID_ARG           # grid limit
    assert conv_ck(x=None) == kda.KDA_ERR_INVALID_ARG
    assert conv_ck(out=ctypes.c_void_p(40)) == kda.KDA_ERR_INVALID_ARG


def test_fp8_calls_reject_bad_arguments_on_host(lib):
    p = kda.params(H=2, d=128)
    P = ctypes.byref(p)
    buf = ctypes.c_void_p(16)  # never dereferenced: every call fails validation first
    # prefill: codes without scales, misaligned scales, no codes at all
    assert lib.kda_prefill_fp8(P, buf, buf, buf, buf, buf, None, buf, 1, 64, None, None, buf,
                               None, None, None, 0, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_fp8(P, buf, buf, buf, buf, buf, None, buf, 1, 64, None, None, buf,
                               ctypes.c_void_p(20), None, None, 0, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_fp8(P, buf, buf, buf, buf, buf, None, buf, 1, 64, None, None, None,
                               buf, None, None, 0, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_fp8(P, None, None, None, None, None, None, buf, 0, 0, None, None,
                               None, None, None, None, 0, None) == kda.KDA_OK
    # decode: codes without scales
    assert lib.kda_decode_step_fused_fp8(P, buf, buf, buf, buf, buf, buf, 2, None, 2, None, None,
                                         buf, None, None) == kda.KDA_ERR_INVALID_ARG


def test_mla_calls_reject_bad_arguments_on_host(lib):
    buf = ctypes.c_void_p(16)  # never dereferenced: every call fails validation first
    assert lib.mla_decode_latent(buf, buf, 0, buf, 2, 0.07, buf, None, 0, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.mla_decode_latent(buf, buf, 64, buf, 2, 0.0, buf, None, 0, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.mla_decode_latent(buf, buf, 64, buf, -1, 0.07, buf, None, 0, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.mla_decode_latent(buf, ctypes.c_void_p(24), 64, buf, 2, 0.07, buf, None, 0,
                                 None) == kda.KDA_ERR_INVALID_ARG
    assert lib.mla_decode_latent(buf, buf, 64, buf, 2, 0.07, buf, ctypes.c_void_p(40), 1 << 20,
                                 None) == kda.KDA_ERR_INVALID_ARG          # misaligned workspace
    assert lib.mla_decode_latent(None, None, 0, None, 0, 0.07, None, None, 0, None) == kda.KDA_OK
    assert lib.mla_decode(buf, buf, buf, buf, buf, 64, buf, 2, None, 0.07, buf, buf, buf, None, 0,
                          None) == kda.KDA_ERR_INVALID_ARG
    assert kda.mla_decode_workspace_size(0, 64) == 0 and kda.mla_decode_workspace_size(4, 0) == 0


def test_wait_probe_rejects_bad_limits_on_host(lib):
    assert lib.kda_wait_probe(0, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_wait_probe(1 << 31, None) == kda.KDA_ERR_INVALID_ARG


def test_host_prefill_workspace_size(lib):
    p = kda.params()
    H, d = 64, 128
    per_row = 2 * (3 * H * d * 2 + H * d * 4 + H * 4 + H * d * 2) + 3 * H * d * 2 + H * 4
    per_seq = H * d * d * 4 + 3 * 3 * H * d * 2
    ws = kda.kda_prefill_host_workspace_size(p, 1, 512)
    assert 512 * per_row + per_seq <= ws <= 512 * per_row + per_seq + 16 * 256
    gated = kda.kda_prefill_host_workspace_size(p, 1, 512, with_gate=True)
    assert gated - ws == 2 * 512 * H * d * 2
    assert kda.kda_prefill_host_workspace_size(p, 1, 100) == 0       # not a chunk multiple
    assert kda.kda_prefill_host_workspace_size(p, 0, 512) == 0
    assert kda.kda_prefill_host_workspace_size(kda.params(d=64), 1, 512) == 0


def test_host_prefill_rejects_bad_arguments_before_any_cuda_call(lib):
    p = kda.params(H=2)
    P = ctypes.byref(p)
    ws_need = kda.kda_prefill_host_workspace_size(p, 2, 64)

    def call(pp=P, cu=(0, 64, 100), T=100, seg=64, ws=4096, wsb=None, x=16, out=16, w=16):
        arr = (ctypes.c_int32 * len(cu))(*cu)
        return lib.kda_prefill_host(pp, x, w, None, arr, len(cu) - 1, T, 16, 16, None, None,
                                    None, out, None, ws, ws_need if wsb is None else wsb,
                                    seg, None)

    assert call(cu=(1, 64, 100)) == kda.KDA_ERR_INVALID_ARG          # does not start at 0
    assert call(cu=(0, 80, 64)) == kda.KDA_ERR_INVALID_ARG           # runs backwards
    assert call(cu=(0, 64, 99)) == kda.KDA_ERR_INVALID_ARG           # does not end at T
    assert call(seg=96) == kda.KDA_ERR_INVALID_ARG                   # not a chunk multiple
    assert call(seg=0) == kda.KDA_ERR_INVALID_ARG
    assert call(x=None) == kda.KDA_ERR_INVALID_ARG
    assert call(out=None) == kda.KDA_ERR_INVALID_ARG
    assert call(w=24) == kda.KDA_ERR_INVALID_ARG                     # misaligned weights
    assert call(wsb=ws_need - 1) == kda.KDA_ERR_WORKSPACE
    assert call(ws=4096 + 16) == kda.KDA_ERR_INVALID_ARG             # workspace not 256-aligned
    assert call(pp=None) == kda.KDA_ERR_INVALID_ARG
    pb = kda.params(H=2, state_dtype=torch.bfloat16)
    assert call(pp=ctypes.byref(pb)) == kda.KDA_ERR_UNSUPPORTED      # fp32 state only


def test_mla_split_workspace_holds_the_partial_sums(lib):
    """A forced split (the tuning override) needs, per split and sequence, the 64 x 512 fp32
    partial latent sums plus each head's running maximum and normaliser."""
    with kda.mla_split(4):
        assert kda.mla_decode_workspace_size(3, 65536) == 4 * 3 * 64 * (512 + 2) * 4
    with kda.mla_split(1):
        assert kda.mla_decode_workspace_size(3, 65536) == 0               # no split, no scratch
    assert lib.mla_set_split_override(65) == kda.KDA_ERR_INVALID_ARG
    assert lib.mla_set_split_override(-1) == kda.KDA_ERR_INVALID_ARG


def test_prefill_form_is_validated(lib):
    """kda_params.prefill_form selects the tensor-core prefill's kernel form explicitly (no
    environment variable is read); values outside the enum are rejected before any launch."""
    for form in (3, -1):
        p = kda.params(H=2)
        p.prefill_form = form
        assert lib.kda_prefill(ctypes.byref(p), *([None] * 6), None, 0, 0, None, None, None,
                               None, None, 0, None) == kda.KDA_ERR_INVALID_ARG
    assert kda.params(H=2, prefill_form="pair").prefill_form == 2


def test_every_call_opens_an_nvtx_range(lib):
    """Each entry point that enqueues GPU work (every kda_status call of the headers but the
    host-side tuning switch) is traced by an NVTX range of its own name."""
    text = ""
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            text += re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
    calls = set(re.findall(r"kda_status\s+((?:kda|mla)_[a-z0-9_]+)\s*\(", text))
    calls -= {"mla_set_split_override"}
    ranges = kda.kda_trace_ranges()
    assert len(ranges) == len(set(ranges))
    assert calls <= set(ranges), sorted(calls - set(ranges))
    src = open(os.path.join(os.path.dirname(kbuild.__file__), "csrc", "kda_trace.h")).read()
    assert "nvtxRangePushA" in src and "nvtxRangePop" in src
