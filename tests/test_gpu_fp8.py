"""GPU parity: the FP8 (E4M3) output quantisation fused into the KDA epilogue.

Two checks.  (1) Parity: the dequantised output against the fp64 oracle (whose quantiser is
the fp64 definition, code = E4M3(x / scale)), within half an E4M3 step of the value (2^-4
relative in the normal range, 2^-10 of the scale below it) plus the output tolerance.
(2) Kernel self-consistency, not parity: with fp32 I/O the kernel's unquantised output is its
own fp32 value, so a model of the device's fp32 quantiser (tests/_kernel_numerics.py) run on
that output must give the same codes and scales bit for bit -- the epilogue quantises the very
values the unquantised launch writes.
The quantised launch leaves the state and conv tail updates bit-identical to the plain one.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gb300 import inputs, kda
from tests import _gpu
from tests._kernel_numerics import fp8_quantize_groups_device
from tests._parity import rms, to64
from tests.test_gpu_core import _decode_reference

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 1e-2}


def _setup(H, d, n, slots_n, K, io, gate, seed):
    C = 3 * H * d
    S0 = inputs.normal((slots_n, H, d, d), seed=seed, dtype=torch.float32, std=0.02)
    cs0 = inputs.normal((slots_n, 3, C), seed=seed + 1, dtype=io)
    w = inputs.normal((C, 4), seed=seed + 2, std=0.5, dtype=io)
    steps = [inputs.decode_inputs(n, H, d, seed=seed + 10 + t, io_dtype=io, gate=gate)
             for t in range(K)]
    norm_w = inputs.normal((d,), seed=seed + 3, dtype=torch.float32) if gate else None
    return S0, cs0, w, steps, norm_w


def _run(p, S0, cs0, w, steps, norm_w, slots, gate, fp8):
    n, H, d = steps[0]["g"].shape
    state, cs = S0.cuda().clone(), cs0.cuda().clone()
    slot_t = torch.tensor(slots, dtype=torch.int32, device="cuda")
    outs = []
    for st in steps:
        common = dict(slot_idx=slot_t, gate_logit=st["gate"].cuda() if gate else None,
                      norm_w=norm_w.cuda() if gate else None)
        if fp8:
            q = torch.empty((n, H, d), dtype=torch.uint8, device="cuda")
            sc = torch.empty((n, H), dtype=torch.float32, device="cuda")
            kda.kda_decode_step_fused_fp8(p, st["x"].cuda(), w.cuda(), cs, st["g"].cuda(),
                                          st["beta"].cuda(), state, q, sc, **common)
            outs.append((q, sc))
        else:
            out = torch.empty((n, H, d), dtype=p.io_torch, device="cuda")
            kda.kda_decode_step_fused(p, st["x"].cuda(), w.cuda(), cs, st["g"].cuda(),
                                      st["beta"].cuda(), state, out, **common)
            outs.append(out)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    return outs, state, cs


@pytest.mark.parametrize("gate", [False, True])
@pytest.mark.parametrize("d", [128, 16])
def test_fp8_codes_are_the_quantisation_of_the_fp32_output(gate, d):
    """Kernel self-consistency: the decode's codes and scales are the device quantiser's
    (fp32 model) of the same launch's unquantised fp32 output, bit for bit."""
    H, n, slots_n, K = 3, 5, 7, 3
    slots = [6, 0, 3, 2, 5]
    io = torch.float32
    p = kda.params(H=H, d=d, io_dtype=io)
    _gpu.lib()
    S0, cs0, w, steps, norm_w = _setup(H, d, n, slots_n, K, io, gate, seed=700)
    plain, st_a, cs_a = _run(p, S0, cs0, w, steps, norm_w, slots, gate, fp8=False)
    quant, st_b, cs_b = _run(p, S0, cs0, w, steps, norm_w, slots, gate, fp8=True)
    # the state and conv-tail updates do not depend on the output format
    assert torch.equal(st_a, st_b) and torch.equal(cs_a, cs_b)
    for o32, (q, sc) in zip(plain, quant):
        want_q, want_sc = fp8_quantize_groups_device(o32.cpu().numpy(), d)
        assert np.array_equal(sc.cpu().numpy(), want_sc[..., 0])
        assert np.array_equal(q.cpu().numpy(), want_q)


@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("gate", [False, True])
def test_fp8_decode_matches_the_oracle(io, gate):
    H, d, n, slots_n, K = 4, 128, 6, 9, 4
    slots = [8, 2, 0, 5, 3, 7]
    p = kda.params(H=H, d=d, io_dtype=io)
    _gpu.lib()
    S0, cs0, w, steps, norm_w = _setup(H, d, n, slots_n, K, io, gate, seed=720)
    quant, state, cs = _run(p, S0, cs0, w, steps, norm_w, slots, gate, fp8=True)
    x_steps = torch.stack([st["x"] for st in steps])
    g_steps = torch.stack([st["g"] for st in steps])
    b_steps = torch.stack([st["beta"] for st in steps])
    gate_steps = torch.stack([st["gate"] for st in steps]) if gate else None
    ref_out, ref_fin, _ = _decode_reference(x_steps, w, cs0, S0, g_steps, b_steps, H, d, slots,
                                            gate_steps, norm_w)
    for t, (q, sc) in enumerate(quant):
        ref = ref_out[t]                                     # [n, H, d] fp64
        sc64 = to64(sc)
        deq = oracle.fp8_dequantize_groups(q.cpu().numpy(), sc64[..., None], d)
        # the scale is the group's amax / 448 up to the output error
        np.testing.assert_allclose(sc64, np.abs(ref).max(-1) / 448.0,
                                   rtol=0, atol=TOL[io] * rms(ref) / 448.0 * 4)
        # half a step of the binade the value or its code lies in (a value just below a
        # binade edge may round up into the next, coarser one)
        y = np.maximum(np.abs(ref), np.abs(deq)) / sc64[..., None]
        half = np.where(y >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 4),
                        2.0 ** -10) * sc64[..., None]
        excess = np.maximum(np.abs(deq - ref) - half * (1 + 2 ** -6), 0.0)
        assert excess.max() <= TOL[io] * rms(ref), f"step {t}: {excess.max() / rms(ref):.3g}"
    st_cpu = state.cpu()
    for s in slots:
        np.testing.assert_allclose(to64(st_cpu[s]), ref_fin[s], rtol=0,
                                   atol=1e-3 * rms(ref_fin[s]))


def test_fp8_decode_rejects_missing_scales():
    H, d, n = 2, 128, 2
    p = kda.params(H=H, d=d)
    _gpu.lib()
    C = 3 * H * d
    x = torch.zeros((n, C), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((C, 4), dtype=torch.bfloat16, device="cuda")
    cs = torch.zeros((n, 3, C), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((n, H, d), device="cuda")
    b = torch.zeros((n, H), device="cuda")
    state = torch.zeros((n, H, d, d), device="cuda")
    q = torch.empty((n, H, d), dtype=torch.uint8, device="cuda")
    lib = kda.load()
    st = lib.kda_decode_step_fused_fp8(
        ctypes.byref(p), x.data_ptr(), w.data_ptr(), cs.data_ptr(), g.data_ptr(),
        b.data_ptr(), state.data_ptr(), n, None, n, None, None, q.data_ptr(), None, None)
    assert st == kda.KDA_ERR_INVALID_ARG


# ---------------------------------------------------------------------------------------
# Prefill
# ---------------------------------------------------------------------------------------

def _prefill_fp8(inp, p, gate):
    c = _gpu.cuda
    T, H, d = inp["q"].shape
    N = inp["cu_seqlens"].numel() - 1
    q8 = torch.zeros((T, H, d), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    fin = torch.empty((N, H, d, d), dtype=p.state_torch, device="cuda")
    kda.kda_prefill_fp8(p, c(inp["q"]), c(inp["k"]), c(inp["v"]), c(inp["g"]), c(inp["beta"]),
                        c(inp["cu_seqlens"]), q8, sc, init_state=c(inp.get("init_state")),
                        final_state=fin, gate_logit=c(inp["gate"]) if gate else None,
                        norm_w=c(inp.get("norm_w")) if gate else None)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    return q8, sc, fin


def _check_against_oracle(q8, sc, inp, p, gate, tol):
    ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                             inp["cu_seqlens"], init_state=inp.get("init_state"),
                             gate=inp.get("gate") if gate else None,
                             norm_w=inp.get("norm_w") if gate else None)["out"]
    d = ref.shape[-1]
    sc64 = to64(sc)
    deq = oracle.fp8_dequantize_groups(q8.cpu().numpy(), sc64[..., None], d)
    y = np.maximum(np.abs(ref), np.abs(deq)) / sc64[..., None]
    half = np.where(y >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 4),
                    2.0 ** -10) * sc64[..., None]
    excess = np.maximum(np.abs(deq - ref) - half * (1 + 2 ** -6), 0.0)
    assert excess.max() <= tol * rms(ref), f"{excess.max() / rms(ref):.3g}"
    np.testing.assert_allclose(sc64, np.abs(ref).max(-1) / 448.0, rtol=0,
                               atol=4 * tol * rms(ref) / 448.0)
    return ref


@pytest.mark.parametrize("path", ["fused", "pair"])
@pytest.mark.parametrize("gate", [False, True])
def test_fp8_prefill_chunked_matches_the_oracle(path, gate):
    """The chunked tensor-core kernel's FP8 epilogue over ragged sequences (full 64-token
    tiles go out by bulk store, ragged tails element by element), both kernel forms."""
    lens = [0, 1, 63, 64, 65, 130, 256]
    inp = inputs.kda_inputs(lens, 2, 128, seed=740, init_state="even", gate=True)
    inp["norm_w"] = inputs.normal((128,), seed=741, dtype=torch.float32)
    p = kda.params(H=2, d=128, prefill_form=path)
    _gpu.lib()
    q8, sc, fin = _prefill_fp8(inp, p, gate)
    _check_against_oracle(q8, sc, inp, p, gate, TOL[torch.bfloat16])
    # the same kernel's bf16 output: the codes dequantise to it within half a step and
    # half a bf16 ulp (both come from the same fp32 value), and the final states are identical
    out, fin0 = _gpu.prefill(inp, p, gate=gate)
    torch.cuda.synchronize()
    assert torch.equal(fin, fin0)
    o = to64(out)
    sc64 = to64(sc)
    deq = oracle.fp8_dequantize_groups(q8.cpu().numpy(), sc64[..., None], 128)
    y = np.maximum(np.abs(o), np.abs(deq)) / sc64[..., None]
    half = np.where(y >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 4),
                    2.0 ** -10) * sc64[..., None]
    ulp = 0.5 * np.exp2(np.floor(np.log2(np.maximum(np.abs(o), 1e-30))) - 7)
    assert (np.abs(deq - o) <= half * (1 + 2 ** -6) + ulp).all()


@pytest.mark.parametrize("gate", [False, True])
def test_fp8_prefill_codes_are_the_quantisation_of_the_fp32_output(gate):
    """Kernel self-consistency: fp32 I/O runs the token-serial kernel, and its fp32 output
    quantised by the device quantiser's fp32 model gives the kernel's codes and scales bit
    for bit; the parity check against the fp64 oracle follows."""
    lens = [5, 0, 70, 33]
    inp = inputs.kda_inputs(lens, 3, 128, seed=750, io_dtype=torch.float32, init_state="all",
                            gate=True)
    inp["norm_w"] = inputs.normal((128,), seed=751, dtype=torch.float32)
    p = kda.params(H=3, d=128, io_dtype=torch.float32)
    _gpu.lib()
    q8, sc, fin = _prefill_fp8(inp, p, gate)
    out, fin0 = _gpu.prefill(inp, p, gate=gate)
    torch.cuda.synchronize()
    assert torch.equal(fin, fin0)
    want_q, want_sc = fp8_quantize_groups_device(out.cpu().numpy(), 128)
    assert np.array_equal(sc.cpu().numpy(), want_sc[..., 0])
    assert np.array_equal(q8.cpu().numpy(), want_q)
    _check_against_oracle(q8, sc, inp, p, gate, TOL[torch.float32])
