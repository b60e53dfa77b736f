"""GPU parity: prologue, conv update, decode and prefill against the fp64 oracle.

Tolerances (stated by the workload definition): fp32 I/O -> max |err| <= 1e-4 of the output
RMS; bf16 I/O -> max |err| <= 1e-2 of the output RMS beyond half a bf16 ulp of the stored value
(the storage rounding any bf16 output must incur), final fp32 state max |err| <= 1e-3 of the
state RMS; conv tails and index bookkeeping bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gb300 import inputs, kda
from tests import _gpu
from tests._parity import excess_over_half_ulp, max_err_rel_rms, out_error, to64

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 1e-2
TOL_STATE = 1e-3


def _oracle_prefill(inp, gate=False, **kw):
    return oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              inp["cu_seqlens"], init_state=inp.get("init_state"),
                              gate=inp.get("gate") if gate else None,
                              norm_w=inp.get("norm_w") if gate else None, **kw)


def _check_prefill(inp, p, gate=False, tol_out=None, tol_state=None):
    out, fin = _gpu.prefill(inp, p, gate=gate)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    ref = _oracle_prefill(inp, gate=gate, scale=p.scale)
    tol_out = tol_out or (TOL_BF16 if p.io_torch == torch.bfloat16 else TOL_F32)
    tol_state = tol_state or (TOL_STATE if p.io_torch == torch.bfloat16 else TOL_F32)
    e_out = out_error(out, ref["out"], p.io_torch)
    if p.state_torch == torch.bfloat16:
        e_st = excess_over_half_ulp(fin, ref["final_state"])
    else:
        e_st = max_err_rel_rms(fin, ref["final_state"])
    assert e_out <= tol_out, f"output error {e_out:.3g} > {tol_out}"
    assert e_st <= tol_state, f"final-state error {e_st:.3g} > {tol_state}"
    return out, fin, e_out, e_st


def test_tiny_fp32_config():
    """B=1, T=64, H=2, d=16, fp32 I/O and state, zero initial state."""
    inp = inputs.kda_inputs([64], 2, 16, seed=0, io_dtype=torch.float32)
    p = kda.params(H=2, d=16, io_dtype=torch.float32)
    _check_prefill(inp, p)


@pytest.mark.parametrize("d,io", [(16, torch.float32), (128, torch.float32),
                                  (128, torch.bfloat16), (16, torch.bfloat16)])
def test_prefill_varlen_edges(d, io):
    """Empty, 1-, 2-token, chunk-1, chunk, chunk+1 and multi-chunk sequences, packed, with
    even-indexed sequences continuing from a nonzero state and the output norm/gate."""
    lens = [0, 1, 2, 63, 64, 65, 130]
    inp = inputs.kda_inputs(lens, 3, d, seed=1, io_dtype=io, init_state="even", gate=True)
    inp["norm_w"] = inputs.normal((d,), seed=2, dtype=torch.float32)
    p = kda.params(H=3, d=d, io_dtype=io)
    _check_prefill(inp, p, gate=True)


def test_prefill_plain_read_and_scale():
    inp = inputs.kda_inputs([100, 37], 2, 128, seed=3, init_state="all")
    p = kda.params(H=2, d=128, scale=128 ** -0.5)
    _check_prefill(inp, p)


def test_prefill_bf16_state_storage():
    inp = inputs.kda_inputs([70, 129], 2, 128, seed=4, init_state="all",
                            state_dtype=torch.bfloat16)
    p = kda.params(H=2, d=128, state_dtype=torch.bfloat16)
    _check_prefill(inp, p)


def test_prefill_packed_equals_separate_bitwise():
    lens = [5, 64, 77, 1]
    inp = inputs.kda_inputs(lens, 2, 128, seed=5, init_state="even")
    p = kda.params(H=2, d=128)
    out, fin = _gpu.prefill(inp, p)
    cu = inp["cu_seqlens"].tolist()
    for n, L in enumerate(lens):
        sl = slice(cu[n], cu[n + 1])
        one = {key: inp[key][sl] for key in ("q", "k", "v", "g", "beta")}
        one["cu_seqlens"] = torch.tensor([0, L], dtype=torch.int32)
        one["init_state"] = inp["init_state"][n:n + 1]
        o1, f1 = _gpu.prefill(one, p)
        assert torch.equal(out[sl], o1)
        assert torch.equal(fin[n], f1[0])


def test_prefill_split_resume():
    """prefill(T1+T2) vs prefill(T2) resumed from prefill(T1)'s final state."""
    inp = inputs.kda_inputs([200], 2, 128, seed=6, init_state="all")
    p = kda.params(H=2, d=128)
    out, fin = _gpu.prefill(inp, p)
    T1 = 77
    a = {key: inp[key][:T1] for key in ("q", "k", "v", "g", "beta")}
    a["cu_seqlens"] = torch.tensor([0, T1], dtype=torch.int32)
    a["init_state"] = inp["init_state"]
    _, fa = _gpu.prefill(a, p)
    b = {key: inp[key][T1:] for key in ("q", "k", "v", "g", "beta")}
    b["cu_seqlens"] = torch.tensor([0, 200 - T1], dtype=torch.int32)
    b["init_state"] = fa.cpu()
    ob, fb = _gpu.prefill(b, p)
    ref = _oracle_prefill(inp)
    assert out_error(ob, ref["out"][T1:], torch.bfloat16) <= TOL_BF16
    assert max_err_rel_rms(fb, ref["final_state"]) <= TOL_STATE


def test_prefill_final_state_may_alias_init():
    inp = inputs.kda_inputs([90, 3], 2, 128, seed=7, init_state="all")
    p = kda.params(H=2, d=128)
    ref_out, ref_fin = _gpu.prefill(inp, p)
    st = _gpu.cuda(inp["init_state"]).clone()
    out = torch.empty_like(ref_out)
    kda.kda_prefill(p, *(_gpu.cuda(inp[x]) for x in ("q", "k", "v", "g", "beta")),
                    _gpu.cuda(inp["cu_seqlens"]), out, init_state=st, final_state=st)
    assert torch.equal(out, ref_out)
    assert torch.equal(st, ref_fin)


# ---------------------------------------------------------------------------------------
# Prologue
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("d,io", [(128, torch.bfloat16), (16, torch.float32)])
@pytest.mark.parametrize("l2", [False, True])
def test_prologue(d, io, l2):
    lens = [0, 1, 2, 3, 17, 40]
    H = 2
    pin = inputs.prologue_inputs(lens, H, d, seed=10, io_dtype=io)
    p = kda.params(H=H, d=d, io_dtype=io)
    _gpu.lib()
    T = sum(lens)
    q = torch.empty((T, H, d), dtype=io, device="cuda")
    k, v = torch.empty_like(q), torch.empty_like(q)
    beta = torch.empty((T, H), dtype=torch.float32, device="cuda")
    g = torch.empty((T, H, d), dtype=torch.float32, device="cuda")
    cs = _gpu.cuda(pin["conv_state"]).clone()
    kda.kda_prologue(p, _gpu.cuda(pin["x"]), _gpu.cuda(pin["conv_w"]), cs,
                     _gpu.cuda(pin["cu_seqlens"]), q, k, v, l2norm_qk=l2,
                     beta_logit=_gpu.cuda(pin["beta_logit"]), g_raw=_gpu.cuda(pin["g_raw"]),
                     beta=beta, g=g)
    torch.cuda.synchronize()
    ref = oracle.prologue(pin["x"], pin["conv_w"], pin["cu_seqlens"], H, d,
                          conv_state=pin["conv_state"], l2norm_qk=l2,
                          beta_logit=pin["beta_logit"], g_raw=pin["g_raw"])
    y = ref["y"].reshape(T, 3, H, d)
    tol = TOL_BF16 if io == torch.bfloat16 else TOL_F32
    for s, t in enumerate((q, k, v)):
        assert out_error(t, y[:, s], io) <= tol
    assert max_err_rel_rms(beta, ref["beta"]) <= 1e-6
    assert np.array_equal(to64(g), ref["g"])
    # the new conv tails are bit-exact copies
    want = torch.from_numpy(ref["conv_state"].view(np.int16 if io == torch.bfloat16 else np.int32))
    got = cs.cpu().view(torch.int16 if io == torch.bfloat16 else torch.int32)
    assert torch.equal(got, want)


# ---------------------------------------------------------------------------------------
# Decode
# ---------------------------------------------------------------------------------------

def test_conv_state_update_bit_exact_tail():
    H, d, n, slots = 2, 128, 5, 8
    C = 3 * H * d
    p = kda.params(H=H, d=d)
    _gpu.lib()
    cs0 = inputs.normal((slots, 3, C), seed=20)
    w = inputs.normal((C, 4), seed=21, std=0.5)
    x = inputs.normal((n, C), seed=22)
    slot = torch.tensor([6, 0, 3, 7, 1], dtype=torch.int32)
    cs = cs0.cuda()
    y = torch.empty((n, C), dtype=torch.bfloat16, device="cuda")
    kda.kda_conv_state_update(p, x.cuda(), w.cuda(), cs, y, slot_idx=slot.cuda())
    torch.cuda.synchronize()
    want = cs0.clone()
    for i, s in enumerate(slot.tolist()):
        want[s] = torch.stack([cs0[s, 1], cs0[s, 2], x[i]])
    assert torch.equal(cs.cpu().view(torch.int16), want.view(torch.int16))
    # y against the oracle's convolution of (old tail, new token)
    for i, s in enumerate(slot.tolist()):
        r = oracle.prologue(x[i:i + 1], w, torch.tensor([0, 1], dtype=torch.int32), H, d,
                            conv_state=cs0[s:s + 1])
        assert out_error(y[i], r["y"][0], torch.bfloat16) <= TOL_BF16


def _decode_reference(x_steps, w, cs0, S0, g_steps, b_steps, H, d, slots, gate_steps=None,
                      norm_w=None):
    """Oracle for n sequences x K decode steps: per sequence, the prologue over its K raw
    tokens from its conv tail, then the recurrence over those K tokens from its state."""
    K, n, C = x_steps.shape
    outs = np.zeros((K, n, H, d))
    finals, tails = {}, {}
    for i, s in enumerate(slots):
        pr = oracle.prologue(x_steps[:, i], w, torch.tensor([0, K], dtype=torch.int32), H, d,
                             conv_state=cs0[s:s + 1])
        y = pr["y"].reshape(K, 3, H, d)
        r = oracle.kda_forward(y[:, 0].copy(), y[:, 1].copy(), y[:, 2].copy(),
                               g_steps[:, i].contiguous(), b_steps[:, i].contiguous(),
                               torch.tensor([0, K], dtype=torch.int32),
                               init_state=S0[s:s + 1],
                               gate=None if gate_steps is None else gate_steps[:, i].contiguous(),
                               norm_w=norm_w)
        outs[:, i] = r["out"]
        finals[s] = r["final_state"][0]
        tails[s] = pr["conv_state"][0]
    return outs, finals, tails


@pytest.mark.parametrize("gate", [False, True])
def test_fused_decode_steps(gate):
    H, d, n, slots_n, K = 4, 128, 6, 9, 10
    C = 3 * H * d
    p = kda.params(H=H, d=d)
    _gpu.lib()
    slots = [8, 2, 0, 5, 3, 7]
    S0 = inputs.normal((slots_n, H, d, d), seed=30, dtype=torch.float32, std=0.02)
    cs0 = inputs.normal((slots_n, 3, C), seed=31)
    w = inputs.normal((C, 4), seed=32, std=0.5)
    steps = [inputs.decode_inputs(n, H, d, seed=100 + t, gate=gate) for t in range(K)]
    state, cs = S0.cuda(), cs0.cuda()
    slot_t = torch.tensor(slots, dtype=torch.int32, device="cuda")
    norm_w = inputs.normal((d,), seed=33, dtype=torch.float32) if gate else None
    outs = []
    for st in steps:
        out = torch.empty((n, H, d), dtype=torch.bfloat16, device="cuda")
        kda.kda_decode_step_fused(p, st["x"].cuda(), w.cuda(), cs, st["g"].cuda(),
                                  st["beta"].cuda(), state, out, slot_idx=slot_t,
                                  gate_logit=st["gate"].cuda() if gate else None,
                                  norm_w=norm_w.cuda() if gate else None)
        outs.append(out)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    x_steps = torch.stack([st["x"] for st in steps])
    g_steps = torch.stack([st["g"] for st in steps])
    b_steps = torch.stack([st["beta"] for st in steps])
    gate_steps = torch.stack([st["gate"] for st in steps]) if gate else None
    ref_out, ref_fin, ref_tail = _decode_reference(x_steps, w, cs0, S0, g_steps, b_steps, H, d,
                                                   slots, gate_steps, norm_w)
    got = torch.stack(outs).cpu()
    assert out_error(got, ref_out, torch.bfloat16) <= TOL_BF16
    st_cpu = state.cpu()
    for s in slots:
        assert max_err_rel_rms(st_cpu[s], ref_fin[s]) <= TOL_STATE
        assert np.array_equal(cs.cpu()[s].view(torch.int16).numpy(),
                              ref_tail[s].view(np.int16))
    untouched = [s for s in range(slots_n) if s not in slots]
    for s in untouched:
        assert torch.equal(st_cpu[s], S0[s]) and torch.equal(cs.cpu()[s], cs0[s])


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_decode_step_post_conv_inputs(state_dtype):
    """kda_decode_step on post-convolution q, k, v drawn directly (N(0,1) bf16)."""
    H, d, n = 3, 128, 7
    p = kda.params(H=H, d=d, state_dtype=state_dtype)
    _gpu.lib()
    inp = inputs.kda_inputs([1] * n, H, d, seed=40, init_state="all", state_dtype=state_dtype)
    state = inp["init_state"].cuda()
    out = torch.empty((n, H, d), dtype=torch.bfloat16, device="cuda")
    kda.kda_decode_step(p, *(inp[x].cuda() for x in ("q", "k", "v", "g", "beta")), state, out)
    torch.cuda.synchronize()
    ref = _oracle_prefill(inp)
    assert out_error(out, ref["out"], torch.bfloat16) <= TOL_BF16
    if state_dtype == torch.bfloat16:
        assert excess_over_half_ulp(state, ref["final_state"]) <= TOL_STATE
    else:
        assert max_err_rel_rms(state, ref["final_state"]) <= TOL_STATE


def test_decode_matches_prefill_over_same_tokens():
    """K decode steps of one sequence == prefill over the same K tokens (within tolerance)."""
    H, d, K = 2, 128, 40
    p = kda.params(H=H, d=d)
    inp = inputs.kda_inputs([K], H, d, seed=41, init_state="all")
    out_pf, fin_pf = _gpu.prefill(inp, p)
    state = inp["init_state"].cuda()
    outs = []
    for t in range(K):
        o = torch.empty((1, H, d), dtype=torch.bfloat16, device="cuda")
        kda.kda_decode_step(p, *(inp[x][t:t + 1].cuda() for x in ("q", "k", "v", "g", "beta")),
                            state, o)
        outs.append(o)
    ref = _oracle_prefill(inp)
    assert out_error(torch.cat(outs), ref["out"], torch.bfloat16) <= TOL_BF16
    assert max_err_rel_rms(state, ref["final_state"]) <= TOL_STATE
    assert max_err_rel_rms(fin_pf, ref["final_state"]) <= TOL_STATE


def test_bounded_wait_that_runs_out_is_reported_and_the_context_survives():
    """Failure detection without a GPU fault: a bounded mbarrier wait on a barrier nothing
    arrives at gives up, raises the sticky flag (KDA_ERR_TIMEOUT) and returns; the flag is
    cleared by the read and the next launches run normally."""
    _gpu.lib()
    kda.kda_wait_probe(20000)
    torch.cuda.synchronize()
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_check_device_error()
    assert ei.value.status == kda.KDA_ERR_TIMEOUT
    kda.kda_check_device_error()  # cleared
    inp = inputs.kda_inputs([70], 2, 128, seed=90)
    p = kda.params(H=2, d=128)
    _check_prefill(inp, p)
    kda.kda_check_device_error()
