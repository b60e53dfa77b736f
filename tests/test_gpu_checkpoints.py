"""GPU parity: prefix-state checkpoints (the state, and the conv tail, saved at token
boundaries inside the sequences of a prefill) against the oracle run on each prefix.

A checkpoint after `pos` tokens of sequence n must equal the final state of a prefill of
that prefix alone (same initial state): the tolerance is the final-state one.  Conv-tail
checkpoints are raw copies and must be bit-exact.  Saving checkpoints must leave the
outputs and final states of the launch bit-identical to a launch without them.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gb300 import inputs, kda
from tests import _gpu
from tests._parity import max_err_rel_rms

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_STATE = 1e-3


def _ckpt_tables(cps):
    """cps: per sequence, its checkpoint positions -> (ckpt_cu, ckpt_pos, list of (n, pos))."""
    cu = [0]
    pos, flat = [], []
    for n, ps in enumerate(cps):
        pos += ps
        flat += [(n, p) for p in ps]
        cu.append(len(pos))
    return (torch.tensor(cu, dtype=torch.int32), torch.tensor(pos, dtype=torch.int32), flat)


def _prefix_state(inp, n, pos, gate):
    """Oracle final state after the first `pos` tokens of sequence n, from its own start."""
    bos = int(inp["cu_seqlens"][n])
    sl = slice(bos, bos + pos)
    init = inp.get("init_state")
    r = oracle.kda_forward(inp["q"][sl], inp["k"][sl], inp["v"][sl], inp["g"][sl],
                           inp["beta"][sl], torch.tensor([0, pos], dtype=torch.int32),
                           init_state=None if init is None else init[n:n + 1],
                           gate=inp["gate"][sl] if gate else None,
                           norm_w=inp.get("norm_w") if gate else None)
    return r["final_state"][0]


def _run(inp, p, ck_cu, ck_pos, gate):
    _gpu.lib()
    c = _gpu.cuda
    T, H, d = inp["q"].shape
    N = inp["cu_seqlens"].numel() - 1
    out = torch.empty((T, H, d), dtype=p.io_torch, device="cuda")
    fin = torch.empty((N, H, d, d), dtype=p.state_torch, device="cuda")
    ck = torch.full((ck_pos.numel(), H, d, d), float("nan"), dtype=p.state_torch,
                    device="cuda")
    kda.kda_prefill_checkpointed(
        p, c(inp["q"]), c(inp["k"]), c(inp["v"]), c(inp["g"]), c(inp["beta"]),
        c(inp["cu_seqlens"]), out, c(ck_cu), c(ck_pos), ck,
        init_state=c(inp.get("init_state")), final_state=fin,
        gate_logit=c(inp["gate"]) if gate else None,
        norm_w=c(inp.get("norm_w")) if gate else None)
    return out, fin, ck


@pytest.mark.parametrize("path", ["fused", "pair", "token_serial"])
def test_prefill_checkpoints_equal_prefix_final_states(path):
    """Chunk-edge and sequence-end checkpoints over ragged sequences (an empty one, a
    one-token one, exact chunk multiples, ragged tails), some with a nonzero initial state,
    through the chunked kernel in both of its forms and through the token-serial kernel."""
    if path == "token_serial":
        d, io = 16, torch.float32
    else:
        d, io = 128, torch.bfloat16
    lens = [200, 0, 64, 130, 1, 256]
    cps = [[64, 128, 192, 200], [], [64], [64, 130], [1], [128, 256]]
    inp = inputs.kda_inputs(lens, 2, d, seed=40, io_dtype=io, init_state="even", gate=True)
    inp["norm_w"] = inputs.normal((d,), seed=41, dtype=torch.float32)
    p = kda.params(H=2, d=d, io_dtype=io,
                   prefill_form="auto" if path == "token_serial" else path)
    ck_cu, ck_pos, flat = _ckpt_tables(cps)

    out, fin, ck = _run(inp, p, ck_cu, ck_pos, gate=True)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    # checkpoints do not change what the launch computes
    out0, fin0 = _gpu.prefill(inp, p, gate=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out0) and torch.equal(fin, fin0)

    tol = TOL_F32 if io == torch.float32 else TOL_STATE
    for j, (n, pos) in enumerate(flat):
        ref = _prefix_state(inp, n, pos, gate=True)
        e = max_err_rel_rms(ck[j], ref)
        assert e <= tol, f"checkpoint {j} (sequence {n}, {pos} tokens): {e:.3g} > {tol}"
        if pos == lens[n]:  # the checkpoint at the sequence end is its final state
            assert torch.equal(ck[j], fin[n])


def test_token_serial_checkpoints_at_any_position():
    """fp32 I/O runs the token-serial kernel, which saves a checkpoint after any token."""
    lens = [70, 5, 131]
    cps = [[1, 3, 37, 69, 70], [2], [1, 64, 100, 130]]
    inp = inputs.kda_inputs(lens, 3, 128, seed=42, io_dtype=torch.float32, init_state="all")
    p = kda.params(H=3, d=128, io_dtype=torch.float32)
    ck_cu, ck_pos, flat = _ckpt_tables(cps)
    out, fin, ck = _run(inp, p, ck_cu, ck_pos, gate=False)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    for j, (n, pos) in enumerate(flat):
        e = max_err_rel_rms(ck[j], _prefix_state(inp, n, pos, gate=False))
        assert e <= TOL_F32, f"checkpoint {j} (sequence {n}, {pos} tokens): {e:.3g}"


@pytest.mark.parametrize("form", ["fused", "pair"])
def test_checkpoint_rule_breaks_are_flagged_not_followed(form):
    """Positions off a chunk edge (chunked kernel), 0, past the sequence end, out of order,
    and a checkpoint range past n_ckpt: skipped, reported as KDA_ERR_BAD_INDEX, and the
    outputs, final states and the valid checkpoints are unaffected."""
    lens = [130, 64, 100]
    inp = inputs.kda_inputs(lens, 2, 128, seed=43, init_state="all")
    p = kda.params(H=2, d=128, prefill_form=form)
    out0, fin0 = _gpu.prefill(inp, p)
    torch.cuda.synchronize()
    ref64 = _prefix_state(inp, 0, 64, gate=False)

    cases = {
        "off_edge": ([[64, 65]], [0, 2, 2, 2]),
        "zero": ([[0, 64]], [0, 2, 2, 2]),
        "past_end": ([[64, 131]], [0, 2, 2, 2]),
        "out_of_order": ([[128, 64]], [0, 2, 2, 2]),
        "range_past_count": ([[64]], [0, 1, 1, 5]),
    }
    for name, (cps, cu) in cases.items():
        ck_pos = torch.tensor(cps[0], dtype=torch.int32)
        ck_cu = torch.tensor(cu, dtype=torch.int32)
        out, fin, ck = _run(inp, p, ck_cu, ck_pos, gate=False)
        torch.cuda.synchronize()
        with pytest.raises(kda.KdaError) as ei:
            kda.kda_check_device_error()
        assert ei.value.status == kda.KDA_ERR_BAD_INDEX, name
        assert torch.equal(out, out0) and torch.equal(fin, fin0), name
        if cps[0][0] == 64:  # the valid first checkpoint is still saved
            assert max_err_rel_rms(ck[0], ref64) <= TOL_STATE, name
    kda.kda_check_device_error()  # the flag was cleared by the last read


@pytest.mark.parametrize("d,io", [(128, torch.bfloat16), (16, torch.float32)])
def test_offsets_outside_the_rows_are_flagged_and_empty(d, io):
    """A sequence whose offsets leave [0, total_tokens] is treated as empty (its final state
    is its initial state) and reported as KDA_ERR_BAD_SEQLENS; the other sequences are
    computed as usual."""
    lens = [64, 64]
    inp = inputs.kda_inputs(lens, 2, d, seed=44, io_dtype=io, init_state="all")
    p = kda.params(H=2, d=d, io_dtype=io)
    good = {key: val for key, val in inp.items()}
    good["cu_seqlens"] = torch.tensor([0, 64], dtype=torch.int32)
    good["init_state"] = inp["init_state"][:1]
    out_g, fin_g = _gpu.prefill(good, p)
    bad = dict(inp)
    bad["cu_seqlens"] = torch.tensor([0, 64, 100000], dtype=torch.int32)
    out_b, fin_b = _gpu.prefill(bad, p)
    torch.cuda.synchronize()
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_check_device_error()
    assert ei.value.status == kda.KDA_ERR_BAD_SEQLENS
    assert torch.equal(out_b[:64], out_g[:64]) and torch.equal(fin_b[0], fin_g[0])
    assert torch.equal(fin_b[1].cpu(), inp["init_state"][1].to(p.state_torch))


@pytest.mark.parametrize("d,io", [(128, torch.bfloat16), (16, torch.float32)])
def test_conv_tail_checkpoints_bit_exact(d, io):
    """The conv tail at a checkpoint equals the tail a prologue over that prefix leaves:
    positions 1 and 2 reach into the sequence's prior tail, later ones are raw inputs."""
    H = 2
    lens = [5, 0, 2, 70]
    cps = [[1, 2, 3, 5], [], [1, 2], [3, 64, 70]]
    pin = inputs.prologue_inputs(lens, H, d, seed=45, io_dtype=io)
    C = 3 * H * d
    p = kda.params(H=H, d=d, io_dtype=io)
    ck_cu, ck_pos, flat = _ckpt_tables(cps)
    _gpu.lib()
    c = _gpu.cuda
    got = torch.zeros((len(flat), 3, C), dtype=io, device="cuda")
    kda.kda_conv_tail_checkpoints(p, c(pin["x"]), c(pin["conv_state"]), c(pin["cu_seqlens"]),
                                  c(ck_cu), c(ck_pos), got)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    ibits = torch.int16 if io == torch.bfloat16 else torch.int32
    nbits = np.int16 if io == torch.bfloat16 else np.int32
    for j, (n, pos) in enumerate(flat):
        bos = int(pin["cu_seqlens"][n])
        r = oracle.prologue(pin["x"][bos:bos + pos], pin["conv_w"],
                            torch.tensor([0, pos], dtype=torch.int32), H, d,
                            conv_state=pin["conv_state"][n:n + 1])
        want = torch.from_numpy(r["conv_state"][0].view(nbits))
        assert torch.equal(got[j].cpu().view(ibits), want), f"checkpoint {j}"

    # without a prior tail the taps before the sequence start are zeros
    got0 = torch.full_like(got, 7.0)
    kda.kda_conv_tail_checkpoints(p, c(pin["x"]), None, c(pin["cu_seqlens"]), c(ck_cu),
                                  c(ck_pos), got0)
    torch.cuda.synchronize()
    r = oracle.prologue(pin["x"][:1], pin["conv_w"], torch.tensor([0, 1], dtype=torch.int32),
                        H, d)
    assert torch.equal(got0[0].cpu().view(ibits), torch.from_numpy(r["conv_state"][0].view(nbits)))

    # a position past its sequence is reported and its row left untouched
    bad_pos = torch.tensor([1, 6], dtype=torch.int32)
    bad_cu = torch.tensor([0, 2, 2, 2, 2], dtype=torch.int32)
    got1 = torch.zeros((2, 3, C), dtype=io, device="cuda")
    kda.kda_conv_tail_checkpoints(p, c(pin["x"]), c(pin["conv_state"]), c(pin["cu_seqlens"]),
                                  c(bad_cu), c(bad_pos), got1)
    torch.cuda.synchronize()
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_check_device_error()
    assert ei.value.status == kda.KDA_ERR_BAD_INDEX
    assert torch.equal(got1[0], got[0]) and not bool(got1[1].any())
