"""GPU edge cases: log-retention far below the safe-forget bound, many short sequences (more
CTA rows than SMs), more heads than SMs.

The safe forget gate's log-retention lower bound of -5 ("Ling-3.1-flash: Grouped Routing and
Two Different MLA Caches", section "KDA replaces a token list with a recurrent matrix") is
applied inside every kernel, so inputs far below it must give the same bits as inputs clamped
at it beforehand, on every prefill path and in decode.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gb300 import inputs, kda
from tests import _gpu
from tests._parity import max_err_rel_rms, out_error

pytestmark = pytest.mark.gpu


def _oracle(inp, gate):
    return oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              inp["cu_seqlens"], init_state=inp.get("init_state"),
                              gate=inp.get("gate") if gate else None,
                              norm_w=inp.get("norm_w") if gate else None)


def _tol(io):
    return 1e-2 if io == torch.bfloat16 else 1e-4


@pytest.mark.parametrize("path", ["pair", "fused", "token-serial"])
def test_log_retention_below_the_bound_gives_the_bits_of_the_bound(path):
    if path == "token-serial":
        d, io = 16, torch.float32
    else:
        d, io = 128, torch.bfloat16
    inp = inputs.kda_inputs([70, 130], 2, d, seed=61, io_dtype=io, init_state="all", gate=True)
    inp["g"] = inputs.uniform(tuple(inp["g"].shape), -50.0, 0.0, seed=62)
    assert float((inp["g"] < -5).float().mean()) > 0.8
    p = kda.params(H=2, d=d, io_dtype=io,
                   prefill_form="auto" if path == "token-serial" else path)
    out_raw, fin_raw = _gpu.prefill(inp, p, gate=True)
    clamped = dict(inp, g=inp["g"].clamp(min=-5.0))
    out_c, fin_c = _gpu.prefill(clamped, p, gate=True)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    assert torch.equal(out_raw, out_c) and torch.equal(fin_raw, fin_c)
    ref = _oracle(inp, True)  # the oracle clamps too
    assert out_error(out_raw, ref["out"], io) <= _tol(io)
    assert max_err_rel_rms(fin_raw, ref["final_state"]) <= (1e-3 if io == torch.bfloat16
                                                            else 1e-4)


def test_decode_log_retention_below_the_bound_gives_the_bits_of_the_bound():
    H, d, n = 4, 128, 5
    p = kda.params(H=H, d=d)
    _gpu.lib()
    S0 = inputs.normal((n, H, d, d), seed=63, dtype=torch.float32, std=0.02).cuda()
    st = inputs.decode_inputs(n, H, d, seed=64)
    q, k, v = (inputs.normal((n, H, d), seed=65 + i).cuda() for i in range(3))
    g = inputs.uniform((n, H, d), -50.0, 0.0, seed=68).cuda()
    beta = st["beta"].cuda()
    outs, states = [], []
    for gg in (g, g.clamp(min=-5.0)):
        state = S0.clone()
        out = torch.empty((n, H, d), dtype=torch.bfloat16, device="cuda")
        kda.kda_decode_step(p, q, k, v, gg, beta, state, out)
        outs.append(out)
        states.append(state)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    assert torch.equal(outs[0], outs[1]) and torch.equal(states[0], states[1])


def test_many_short_sequences():
    """1200 sequences of 0-70 tokens: more (head, sequence) CTAs than SMs, most of them a single
    ragged chunk, a fifth of them empty."""
    rng = np.random.default_rng(71)
    lens = [int(x) for x in rng.integers(0, 71, size=1200)]
    lens = [0 if i % 5 == 0 else L for i, L in enumerate(lens)]
    inp = inputs.kda_inputs(lens, 2, 128, seed=72, init_state="even", gate=True)
    p = kda.params(H=2, d=128)
    out, fin = _gpu.prefill(inp, p, gate=True)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    ref = _oracle(inp, True)
    assert out_error(out, ref["out"], torch.bfloat16) <= 1e-2
    assert max_err_rel_rms(fin, ref["final_state"]) <= 1e-3
    # the empty sequences hand their initial state straight on
    empty = [i for i, L in enumerate(lens) if L == 0]
    assert torch.equal(fin[empty].cpu(), inp["init_state"][empty])


def test_more_heads_than_sms():
    inp = inputs.kda_inputs([1, 64, 65], 160, 128, seed=73, init_state="all")
    p = kda.params(H=160, d=128)
    out, fin = _gpu.prefill(inp, p)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    ref = _oracle(inp, False)
    assert out_error(out, ref["out"], torch.bfloat16) <= 1e-2
    assert max_err_rel_rms(fin, ref["final_state"]) <= 1e-3


@pytest.mark.parametrize("seed", range(10))
def test_prefill_random_batches(seed):
    """Seeded random packed batches on both tensor-core forms: 1-6 sequences of 0-400 tokens
    (chunk edges and one-token tails among them), 1-3 heads, the norm and gate on or off, an
    initial state on all, some or none of the sequences; every (sequence, head) unit against
    the oracle."""
    rng = np.random.default_rng(3000 + seed)
    n = int(rng.integers(1, 7))
    lens = [int(x) for x in rng.integers(0, 401, size=n)]
    edges = [0, 1, 63, 64, 65, 128, 129]
    lens[int(rng.integers(0, n))] = edges[seed % len(edges)]
    H = int(rng.integers(1, 4))
    gate = bool(seed % 2)
    init = [None, "all", "even"][seed % 3]
    form = "pair" if seed % 4 < 2 else "fused"
    inp = inputs.kda_inputs(lens, H, 128, seed=3100 + seed, init_state=init, gate=gate)
    p = kda.params(H=H, d=128, prefill_form=form)
    out, fin = _gpu.prefill(inp, p, gate=gate)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    ref = _oracle(inp, gate)
    cu = inp["cu_seqlens"].tolist()
    for s in range(n):
        if lens[s] == 0:
            continue
        for h in range(H):
            e = out_error(out[cu[s]:cu[s + 1], h], ref["out"][cu[s]:cu[s + 1], h], torch.bfloat16)
            assert e <= 1e-2, f"seed {seed}: sequence {s} (length {lens[s]}), head {h}: {e:.3g}"
    assert max_err_rel_rms(fin, ref["final_state"]) <= 1e-3
