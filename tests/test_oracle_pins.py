"""Pins for the oracle: checks against what the pages and the mathematics fix.

Nothing here re-types the oracle's own loop.  Each test uses an independent route: a value
printed on the pages (tests/golden), a hand-worked example, a closed form, an invariant the
pages state, a special case that reduces to a library routine (numpy matmul/convolve, scipy
expit), brute force on tiny inputs, or a second derivation (the chunkwise WY form).
"""
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from hybrid_linear_attention_gb300 import inputs
from tests._chunk_form import chunked_head

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_kv(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, val = line.split()
                vals[key] = float(val)
    return vals


def _rand_case(T, H, d, seed, dtype=torch.float32, init=False, lengths=None):
    lengths = lengths or [T]
    return inputs.kda_inputs(lengths, H, d, seed=seed, io_dtype=dtype,
                             init_state="all" if init else None)


def _f64(t):
    return t.double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


# ---------------------------------------------------------------------------------------
# Payload figures printed on the pages
# ---------------------------------------------------------------------------------------

def test_state_bytes_match_pages():
    gv = _golden_kv("payload.txt")
    H, d, L = int(gv["heads"]), int(gv["head_dim"]), int(gv["kda_layers"])
    per_layer = oracle.state_bytes(H, d, d, 4)
    assert per_layer // 4 == gv["state_values_per_layer"] == 64 * 128 * 128
    assert per_layer == 64 * 128 * 128 * 4
    assert L * per_layer == gv["state_fp32_mib_per_sequence"] * 2**20
    assert L * oracle.state_bytes(H, d, d, 2) == gv["state_bf16_mib_per_sequence"] * 2**20


def test_conv_tail_bytes_match_pages():
    gv = _golden_kv("payload.txt")
    H, d, L = int(gv["heads"]), int(gv["head_dim"]), int(gv["kda_layers"])
    tails = L * oracle.conv_tail_bytes(H, d, int(gv["conv_width"]), 2)
    assert tails == 9_289_728
    assert tails < gv["conv_tail_upper_bound_mib"] * 2**20          # "under 10 MiB"
    assert round(tails / 1e6) == gv["conv_tail_approx_mb"]           # "9 MB"


# ---------------------------------------------------------------------------------------
# Hand-worked example
# ---------------------------------------------------------------------------------------

def test_worked_example_d2():
    rows, S_rows = [], []
    with open(os.path.join(GOLDEN, "worked_example_d2.txt")) as f:
        for line in f:
            p = line.split()
            if not p or p[0].startswith("#"):
                continue
            if p[0] == "t":
                rows.append([float(x) for x in p[2:]])
            elif p[0] == "S":
                S_rows.append([float(x) for x in p[1:]])
    rows = np.array(rows)
    T = rows.shape[0]
    k = rows[:, 0:2].reshape(T, 1, 2).astype(np.float32)
    v = rows[:, 2:4].reshape(T, 1, 2).astype(np.float32)
    q = rows[:, 4:6].reshape(T, 1, 2).astype(np.float32)
    g = np.log(rows[:, 6:8]).reshape(T, 1, 2).astype(np.float32)
    beta = rows[:, 8].reshape(T, 1).astype(np.float32)
    r = oracle.kda_forward(q, k, v, g, beta, np.array([0, T], np.int32), qk_l2norm=False)
    np.testing.assert_allclose(r["out"][:, 0, :], rows[:, 9:11], rtol=0, atol=1e-7)
    np.testing.assert_allclose(r["final_state"][0, 0], np.array(S_rows), rtol=0, atol=1e-7)


# ---------------------------------------------------------------------------------------
# Invariants and closed forms
# ---------------------------------------------------------------------------------------

def test_no_decay_no_write_leaves_state_unchanged():
    """alpha = 1, beta = 0: the state is untouched and every read is S0^T q (numpy matmul)."""
    c = _rand_case(37, 3, 16, seed=1, init=True)
    g = torch.zeros_like(c["g"])
    beta = torch.zeros_like(c["beta"])
    r = oracle.kda_forward(c["q"], c["k"], c["v"], g, beta, c["cu_seqlens"],
                           init_state=c["init_state"], l2_eps=0.0)
    S0 = _f64(c["init_state"])
    assert np.array_equal(r["final_state"], S0)
    qn = _f64(c["q"]) / np.linalg.norm(_f64(c["q"]), axis=-1, keepdims=True)
    want = np.einsum("hij,thi->thj", S0[0], qn)
    np.testing.assert_allclose(r["out"], want, rtol=1e-12, atol=1e-14)


def test_pure_decay_closed_form():
    """beta = 0, any alpha: S_T = Diag(prod alpha) S0, and each read sees the decay so far."""
    c = _rand_case(23, 2, 8, seed=2, init=True)
    beta = torch.zeros_like(c["beta"])
    r = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], beta, c["cu_seqlens"],
                           init_state=c["init_state"], l2_eps=0.0)
    S0 = _f64(c["init_state"])[0]
    cum = np.cumsum(_f64(c["g"]), axis=0)  # [T, H, d]
    np.testing.assert_allclose(r["final_state"][0], np.exp(cum[-1])[:, :, None] * S0,
                               rtol=1e-12, atol=0)
    qn = _f64(c["q"]) / np.linalg.norm(_f64(c["q"]), axis=-1, keepdims=True)
    want = np.einsum("thi,hij->thj", qn * np.exp(cum), S0)
    np.testing.assert_allclose(r["out"], want, rtol=1e-11, atol=1e-15)


def test_clamp_at_safe_forget_bound():
    """Log-retention below the -5 lower bound acts exactly like -5."""
    c = _rand_case(19, 2, 8, seed=3, init=True)
    g_low = c["g"].clone()
    g_low[::2] = -50.0
    g_bound = c["g"].clone()
    g_bound[::2] = -5.0
    a = oracle.kda_forward(c["q"], c["k"], c["v"], g_low, c["beta"], c["cu_seqlens"],
                           init_state=c["init_state"])
    b = oracle.kda_forward(c["q"], c["k"], c["v"], g_bound, c["beta"], c["cu_seqlens"],
                           init_state=c["init_state"])
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["final_state"], b["final_state"])


@pytest.mark.parametrize("seed", [4, 5, 6])
def test_delta_write_corrects_prediction_exactly(seed):
    """beta = 1 and unit k: after the write, S^T k = v exactly, for any alpha and prior
    state -- the prediction for the current key is corrected all the way to v."""
    c = _rand_case(11, 2, 16, seed=seed, init=True)
    beta = torch.ones_like(c["beta"])
    for T in (1, 5, 11):
        cu = np.array([0, T], np.int32)
        r = oracle.kda_forward(c["q"][:T], c["k"][:T], c["v"][:T], c["g"][:T], beta[:T], cu,
                               init_state=c["init_state"], l2_eps=0.0)
        kT = _f64(c["k"][T - 1])
        kT = kT / np.linalg.norm(kT, axis=-1, keepdims=True)
        pred = np.einsum("hij,hi->hj", r["final_state"][0], kT)
        np.testing.assert_allclose(pred, _f64(c["v"][T - 1]), rtol=0, atol=1e-12)


def test_orthonormal_keys_are_retrieved():
    """Orthonormal keys, alpha = 1, beta = 1, S0 = 0: reading with k_i returns v_i."""
    d, m = 16, 12
    rng = np.random.default_rng(7)
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    keys = Qm[:, :m].T.astype(np.float32)               # m orthonormal rows (fp32)
    keys64 = keys.astype(np.float64)
    # the keys are stored in fp32, so they are orthonormal only to fp32 rounding; the
    # tolerance scales with that measured departure
    v = rng.standard_normal((m, d)).astype(np.float32)
    q = np.zeros((m, 1, d), np.float32)
    q[-1, 0] = keys[0]                                    # last read asks for key 0
    g = np.zeros((m, 1, d), np.float32)
    beta = np.ones((m, 1), np.float32)
    r = oracle.kda_forward(q, keys[:, None, :], v[:, None, :], g, beta,
                           np.array([0, m], np.int32), qk_l2norm=False)
    S = r["final_state"][0, 0]
    ortho_err = np.abs(keys64 @ keys64.T - np.eye(m)).max()   # fp32 rounding of the keys
    for i in range(m):
        np.testing.assert_allclose(S.T @ keys64[i], v[i], rtol=0, atol=200 * ortho_err + 1e-12)
    np.testing.assert_allclose(r["out"][-1, 0], v[0], rtol=0, atol=200 * ortho_err + 1e-12)


def test_one_token_from_zero_state():
    """From S0 = 0 a single token reads o = beta (k.q) v (scale 1)."""
    c = _rand_case(1, 4, 16, seed=8)
    r = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                           l2_eps=0.0)
    qn = _f64(c["q"][0]) / np.linalg.norm(_f64(c["q"][0]), axis=-1, keepdims=True)
    kn = _f64(c["k"][0]) / np.linalg.norm(_f64(c["k"][0]), axis=-1, keepdims=True)
    want = (_f64(c["beta"][0]) * (qn * kn).sum(-1))[:, None] * _f64(c["v"][0])
    np.testing.assert_allclose(r["out"][0], want, rtol=1e-13, atol=1e-16)


def test_scale_multiplies_output_only():
    c = _rand_case(9, 2, 8, seed=9, init=True)
    a = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                           init_state=c["init_state"])
    b = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                           init_state=c["init_state"], scale=1 / np.sqrt(8))
    np.testing.assert_allclose(b["out"], a["out"] / np.sqrt(8), rtol=1e-14)
    assert np.array_equal(a["final_state"], b["final_state"])


def test_l2_normalisation_is_scale_invariant():
    """q, k are L2-normalised: scaling them by a constant changes nothing (eps aside)."""
    c = _rand_case(13, 2, 8, seed=10, init=True)
    a = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                           init_state=c["init_state"], l2_eps=0.0)
    b = oracle.kda_forward(c["q"] * 4, c["k"] * 0.25, c["v"], c["g"], c["beta"],
                           c["cu_seqlens"], init_state=c["init_state"], l2_eps=0.0)
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------------------------------
# Brute force on tiny inputs: the unrolled product form
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("d,T,seed", [(2, 3, 11), (4, 7, 12), (8, 12, 13)])
def test_matches_unrolled_product_form(d, T, seed):
    """S_T = prod_t (I - b_t k_t k_t^T) Diag(a_t) S0 + sum_s [prod_{r>s} (...)] b_s k_s v_s^T,
    o_t = S_t^T q_t -- built from explicit d x d matrices, no recurrence loop shared."""
    c = _rand_case(T, 1, d, seed=seed, init=True)
    r = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                           init_state=c["init_state"], l2_eps=0.0)
    q = _f64(c["q"][:, 0]); k = _f64(c["k"][:, 0]); v = _f64(c["v"][:, 0])
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    a = np.exp(np.maximum(_f64(c["g"][:, 0]), -5.0))
    b = _f64(c["beta"][:, 0])
    S0 = _f64(c["init_state"][0, 0])
    M = [(np.eye(d) - b[t] * np.outer(k[t], k[t])) @ np.diag(a[t]) for t in range(T)]
    for t_end in range(1, T + 1):
        prod_all = np.eye(d)
        for t in range(t_end):
            prod_all = M[t] @ prod_all
        S = prod_all @ S0
        for s in range(t_end):
            tail = np.eye(d)
            for t in range(s + 1, t_end):
                tail = M[t] @ tail
            S = S + tail @ (b[s] * np.outer(k[s], v[s]))
        np.testing.assert_allclose(r["out"][t_end - 1, 0], S.T @ q[t_end - 1], rtol=1e-11,
                                   atol=1e-13)
    np.testing.assert_allclose(r["final_state"][0, 0], S, rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------------------------------
# Second derivation: the chunkwise WY/UT form
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("C", [1, 16, 64])
@pytest.mark.parametrize("T", [1, 45, 130])
def test_chunk_form_equals_recurrence(C, T):
    c = _rand_case(T, 2, 16, seed=20 + T, init=True)
    r = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                           init_state=c["init_state"], scale=0.5)
    for h in range(2):
        o, S = chunked_head(_f64(c["q"][:, h]), _f64(c["k"][:, h]), _f64(c["v"][:, h]),
                            _f64(c["g"][:, h]), _f64(c["beta"][:, h]),
                            _f64(c["init_state"][0, h]), C, scale=0.5)
        np.testing.assert_allclose(r["out"][:, h], o, rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(r["final_state"][0, h], S, rtol=1e-9, atol=1e-12)


# ---------------------------------------------------------------------------------------
# Stability, independence of heads and sequences, resume
# ---------------------------------------------------------------------------------------

def test_state_norm_growth_bound():
    """With unit keys, ||I - b k k^T|| <= 1 and alpha <= 1, so ||S_t|| <= ||S_t-1|| + b ||v||."""
    c = _rand_case(200, 2, 16, seed=30, init=True)
    r = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                           init_state=c["init_state"], l2_eps=0.0, want_state_norm=True)
    for h in range(2):
        norms = r["state_norm"][h]
        prev = np.concatenate([[np.linalg.norm(_f64(c["init_state"][0, h]))], norms[:-1]])
        bound = prev + _f64(c["beta"][:, h]) * np.linalg.norm(_f64(c["v"][:, h]), axis=1)
        assert np.all(norms <= bound * (1 + 1e-12))


def test_heads_are_independent_and_permute():
    c = _rand_case(30, 4, 8, seed=31, init=True)
    perm = [2, 0, 3, 1]
    a = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                           init_state=c["init_state"])
    b = oracle.kda_forward(c["q"][:, perm], c["k"][:, perm], c["v"][:, perm], c["g"][:, perm],
                           c["beta"][:, perm], c["cu_seqlens"],
                           init_state=c["init_state"][:, perm])
    assert np.array_equal(b["out"], a["out"][:, perm])
    assert np.array_equal(b["final_state"], a["final_state"][:, perm])


def test_packed_batch_equals_separate_sequences():
    lens = [5, 0, 17, 1, 64]
    c = inputs.kda_inputs(lens, 2, 8, seed=32, io_dtype=torch.bfloat16, init_state="even")
    packed = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                                init_state=c["init_state"])
    cu = c["cu_seqlens"].tolist()
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        one = oracle.kda_forward(c["q"][sl], c["k"][sl], c["v"][sl], c["g"][sl], c["beta"][sl],
                                 np.array([0, lens[n]], np.int32),
                                 init_state=c["init_state"][n:n + 1])
        assert np.array_equal(packed["out"][sl], one["out"])
        assert np.array_equal(packed["final_state"][n], one["final_state"][0])
    # an empty sequence hands its initial state straight through
    assert np.array_equal(packed["final_state"][1], _f64(c["init_state"][1]))


def test_split_resume_equals_full_run():
    """prefill(T1 + T2) == prefill(T2, init = final of prefill(T1)): a saved state is a
    valid checkpoint at a token boundary."""
    c = _rand_case(90, 2, 16, seed=33, init=True)
    full = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                              init_state=c["init_state"])
    for T1 in (1, 37, 64):
        a = oracle.kda_forward(c["q"][:T1], c["k"][:T1], c["v"][:T1], c["g"][:T1],
                               c["beta"][:T1], np.array([0, T1], np.int32),
                               init_state=c["init_state"])
        b = oracle.kda_forward(c["q"][T1:], c["k"][T1:], c["v"][T1:], c["g"][T1:],
                               c["beta"][T1:], np.array([0, 90 - T1], np.int32),
                               init_state=a["final_state"])
        np.testing.assert_allclose(b["out"], full["out"][T1:], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(b["final_state"], full["final_state"], rtol=1e-12,
                                   atol=1e-15)


def test_unit_subset_matches_full_run():
    c = inputs.kda_inputs([7, 20], 3, 8, seed=34, init_state="all")
    full = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                              init_state=c["init_state"])
    sub = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                             init_state=c["init_state"], units=[(1, 2), (0, 1)])
    assert np.array_equal(sub["unit_out"][0], full["out"][7:27, 2])
    assert np.array_equal(sub["final_state"][1], full["final_state"][0, 1])


# ---------------------------------------------------------------------------------------
# Output norm and sigmoid gate
# ---------------------------------------------------------------------------------------

def test_output_norm_with_open_gate_has_unit_rms():
    """gate -> +inf, w = 1: every head's output row has RMS 1 (up to eps)."""
    c = _rand_case(25, 2, 16, seed=40, init=True)
    gate = torch.full((25, 2, 16), 100.0)
    r = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                           init_state=c["init_state"], gate=gate, norm_eps=0.0)
    rms = np.sqrt((r["out"] ** 2).mean(-1))
    np.testing.assert_allclose(rms, 1.0, rtol=1e-13)


def test_output_norm_gate_and_weight():
    """With gate logits z and weight w, out / (w sigmoid(z)) is the RMS-normalised read."""
    c = _rand_case(25, 2, 16, seed=41, init=True)
    gate = inputs.normal((25, 2, 16), seed=42, dtype=torch.float32)
    w = inputs.normal((16,), seed=43, dtype=torch.float32)
    plain = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                               init_state=c["init_state"])["out"]
    gated = oracle.kda_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                               init_state=c["init_state"], gate=gate, norm_w=w,
                               norm_eps=1e-6)["out"]
    rms = np.sqrt((plain ** 2).mean(-1, keepdims=True) + 1e-6)
    want = plain / rms * _f64(w) * expit(_f64(gate))
    np.testing.assert_allclose(gated, want, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------------------------------
# Prologue: short convolution, SiLU, q/k normalisation, gate activations, conv tail
# ---------------------------------------------------------------------------------------

def test_conv_identity_tap_is_silu():
    """Weights [0, 0, 0, 1] make the convolution the identity: y = SiLU(x) = x sigmoid(x)."""
    H, d = 2, 8
    p = inputs.prologue_inputs([9, 4], H, d, seed=50)
    w = torch.zeros(3 * H * d, 4, dtype=torch.bfloat16)
    w[:, 3] = 1.0
    r = oracle.prologue(p["x"], w, p["cu_seqlens"], H, d, conv_state=p["conv_state"])
    x = _f64(p["x"])
    np.testing.assert_allclose(r["y"], x * expit(x), rtol=1e-15, atol=0)


def test_conv_matches_numpy_convolve_with_history():
    H, d = 1, 8
    lens = [1, 2, 3, 11]
    p = inputs.prologue_inputs(lens, H, d, seed=51)
    r = oracle.prologue(p["x"], p["conv_w"], p["cu_seqlens"], H, d, conv_state=p["conv_state"])
    x, w, st = _f64(p["x"]), _f64(p["conv_w"]), _f64(p["conv_state"])
    cu = p["cu_seqlens"].tolist()
    for n in range(len(lens)):
        for c in range(3 * H * d):
            hist = np.concatenate([st[n, :, c], x[cu[n]:cu[n + 1], c]])
            # causal correlation: y[t] = sum_j w[j] x[t-3+j]  ==  convolve with reversed taps
            pre = np.convolve(hist, w[c, ::-1], mode="valid")
            np.testing.assert_allclose(r["y"][cu[n]:cu[n + 1], c], pre * expit(pre),
                                       rtol=1e-13, atol=1e-15)


def test_conv_without_state_pads_with_zeros():
    H, d = 1, 4
    p = inputs.prologue_inputs([6], H, d, seed=52, conv_state=False)
    a = oracle.prologue(p["x"], p["conv_w"], p["cu_seqlens"], H, d)
    zeros = torch.zeros(1, 3, 3 * H * d, dtype=torch.bfloat16)
    b = oracle.prologue(p["x"], p["conv_w"], p["cu_seqlens"], H, d, conv_state=zeros)
    assert np.array_equal(a["y"], b["y"])
    assert np.array_equal(a["conv_state"], b["conv_state"])


def test_conv_tail_brute_force_indexing():
    """The new tail is the last three raw inputs, reaching into the old tail when a
    sequence is shorter than three tokens (byte-exact)."""
    H, d = 1, 4
    lens = [0, 1, 2, 3, 7]
    p = inputs.prologue_inputs(lens, H, d, seed=53)
    r = oracle.prologue(p["x"], p["conv_w"], p["cu_seqlens"], H, d, conv_state=p["conv_state"])
    xb = p["x"].view(torch.int16).numpy().view(np.uint16)
    sb = p["conv_state"].view(torch.int16).numpy().view(np.uint16)
    cu = p["cu_seqlens"].tolist()
    for n, L in enumerate(lens):
        hist = np.concatenate([sb[n], xb[cu[n]:cu[n + 1]]], axis=0)   # [3 + L, C]
        assert np.array_equal(r["conv_state"][n], hist[-3:])


def test_prologue_l2_and_gate_activations():
    H, d = 2, 16
    p = inputs.prologue_inputs([10], H, d, seed=54)
    r = oracle.prologue(p["x"], p["conv_w"], p["cu_seqlens"], H, d, conv_state=p["conv_state"],
                        l2norm_qk=True, l2_eps=0.0, beta_logit=p["beta_logit"],
                        g_raw=p["g_raw"] - 1.0)
    y = r["y"].reshape(10, 3, H, d)
    np.testing.assert_allclose(np.linalg.norm(y[:, :2], axis=-1), 1.0, rtol=1e-14)
    plain = oracle.prologue(p["x"], p["conv_w"], p["cu_seqlens"], H, d,
                            conv_state=p["conv_state"])["y"].reshape(10, 3, H, d)
    assert np.array_equal(y[:, 2], plain[:, 2])          # v is not normalised
    np.testing.assert_allclose(r["beta"], expit(_f64(p["beta_logit"])), rtol=1e-15)
    np.testing.assert_array_equal(r["g"], np.maximum(_f64(p["g_raw"] - 1.0), -5.0))


# ---------------------------------------------------------------------------------------
# FP8 E4M3 output quantisation
# ---------------------------------------------------------------------------------------

def test_fp8_e4m3_codes_pinned_by_the_format():
    """Codes fixed by the E4M3 layout (sign, 4 exponent bits with bias 7, 3 mantissa bits,
    no infinities, largest finite 448): exact values, ties to the even code, subnormals,
    saturation."""
    table = [
        (0.0, 0x00), (-0.0, 0x80), (1.0, 0x38), (-1.0, 0xB8), (0.5, 0x30), (448.0, 0x7E),
        (-448.0, 0xFE), (240.0, 0x77), (2.0 ** -6, 0x08), (2.0 ** -9, 0x01),
        (7 * 2.0 ** -9, 0x07),
        (1.0625, 0x38),          # halfway 1 | 1.125: even mantissa 0
        (1.1875, 0x3A),          # halfway 1.125 | 1.25: even mantissa 2
        (2.0 ** -10, 0x00),      # halfway 0 | 2^-9: even code 0
        (3 * 2.0 ** -10, 0x02),  # halfway 2^-9 | 2^-8: even code 2
        (15 * 2.0 ** -10, 0x08), # halfway 7*2^-9 | 2^-6: rounds up into the normal binade
        (464.0, 0x7E), (480.0, 0x7E), (1e6, 0x7E), (-1e6, 0xFE), (np.inf, 0x7E),
    ]
    x = np.array([v for v, _ in table])
    got = oracle.fp8_e4m3_encode(x)
    assert [int(c) for c in got] == [c for _, c in table]
    assert oracle.fp8_e4m3_encode(np.array([np.nan]))[0] == 0x7F


def test_fp8_e4m3_matches_the_library_conversion():
    """In range, the encoder is the round-to-nearest-even conversion torch implements for
    float8_e4m3fn (fp64 and fp32 inputs)."""
    rng = np.random.default_rng(60)
    x = rng.standard_normal(100000) * np.exp2(rng.uniform(-12, 9, 100000))
    x = x[np.abs(x) <= 448.0]
    for arr in (x, x.astype(np.float32)):
        want = torch.from_numpy(arr).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(oracle.fp8_e4m3_encode(arr), want)


def test_fp8_e4m3_every_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.fp8_e4m3_decode(codes)
    assert np.array_equal(oracle.fp8_e4m3_encode(vals), codes)
    assert np.isnan(oracle.fp8_e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    pos = np.sort(vals[vals > 0])
    assert pos[0] == 2.0 ** -9 and pos[-1] == 448.0 and len(np.unique(pos)) == 126


def test_fp8_group_quantisation_bounds():
    """Each group's largest magnitude lands on +-448 (code 0x7E / 0xFE); every value comes
    back within half a step of its binade (2^-4 relative in the normal range, 2^-10 of the
    scale in the subnormal one)."""
    rng = np.random.default_rng(61)
    x = rng.standard_normal((37, 3, 256)) * np.exp2(rng.uniform(-6, 6, (37, 3, 1)))
    codes, scales = oracle.fp8_quantize_groups(x, 128)
    assert scales.shape == (37, 3, 2)
    xg = x.reshape(37, 3, 2, 128)
    np.testing.assert_allclose(scales, np.abs(xg).max(-1) / 448.0, rtol=1e-15)
    cg = codes.reshape(37, 3, 2, 128)
    top = np.abs(xg).argmax(-1)
    assert np.isin(np.take_along_axis(cg, top[..., None], -1), [0x7E, 0xFE]).all()
    deq = oracle.fp8_dequantize_groups(codes, scales, 128).reshape(xg.shape)
    y = np.abs(xg) / scales[..., None]
    half = np.where(y >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 4),
                    2.0 ** -10)
    assert (np.abs(deq - xg) <= half * scales[..., None] * (1 + 1e-12)).all()
    # an all-zero group keeps a positive scale and zero codes
    z_codes, z_scales = oracle.fp8_quantize_groups(np.zeros((2, 128)), 128)
    assert (z_codes == 0).all() and (z_scales > 0).all()


# ---------------------------------------------------------------------------------------
# Absorbed gated-MLA decode
# ---------------------------------------------------------------------------------------

def _mla_case(B, H, L, seed, lengths=None):
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std).to(torch.bfloat16)
    return dict(q_nope=bf(B, H, 128), q_rope=bf(B, H, 64), c=bf(B, L, 512), r=bf(B, L, 64),
                w_uk=bf(H, 128, 512, std=0.05), w_uv=bf(H, 128, 512, std=0.05),
                gate=bf(B, H), lengths=np.array(lengths if lengths is not None else [L] * B))


def test_mla_absorbed_path_equals_the_expanded_one():
    """The pages' identity: moving W_K,i into the query and W_V,i after the latent sum gives
    the same attention function as expanding every cached position."""
    m = _mla_case(4, 6, 23, seed=70, lengths=[23, 1, 7, 16])
    args = (m["q_nope"], m["q_rope"], m["c"], m["r"], m["lengths"], m["w_uk"], m["w_uv"],
            m["gate"])
    e, a = oracle.mla_decode_expanded(*args), oracle.mla_decode_absorbed(*args)
    np.testing.assert_allclose(a, e, rtol=0, atol=1e-12 * np.abs(e).max())


def test_mla_one_cached_position_returns_its_value():
    m = _mla_case(2, 3, 5, seed=71, lengths=[1, 1])
    out = oracle.mla_decode_absorbed(m["q_nope"], m["q_rope"], m["c"], m["r"], m["lengths"],
                                     m["w_uk"], m["w_uv"], m["gate"])
    c0 = m["c"][:, 0].double().numpy()
    wv = m["w_uv"].double().numpy()
    sig = expit(m["gate"].double().numpy())
    want = np.einsum("hvl,bl->bhv", wv, c0) * sig[..., None]
    np.testing.assert_allclose(out, want, rtol=1e-13, atol=1e-15)


def test_mla_zero_query_averages_the_values():
    m = _mla_case(2, 2, 6, seed=72, lengths=[6, 3])
    z = torch.zeros_like(m["q_nope"]), torch.zeros_like(m["q_rope"])
    out = oracle.mla_decode_expanded(z[0], z[1], m["c"], m["r"], m["lengths"], m["w_uk"],
                                     m["w_uv"], m["gate"])
    wv = m["w_uv"].double().numpy()
    sig = expit(m["gate"].double().numpy())
    for b, L in enumerate(m["lengths"]):
        mean_c = m["c"][b, :L].double().numpy().mean(0)
        np.testing.assert_allclose(out[b], (wv @ mean_c) * sig[b][:, None], rtol=1e-12)


def test_mla_latent_attention_brute_force_and_lse():
    """The attention core against scalar loops, and its log-sum-exp against scipy's."""
    from scipy.special import logsumexp
    rng = np.random.default_rng(73)
    q = rng.standard_normal((1, 2, 576))
    kv = rng.standard_normal((1, 3, 576))
    z, lse = oracle.mla_latent_attention(q, kv, np.array([3]), scale=0.05)
    for i in range(2):
        s = [0.05 * sum(q[0, i, d] * kv[0, t, d] for d in range(576)) for t in range(3)]
        w = [np.exp(x - max(s)) for x in s]
        for dd in (0, 7, 511):
            want = sum(w[t] * kv[0, t, dd] for t in range(3)) / sum(w)
            assert abs(z[0, i, dd] - want) <= 1e-12 * max(1.0, abs(want))
        assert abs(lse[0, i] - logsumexp(s)) <= 1e-12 * abs(lse[0, i])
    z0, l0 = oracle.mla_latent_attention(q, kv, np.array([0]))
    assert not z0.any() and np.isneginf(l0).all()
