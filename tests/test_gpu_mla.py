"""GPU parity: the absorbed gated-MLA decode against the fp64 oracle.

Tolerance: bf16 operands with fp32 accumulation (the softmax weights are rounded to bf16 as
tensor-core operands, the normaliser sums the same rounded weights), so the bound is the bf16
one of the KDA path: max |err| <= 1e-2 of the output RMS, beyond half a bf16 ulp for outputs
stored in bf16.  Cache rows at or past a sequence's length hold NaN here: they must not
reach the result.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gb300 import kda
from tests import _gpu
from tests._parity import max_err_rel_rms, out_error, to64

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _case(lengths, L, seed, q_std=1.0):
    g = torch.Generator().manual_seed(seed)
    B = len(lengths)
    bf = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std).to(torch.bfloat16)
    cache = bf(B, L, 576)
    for b, n in enumerate(lengths):  # rows past the length: NaN, never to be read into z
        if 0 <= n < L:
            cache[b, n:] = float("nan")
    return dict(q_cat=bf(B, 64, 576, std=q_std), cache=cache,
                lengths=torch.tensor(lengths, dtype=torch.int32),
                q_nope=bf(B, 64, 128), q_rope=bf(B, 64, 64),
                w_uk=bf(64, 128, 512, std=0.05), w_uv=bf(64, 128, 512, std=0.05),
                gate=bf(B, 64))


def _latent(m):
    _gpu.lib()
    z = torch.full((m["q_cat"].shape[0], 64, 512), 7.0, device="cuda")
    kda.mla_decode_latent(m["q_cat"].cuda(), m["cache"].cuda(), m["lengths"].cuda(), z)
    torch.cuda.synchronize()
    return z


@pytest.mark.parametrize("q_std", [1.0, 4.0])
def test_latent_attention_matches_the_oracle(q_std):
    """Ragged lengths around the 64-position tile edges (1, 127, 128, 129, 300), peaked
    scores (q_std 4: the running max moves and Z is rescaled), NaN past every length."""
    lengths = [1, 127, 128, 129, 300, 256]
    m = _case(lengths, 320, seed=800 + int(q_std), q_std=q_std)
    z = _latent(m)
    kda.kda_check_device_error()
    clean = m["cache"].clone()
    for b, n in enumerate(lengths):
        clean[b, n:] = 0
    ref, _ = oracle.mla_latent_attention(m["q_cat"], clean, np.array(lengths),
                                         scale=kda.MLA_SCALE)
    for b in range(len(lengths)):
        e = max_err_rel_rms(z[b], ref[b])
        assert e <= TOL, f"sequence {b} (length {lengths[b]}): {e:.3g}"
    assert torch.isfinite(z).all()


def test_latent_attention_long_cache_sampled():
    """The bench's cache length (4096 positions, 32 tiles) on a few sequences."""
    lengths = [4096, 4000, 2049]
    m = _case(lengths, 4096, seed=810)
    z = _latent(m)
    kda.kda_check_device_error()
    clean = m["cache"].clone()
    for b, n in enumerate(lengths):
        clean[b, n:] = 0
    ref, _ = oracle.mla_latent_attention(m["q_cat"], clean, np.array(lengths),
                                         scale=kda.MLA_SCALE)
    assert max_err_rel_rms(z, ref) <= TOL


def test_empty_and_out_of_range_lengths():
    """Length 0 gives z = 0; a length outside 0..cache_len is treated as 0 and reported."""
    m = _case([0, 5, -1, 1000], 64, seed=820)
    z = _latent(m)
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_check_device_error()
    assert ei.value.status == kda.KDA_ERR_BAD_INDEX
    assert not z[0].any() and not z[2].any() and not z[3].any()
    clean = m["cache"][1:2].clone()
    clean[0, 5:] = 0
    ref, _ = oracle.mla_latent_attention(m["q_cat"][1:2], clean, np.array([5]),
                                         scale=kda.MLA_SCALE)
    assert max_err_rel_rms(z[1:2], ref) <= TOL


def test_mla_decode_matches_the_expanded_oracle():
    """The whole step (absorption, latent attention, value up-projection, gate) against the
    pages' expanded reference path computed in fp64."""
    lengths = [300, 1, 129, 64]
    m = _case(lengths, 320, seed=830)
    _gpu.lib()
    B = len(lengths)
    q_cat = torch.empty((B, 64, 576), dtype=torch.bfloat16, device="cuda")
    z = torch.empty((B, 64, 512), device="cuda")
    out = torch.empty((B, 64, 128), dtype=torch.bfloat16, device="cuda")
    c = _gpu.cuda
    kda.mla_decode(c(m["q_nope"]), c(m["q_rope"]), c(m["w_uk"]), c(m["w_uv"]), c(m["cache"]),
                   c(m["lengths"]), c(m["gate"]), q_cat, z, out)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    # the absorbed query: the oracle's fp64 value within the bf16 rounding of the operand
    qa = oracle.mla_absorb(m["q_nope"], m["q_rope"], m["w_uk"])
    assert out_error(q_cat.cpu(), qa, torch.bfloat16) <= TOL
    clean = m["cache"].clone()
    for b, n in enumerate(lengths):
        clean[b, n:] = 0
    ref = oracle.mla_decode_expanded(m["q_nope"], m["q_rope"], clean[..., :512],
                                     clean[..., 512:], np.array(lengths), m["w_uk"], m["w_uv"],
                                     m["gate"], scale=kda.MLA_SCALE)
    assert out_error(out.cpu(), ref, torch.bfloat16) <= TOL


def _latent_ws(m, ws_bytes=None):
    """The latent attention with a split workspace (the size the library asks for, or less)."""
    _gpu.lib()
    B, L = m["cache"].shape[:2]
    need = kda.mla_decode_workspace_size(B, L)
    assert need > 0, "a small batch over a long cache is split"
    n = need if ws_bytes is None else ws_bytes
    ws = torch.empty((n + 3) // 4, dtype=torch.float32, device="cuda")
    z = torch.full((B, 64, 512), 7.0, device="cuda")
    kda.mla_decode_latent(m["q_cat"].cuda(), m["cache"].cuda(), m["lengths"].cuda(), z,
                          workspace=ws)
    torch.cuda.synchronize()
    return z


@pytest.mark.parametrize("q_std", [1.0, 4.0])
def test_split_latent_attention_matches_the_oracle(q_std):
    """A small batch over a long cache: each sequence's positions are split across CTAs whose
    partial sums are merged.  Lengths that leave some splits empty (1, 513) or ragged
    (2049, 4000), and peaked scores (q_std 4) so each split's maximum differs."""
    lengths = [4096, 1, 513, 2049, 4000]
    m = _case(lengths, 4096, seed=840 + int(q_std), q_std=q_std)
    z = _latent_ws(m)
    kda.kda_check_device_error()
    clean = m["cache"].clone()
    for b, n in enumerate(lengths):
        clean[b, n:] = 0
    ref, _ = oracle.mla_latent_attention(m["q_cat"], clean, np.array(lengths),
                                         scale=kda.MLA_SCALE)
    for b in range(len(lengths)):
        e = max_err_rel_rms(z[b], ref[b])
        assert e <= TOL, f"sequence {b} (length {lengths[b]}): {e:.3g}"
    # without a workspace the same call runs one CTA per sequence: same values within rounding
    z1 = _latent(m)
    assert max_err_rel_rms(z1, z.double().cpu()) <= TOL


def test_split_with_a_short_workspace_and_empty_sequences():
    """A workspace for two splits only (the call uses what fits); a sequence of length 0 and
    one with an out-of-range length still give z = 0 through the merge."""
    lengths = [2048, 0, 1500, -3]
    m = _case(lengths, 2048, seed=850)
    two = 2 * 4 * 64 * 514 * 4
    z = _latent_ws(m, ws_bytes=two)
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_check_device_error()
    assert ei.value.status == kda.KDA_ERR_BAD_INDEX
    assert not z[1].any() and not z[3].any()
    clean = m["cache"].clone()
    clean[2, 1500:] = 0
    ref, _ = oracle.mla_latent_attention(m["q_cat"][[0, 2]], clean[[0, 2]],
                                         np.array([2048, 1500]), scale=kda.MLA_SCALE)
    assert max_err_rel_rms(z[[0, 2]], ref) <= TOL


def test_split_mla_decode_matches_the_expanded_oracle():
    """The whole step with a split workspace on two long sequences."""
    lengths = [3000, 4096]
    m = _case(lengths, 4096, seed=860)
    _gpu.lib()
    B = len(lengths)
    ws = torch.empty(kda.mla_decode_workspace_size(B, 4096) // 4, dtype=torch.float32,
                     device="cuda")
    q_cat = torch.empty((B, 64, 576), dtype=torch.bfloat16, device="cuda")
    z = torch.empty((B, 64, 512), device="cuda")
    out = torch.empty((B, 64, 128), dtype=torch.bfloat16, device="cuda")
    c = _gpu.cuda
    kda.mla_decode(c(m["q_nope"]), c(m["q_rope"]), c(m["w_uk"]), c(m["w_uv"]), c(m["cache"]),
                   c(m["lengths"]), c(m["gate"]), q_cat, z, out, workspace=ws)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    clean = m["cache"].clone()
    clean[0, 3000:] = 0
    ref = oracle.mla_decode_expanded(m["q_nope"], m["q_rope"], clean[..., :512],
                                     clean[..., 512:], np.array(lengths), m["w_uk"], m["w_uv"],
                                     m["gate"], scale=kda.MLA_SCALE)
    assert out_error(out.cpu(), ref, torch.bfloat16) <= TOL


@pytest.mark.parametrize("seed", range(12))
def test_latent_attention_random_batches(seed):
    """Seeded random batches: 1-20 sequences, lengths 0..cache length (tile edges, one-position
    tails, empty sequences), cache lengths 64-1,100, peaked or flat scores, and a forced split
    of 1, 2, 3 or 5 CTAs per sequence (the merge of partial sums): every sequence against the
    oracle; an empty sequence gives exactly zero."""
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 21))
    L = int(rng.integers(1, 18)) * 64 + int(rng.integers(0, 2)) * int(rng.integers(1, 64))
    lengths = [int(x) for x in rng.integers(0, L + 1, size=B)]
    lengths[0] = L  # one full cache
    if B > 2:
        lengths[1] = 0
    q_std = float(rng.choice([1.0, 4.0]))
    split = int(rng.choice([1, 2, 3, 5]))
    m = _case(lengths, L, seed=2000 + seed, q_std=q_std)
    _gpu.lib()
    n_ws = 0
    with kda.mla_split(split):
        n_ws = kda.mla_decode_workspace_size(B, L)
        ws = torch.empty(max(n_ws // 4, 1), dtype=torch.float32, device="cuda") if n_ws else None
        z = torch.full((B, 64, 512), 7.0, device="cuda")
        kda.mla_decode_latent(m["q_cat"].cuda(), m["cache"].cuda(), m["lengths"].cuda(), z,
                              workspace=ws)
        torch.cuda.synchronize()
    kda.kda_check_device_error()
    assert torch.isfinite(z).all()
    clean = m["cache"].clone()
    for b, n in enumerate(lengths):
        clean[b, n:] = 0
    ref, _ = oracle.mla_latent_attention(m["q_cat"], clean, np.array(lengths),
                                         scale=kda.MLA_SCALE)
    for b in range(B):
        if lengths[b] == 0:
            assert bool((z[b] == 0).all()), f"sequence {b}: empty, not zero"
            continue
        e = max_err_rel_rms(z[b], ref[b])
        assert e <= TOL, f"seed {seed}, split {split}, sequence {b} (length {lengths[b]}): {e:.3g}"
