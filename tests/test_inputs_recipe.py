"""The seeded input recipe (no GPU): the synthetic workloads have the distributions and shapes
the workload definitions give, and the same seed gives the same arrays.

Workloads: q, k, v ~ N(0, 1); per-channel log-retention ~ U(-5, 0); beta = sigmoid(N(0, 1))
per head-token; initial states ~ N(0, 0.02), on every sequence or on the even-indexed ones;
packed variable-length batch of 32 lengths log-uniform in [512, 65536] re-drawn until the
total lies in [450K, 550K].
"""
import math

import numpy as np
import torch

from hybrid_linear_attention_gb300 import inputs


def test_same_seed_same_arrays_different_seed_different_arrays():
    a = inputs.kda_inputs([70, 5], 2, 16, seed=3, init_state="even", gate=True)
    b = inputs.kda_inputs([70, 5], 2, 16, seed=3, init_state="even", gate=True)
    c = inputs.kda_inputs([70, 5], 2, 16, seed=4, init_state="even", gate=True)
    for key in a:
        assert torch.equal(a[key], b[key]), key
    assert not torch.equal(a["q"], c["q"])


def test_distributions_of_the_prefill_workload():
    inp = inputs.kda_inputs([4096], 8, 128, seed=0, init_state="all")
    q = inp["q"].float()
    assert q.dtype == torch.float32 and inp["q"].dtype == torch.bfloat16
    assert abs(float(q.mean())) < 0.01 and abs(float(q.std()) - 1.0) < 0.01
    g = inp["g"]
    assert g.dtype == torch.float32 and float(g.min()) >= -5.0 and float(g.max()) <= 0.0
    assert abs(float(g.mean()) + 2.5) < 0.01                       # U(-5, 0)
    assert abs(float(g.var()) - 25.0 / 12.0) < 0.02
    beta = inp["beta"].double()
    z = torch.log(beta / (1 - beta))                                # logit -> N(0, 1)
    assert abs(float(z.mean())) < 0.03 and abs(float(z.std()) - 1.0) < 0.03
    s0 = inp["init_state"]
    assert abs(float(s0.std()) - 0.02) < 2e-4
    assert tuple(s0.shape) == (1, 8, 128, 128)


def test_even_sequences_continue_from_a_state_odd_ones_start_from_zero():
    inp = inputs.kda_inputs([3, 4, 5, 6], 2, 16, seed=1, init_state="even")
    s0 = inp["init_state"]
    assert all(float(s0[n].abs().sum()) > 0 for n in (0, 2))
    assert all(float(s0[n].abs().sum()) == 0 for n in (1, 3))


def test_varlen_batch_recipe():
    lens, seed = inputs.varlen_lengths(n_seqs=32, seed=0)
    assert len(lens) == 32 and all(512 <= L <= 65536 for L in lens)
    assert 450_000 <= sum(lens) <= 550_000
    assert inputs.varlen_lengths(n_seqs=32, seed=0) == (lens, seed)
    # log-uniform: the mean log-length over ten accepted batches sits near the middle of
    # [ln 512, ln 65536] (the total's window pulls it up a little)
    logs = [np.log(inputs.varlen_lengths(n_seqs=32, seed=s)[0]).mean() for s in range(0, 200, 20)]
    mid = (math.log(512) + math.log(65536)) / 2
    assert abs(float(np.mean(logs)) - mid) < 0.3
    cu = inputs.cu_seqlens_from_lengths(lens)
    assert cu.dtype == torch.int32 and int(cu[0]) == 0 and int(cu[-1]) == sum(lens)
    assert torch.all(cu[1:] - cu[:-1] == torch.tensor(lens, dtype=torch.int32))


def test_prologue_and_decode_draws():
    pin = inputs.prologue_inputs([100, 28], 2, 128, seed=2)
    assert tuple(pin["x"].shape) == (128, 3 * 2 * 128)
    assert tuple(pin["conv_w"].shape) == (3 * 2 * 128, 4)
    assert abs(float(pin["conv_w"].float().std()) - 0.5) < 0.02
    assert tuple(pin["conv_state"].shape) == (2, 3, 3 * 2 * 128)
    dec = inputs.decode_inputs(256, 4, 128, seed=3, gate=True)
    assert tuple(dec["x"].shape) == (256, 3 * 4 * 128)
    assert tuple(dec["g"].shape) == (256, 4, 128) and float(dec["g"].min()) >= -5.0
    assert tuple(dec["beta"].shape) == (256, 4) and tuple(dec["gate"].shape) == (256, 4, 128)
