"""Multi-token decode (a speculative draft of K tokens per sequence, the state after every
token kept for rollback) and the commit of the accepted steps, against the oracle run on
each prefix of the draft; plus the device-side index checks of the decode paths."""
import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gb300 import inputs, kda
from tests import _gpu
from tests._parity import max_err_rel_rms, out_error

pytestmark = pytest.mark.gpu

H, D = 4, 128


def _draft(n_seqs, K, n_slots, seed):
    rows = n_seqs * K
    return {
        "q": inputs.normal((rows, H, D), seed=seed, device="cuda"),
        "k": inputs.normal((rows, H, D), seed=seed + 1, device="cuda"),
        "v": inputs.normal((rows, H, D), seed=seed + 2, device="cuda"),
        "g": inputs.uniform((rows, H, D), -5.0, 0.0, seed=seed + 3, device="cuda"),
        "beta": inputs.beta_draw((rows, H), seed=seed + 4, device="cuda"),
        "pool": inputs.normal((n_slots, H, D, D), seed=seed + 5, device="cuda",
                              dtype=torch.float32, std=0.02),
    }


def _oracle_prefixes(d, n, K, slot):
    """Outputs of the K tokens and the state after each prefix, from the pool state."""
    sl = slice(n * K, (n + 1) * K)
    init = d["pool"][slot:slot + 1].cpu()
    outs, states = None, []
    for L in range(1, K + 1):
        s2 = slice(n * K, n * K + L)
        r = oracle.kda_forward(d["q"][s2].cpu(), d["k"][s2].cpu(), d["v"][s2].cpu(),
                               d["g"][s2].cpu(), d["beta"][s2].cpu(),
                               np.array([0, L], np.int32), init_state=init)
        states.append(r["final_state"][0])
        if L == K:
            outs = r["out"]
    return outs, states


@pytest.mark.parametrize("K", [1, 3, 9])
def test_decode_multi_matches_oracle_prefixes(K):
    n_seqs, n_slots = 5, 8
    d = _draft(n_seqs, K, n_slots, seed=700 + K)
    p = kda.params(H=H, d=D)
    _gpu.lib()
    slot = torch.tensor([6, 0, 3, 7, 1], dtype=torch.int32, device="cuda")
    pool0 = d["pool"].clone()
    out = torch.empty((n_seqs * K, H, D), dtype=torch.bfloat16, device="cuda")
    steps = torch.empty((n_seqs * K, H, D, D), dtype=torch.float32, device="cuda")
    kda.kda_decode_multi(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["pool"], out, K,
                         slot_idx=slot, step_states=steps, commit_final=True)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    used = set(slot.tolist())
    for n, s in enumerate(slot.tolist()):
        ro, rs = _oracle_prefixes({**d, "pool": pool0}, n, K, s)
        assert out_error(out[n * K:(n + 1) * K].cpu(), ro, torch.bfloat16) <= 1e-2
        for i in range(K):
            assert max_err_rel_rms(steps[n * K + i].cpu(), rs[i]) <= 1e-3
        # the committed pool state is the last step's state, bit for bit
        assert torch.equal(d["pool"][s], steps[n * K + K - 1])
    for s in range(n_slots):  # slots nobody uses are untouched
        if s not in used:
            assert torch.equal(d["pool"][s], pool0[s])


def test_decode_multi_with_one_token_is_decode_step():
    n_seqs, n_slots = 6, 6
    d = _draft(n_seqs, 1, n_slots, seed=760)
    p = kda.params(H=H, d=D)
    _gpu.lib()
    pool_a, pool_b = d["pool"].clone(), d["pool"].clone()
    out_a = torch.empty((n_seqs, H, D), dtype=torch.bfloat16, device="cuda")
    out_b = torch.empty_like(out_a)
    kda.kda_decode_step(p, d["q"], d["k"], d["v"], d["g"], d["beta"], pool_a, out_a)
    kda.kda_decode_multi(p, d["q"], d["k"], d["v"], d["g"], d["beta"], pool_b, out_b, 1,
                         commit_final=True)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(pool_a, pool_b)


def test_state_accept_commits_the_accepted_step():
    n_seqs, K, n_slots = 5, 4, 7
    d = _draft(n_seqs, K, n_slots, seed=780)
    p = kda.params(H=H, d=D)
    _gpu.lib()
    slot = torch.tensor([2, 5, 0, 6, 3], dtype=torch.int32, device="cuda")
    pool0 = d["pool"].clone()
    out = torch.empty((n_seqs * K, H, D), dtype=torch.bfloat16, device="cuda")
    steps = torch.empty((n_seqs * K, H, D, D), dtype=torch.float32, device="cuda")
    kda.kda_decode_multi(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["pool"], out, K,
                         slot_idx=slot, step_states=steps, commit_final=False)
    torch.cuda.synchronize()
    assert torch.equal(d["pool"], pool0)  # nothing committed yet
    acc = torch.tensor([0, 1, 4, 2, 3], dtype=torch.int32, device="cuda")
    kda.kda_state_accept(p, steps, acc, d["pool"], K, slot_idx=slot)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    for n, (s, a) in enumerate(zip(slot.tolist(), acc.tolist())):
        want = pool0[s] if a == 0 else steps[n * K + a - 1]
        assert torch.equal(d["pool"][s], want)
    # and the accepted state is the oracle's state after that many draft tokens
    ro, rs = _oracle_prefixes({**d, "pool": pool0}, 3, K, 6)
    assert max_err_rel_rms(d["pool"][6].cpu(), rs[1]) <= 1e-3


def test_out_of_range_indices_are_flagged_not_followed():
    """A slot outside the pool (and an accept length outside 0..K) is skipped by the kernels'
    own bounds checks and reported; the other sequences are still served."""
    n_seqs, K, n_slots = 3, 2, 4
    d = _draft(n_seqs, K, n_slots, seed=790)
    p = kda.params(H=H, d=D)
    _gpu.lib()
    pool0 = d["pool"].clone()
    slot = torch.tensor([1, 9, 2], dtype=torch.int32, device="cuda")  # 9 is outside the pool
    out = torch.zeros((n_seqs * K, H, D), dtype=torch.bfloat16, device="cuda")
    kda.kda_decode_multi(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["pool"], out, K,
                         slot_idx=slot, commit_final=True)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_check_device_error()
    assert e.value.status == -6
    assert torch.equal(d["pool"][0], pool0[0]) and torch.equal(d["pool"][3], pool0[3])
    assert not torch.equal(d["pool"][1], pool0[1]) and not torch.equal(d["pool"][2], pool0[2])
    assert torch.count_nonzero(out[2:4].float()) == 0  # sequence 1 skipped
    steps = torch.zeros((n_seqs * K, H, D, D), dtype=torch.float32, device="cuda")
    acc = torch.tensor([1, 0, 5], dtype=torch.int32, device="cuda")  # 5 > K
    kda.kda_state_accept(p, steps, acc, d["pool"], K)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_check_device_error()
    assert e.value.status == -6
    kda.kda_check_device_error()  # the flag was cleared
