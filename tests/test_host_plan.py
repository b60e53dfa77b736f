"""Host logic of kda_prefill_host (no GPU): the segments it cuts a packed batch into.

Bit-exactness with one kda_prefill over the whole batch rests on these properties, checked
here on seeded random batches through the C ABI's plan query: the segments tile [0, T) in
order, none holds more than the segment size, and every inner boundary lies a multiple of 64
tokens after the start of the sequence it falls in (so each sequence is cut only at one of its
own chunk edges); the last two segment sizes of rows are cut in halves.
"""
import bisect

import numpy as np
import pytest
import torch

from hybrid_linear_attention_gb300 import build as kbuild
from hybrid_linear_attention_gb300 import kda


@pytest.fixture(scope="module", autouse=True)
def lib():
    kbuild.build()
    return kda.load()


def _cu(lengths):
    return torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)


def _check(lengths, S):
    cu = _cu(lengths)
    T = int(cu[-1])
    b = kda.kda_prefill_host_plan(cu, S)
    assert b[0] == 0 and b[-1] == T
    assert all(x < y for x, y in zip(b, b[1:]))
    assert all(y - x <= S for x, y in zip(b, b[1:]))
    cl = cu.tolist()
    for r in b[1:-1]:
        n = bisect.bisect_right(cl, r) - 1  # the sequence holding row r
        assert cl[n] < r < cl[n + 1] or r == cl[n]
        assert (r - cl[n]) % 64 == 0
    return b


def test_single_sequence_halves_its_last_rows():
    assert _check([4096], 512) == [0, 512, 1024, 1536, 2048, 2560, 3072, 3584, 3840, 3968,
                                   4032, 4096]
    assert _check([1000], 256)[-1] == 1000
    assert _check([64], 64) == [0, 64]
    assert _check([3], 64) == [0, 3]


def test_random_packed_batches():
    rng = np.random.default_rng(7)
    for _ in range(300):
        n = int(rng.integers(1, 14))
        pick = [0, 0, 1, 2, 3, 63, 64, 65, 127, 128, 129]
        lens = [int(rng.choice(pick)) if rng.random() < 0.6 else int(rng.integers(0, 900))
                for _ in range(n)]
        _check(lens, 64 * int(rng.integers(1, 10)))


def test_empty_batch_and_bad_offsets():
    assert kda.kda_prefill_host_plan(_cu([0, 0]), 64) == [0]
    lib = kda.load()
    bad = (np.array([0, 70, 60], dtype=np.int32), np.array([1, 5, 9], dtype=np.int32))
    for cu in bad:
        assert lib.kda_prefill_host_plan(cu.ctypes.data, 2, int(cu[-1]), 64, None, 0) == -1
    good = np.array([0, 70, 130], dtype=np.int32)
    assert lib.kda_prefill_host_plan(good.ctypes.data, 2, 130, 96, None, 0) == -1  # not 64k
    assert lib.kda_prefill_host_plan(good.ctypes.data, 2, 131, 64, None, 0) == -1  # T mismatch
    assert lib.kda_prefill_host_plan(good.ctypes.data, 2, 130, 64, None, 0) > 0
