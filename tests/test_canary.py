"""The guard-band helper itself, on the CPU: a view into a guarded buffer has the requested
shape, dtype and 16-byte alignment, and a write past its end is caught."""
import pytest
import torch

from tests import _canary


def test_guarded_view_and_overwrite_detection(monkeypatch):
    reg = _canary.Registry()
    t = _canary._guarded_alloc(reg, (3, 5), torch.bfloat16, "cpu")
    assert t.shape == (3, 5) and t.dtype == torch.bfloat16 and t.is_contiguous()
    assert t.data_ptr() % 16 == 0
    t.fill_(1.0)
    reg.check()                                  # in-bounds writes leave the bands alone
    t2 = _canary._guarded_alloc(reg, (4,), torch.float32, "cpu")
    buf = reg.bufs[-1][0]
    buf[_canary.GUARD + 16] = 0                  # one byte past the 16-byte tensor
    with pytest.raises(AssertionError, match="guard band"):
        reg.check()
    empty = _canary._guarded_alloc(reg, (0, 7), torch.float32, "cpu")
    assert empty.numel() == 0 and empty.shape == (0, 7)
    del t2
