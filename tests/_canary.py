"""Guard bands around the device buffers a GPU test allocates (a host-side stand-in for a
memory checker): while a test marked gpu runs, torch.empty / empty_like / zeros / full on a
CUDA device return a view into a larger byte buffer whose 256-byte bands before and after the
tensor hold a fixed pattern.  After the test the bands are compared with the pattern; a write
outside a tensor's bounds into either band fails the test.  The view starts 256 bytes into
its buffer, so the 16-byte alignment the library requires is kept.
"""
import contextlib

import torch

GUARD = 256
PATTERN = 0xA5
# the allocators as torch defines them (the guarded versions below must not call themselves)
_EMPTY, _EMPTY_LIKE, _ZEROS, _FULL = torch.empty, torch.empty_like, torch.zeros, torch.full


class Registry:
    def __init__(self):
        self.bufs = []

    def check(self):
        if not self.bufs:
            return
        if any(buf.is_cuda for buf, _ in self.bufs):
            torch.cuda.synchronize()
        bad = []
        for buf, what in self.bufs:
            head = buf[:GUARD]
            tail = buf[buf.numel() - GUARD:]
            if not (bool((head == PATTERN).all()) and bool((tail == PATTERN).all())):
                bad.append(what)
        self.bufs.clear()
        assert not bad, f"guard band overwritten around: {bad}"


def _is_cuda(device):
    if device is None:
        return False
    return torch.device(device).type == "cuda"


def _guarded_alloc(reg, shape, dtype, device):
    dtype = dtype or torch.get_default_dtype()
    shape = tuple(int(s) for s in shape)
    n = 1
    for s in shape:
        n *= s
    nbytes = n * _EMPTY((), dtype=dtype).element_size()
    buf = _FULL((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=device)
    t = buf[GUARD:GUARD + nbytes].view(dtype).view(shape)
    reg.bufs.append((buf, f"{dtype} {list(shape)}"))
    return t


def _shape(args, kw):
    if "size" in kw:
        s = kw.pop("size")
        return tuple(s) if isinstance(s, (tuple, list, torch.Size)) else (s,)
    if len(args) == 1 and isinstance(args[0], (tuple, list, torch.Size)):
        return tuple(args[0])
    return tuple(args)


@contextlib.contextmanager
def guarded(monkeypatch):
    reg = Registry()
    orig_empty, orig_empty_like, orig_zeros, orig_full = _EMPTY, _EMPTY_LIKE, _ZEROS, _FULL
    plain = {"dtype", "device"}

    def empty(*args, **kw):
        if _is_cuda(kw.get("device")) and set(kw) <= plain | {"size"}:
            kw = dict(kw)
            return _guarded_alloc(reg, _shape(args, kw), kw.get("dtype"), kw["device"])
        return orig_empty(*args, **kw)

    def zeros(*args, **kw):
        if _is_cuda(kw.get("device")) and set(kw) <= plain | {"size"}:
            kw = dict(kw)
            return _guarded_alloc(reg, _shape(args, kw), kw.get("dtype"), kw["device"]).zero_()
        return orig_zeros(*args, **kw)

    def full(size, fill_value, **kw):
        if _is_cuda(kw.get("device")) and set(kw) <= plain:
            t = _guarded_alloc(reg, tuple(size), kw.get("dtype"), kw["device"])
            return t.fill_(fill_value)
        return orig_full(size, fill_value, **kw)

    def empty_like(x, **kw):
        dev = kw.get("device", x.device)
        if (_is_cuda(dev) and set(kw) <= plain and x.is_contiguous()
                and x.layout == torch.strided):
            return _guarded_alloc(reg, x.shape, kw.get("dtype", x.dtype), dev)
        return orig_empty_like(x, **kw)

    monkeypatch.setattr(torch, "empty", empty)
    monkeypatch.setattr(torch, "zeros", zeros)
    monkeypatch.setattr(torch, "full", full)
    monkeypatch.setattr(torch, "empty_like", empty_like)
    try:
        yield reg
    finally:
        monkeypatch.setattr(torch, "empty", orig_empty)
        monkeypatch.setattr(torch, "zeros", orig_zeros)
        monkeypatch.setattr(torch, "full", orig_full)
        monkeypatch.setattr(torch, "empty_like", orig_empty_like)
