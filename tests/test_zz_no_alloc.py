"""The no-allocation form of the MLA latent attention (mla_decode_latent_noalloc): the split
partial sums live in a fixed device buffer inside the library, so the call takes no
workspace.  It must give the same bits as mla_decode_latent with a workspace of the size
mla_decode_workspace_size() asks for, and refuse, before launching anything, a split that
would need more than the fixed buffer (KDA_ERR_WORKSPACE).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gb300 import build as kbuild
from hybrid_linear_attention_gb300 import kda
from tests._parity import max_err_rel_rms

STATIC_BYTES = 24 << 20


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load()


def test_exported_and_host_checks(lib):
    """Exported; bad arguments rejected; an oversize split refused on the host."""
    assert hasattr(lib, "mla_decode_latent_noalloc")
    buf = ctypes.c_void_p(256)  # aligned, never dereferenced: every case returns before a launch
    f = lib.mla_decode_latent_noalloc
    assert f(None, None, 0, None, 0, 0.07, None, None) == kda.KDA_OK
    assert f(None, buf, 64, buf, 2, 0.07, buf, None) == kda.KDA_ERR_INVALID_ARG
    assert f(buf, buf, 64, buf, 2, 0.0, buf, None) == kda.KDA_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(24), buf, 64, buf, 2, 0.07, buf, None) == kda.KDA_ERR_INVALID_ARG
    with kda.mla_split(64):  # 64 splits x 16 sequences: 135 MB of partials
        assert kda.mla_decode_workspace_size(16, 65536) > STATIC_BYTES
        assert f(buf, buf, 65536, buf, 16, 0.07, buf, None) == kda.KDA_ERR_WORKSPACE
    with kda.mla_split(2):  # 2 x 16 sequences fit
        assert 0 < kda.mla_decode_workspace_size(16, 65536) <= STATIC_BYTES


def _case(lengths, L, seed):
    g = torch.Generator().manual_seed(seed)
    B = len(lengths)
    cache = torch.randn(B, L, 576, generator=g).to(torch.bfloat16)
    for b, n in enumerate(lengths):
        cache[b, n:] = float("nan")
    q = torch.randn(B, 64, 576, generator=g).to(torch.bfloat16)
    return q, cache, torch.tensor(lengths, dtype=torch.int32)


@pytest.mark.gpu
@pytest.mark.parametrize("lengths,L", [([4096, 1, 2500, 4000], 4096),  # split 8 ways
                                       ([300] * 200, 320)])             # one CTA per sequence
def test_noalloc_equals_the_workspace_call(lengths, L):
    from tests import _gpu
    _gpu.lib()
    q, cache, lens = _case(lengths, L, seed=900 + L)
    qc, cc, lc = q.cuda(), cache.cuda(), lens.cuda()
    B = len(lengths)
    n = kda.mla_decode_workspace_size(B, L)
    assert n <= STATIC_BYTES
    ws = torch.empty(max(n // 4, 1), dtype=torch.float32, device="cuda")
    z_ws = torch.full((B, 64, 512), 7.0, device="cuda")
    z_na = torch.full((B, 64, 512), 5.0, device="cuda")
    kda.mla_decode_latent(qc, cc, lc, z_ws, workspace=ws if n else None)
    kda.mla_decode_latent_noalloc(qc, cc, lc, z_na)
    kda.mla_decode_latent_noalloc(qc, cc, lc, z_na)  # the buffer is reused call after call
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    assert torch.equal(z_na, z_ws)
    clean = cache.clone()
    for b, m in enumerate(lengths):
        clean[b, m:] = 0
    pick = [0, 1, B - 1]
    ref, _ = oracle.mla_latent_attention(q[pick], clean[pick], np.array(lengths)[pick],
                                         scale=kda.MLA_SCALE)
    assert max_err_rel_rms(z_na[pick], ref) <= 1e-2


@pytest.mark.gpu
def test_noalloc_refuses_oversize_without_launching():
    from tests import _gpu
    _gpu.lib()
    q, cache, lens = _case([64] * 8, 64, seed=950)
    z = torch.full((8, 64, 512), 3.0, device="cuda")
    with kda.mla_split(64), pytest.raises(kda.KdaError) as ei:  # 64 x 8: 67 MB of partials
        kda.mla_decode_latent_noalloc(q.cuda(), cache.cuda(), lens.cuda(), z)
    assert ei.value.status == kda.KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((z == 3.0).all())
