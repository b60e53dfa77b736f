"""GPU tests of kda_prefill_host: the prologue + prefill of a batch held in host memory,
streamed through the GPU in chunk-aligned token segments.

Each sequence is chunked as one kda_prefill over the whole batch chunks it, and a cut
sequence's fp32 state and conv tail are carried on the device.  So the outputs, final states
and conv tails must be the same bits as the device path (kda_prologue, then one kda_prefill)
on device copies of the same inputs, whenever both runs take the same kernel form (here:
few sequences x heads, the cluster-pair form on both sides).  One case is also checked
against the fp64 oracle, and the conv tails bit-exactly against the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gb300 import inputs, kda
from tests import _gpu
from tests._parity import max_err_rel_rms, out_error

pytestmark = pytest.mark.gpu


def _case(lengths, H, d, io, *, seed, init, conv, gate):
    pin = inputs.prologue_inputs(lengths, H, d, seed=seed, io_dtype=io, conv_state=conv)
    extra = inputs.kda_inputs(lengths, H, d, seed=seed, io_dtype=io,
                              init_state="even" if init else None, gate=gate)
    if gate:
        extra["norm_w"] = inputs.normal((d,), seed=seed * 32 + 17, dtype=torch.float32,
                                        std=0.5) + 1.0
    return pin, extra


def _device_path(p, pin, extra, gate):
    """kda_prologue (conv tail in place, beta = sigmoid) then one kda_prefill on device copies."""
    c = _gpu.cuda
    T = pin["x"].shape[0]
    N = pin["cu_seqlens"].numel() - 1
    H, d = p.H, p.d_k
    io = p.io_torch
    cs = c(pin.get("conv_state"))
    q = torch.empty((T, H, d), dtype=io, device="cuda")
    k, v = torch.empty_like(q), torch.empty_like(q)
    beta = torch.empty((T, H), dtype=torch.float32, device="cuda")
    cu = c(pin["cu_seqlens"])
    kda.kda_prologue(p, c(pin["x"]), c(pin["conv_w"]), cs, cu, q, k, v,
                     beta_logit=c(pin["beta_logit"]), beta=beta)
    out = torch.empty_like(q)
    fin = torch.empty((N, H, d, d), dtype=torch.float32, device="cuda")
    kda.kda_prefill(p, q, k, v, c(pin["g_raw"]), beta, cu, out,
                    init_state=c(extra.get("init_state")), final_state=fin,
                    gate_logit=c(extra["gate"]) if gate else None,
                    norm_w=c(extra["norm_w"]) if gate else None)
    torch.cuda.synchronize()
    kda.kda_check_device_error()
    return out.cpu(), fin.cpu(), None if cs is None else cs.cpu()


def _pinned(t):
    return None if t is None else t.contiguous().pin_memory()


def _host_path(p, pin, extra, gate, seg, stream=None):
    _gpu.lib()
    T = pin["x"].shape[0]
    N = pin["cu_seqlens"].numel() - 1
    H, d = p.H, p.d_k
    io = p.io_torch
    cs = _pinned(pin.get("conv_state"))
    out = torch.empty((T, H, d), dtype=io).pin_memory()
    fin = torch.empty((N, H, d, d), dtype=torch.float32).pin_memory()
    ws = torch.empty(kda.kda_prefill_host_workspace_size(p, N, seg, with_gate=gate),
                     dtype=torch.uint8, device="cuda")
    ws.fill_(0xA5)  # the call must not depend on what the workspace held
    if stream is not None:  # the device buffers above were written on the current stream
        stream.wait_stream(torch.cuda.current_stream())
    kda.kda_prefill_host(p, _pinned(pin["x"]), _gpu.cuda(pin["conv_w"]), cs,
                         pin["cu_seqlens"].cpu().contiguous(), _pinned(pin["beta_logit"]),
                         _pinned(pin["g_raw"]), out, workspace=ws, segment_tokens=seg,
                         init_state=_pinned(extra.get("init_state")), final_state=fin,
                         gate_logit=_pinned(extra["gate"]) if gate else None,
                         norm_w=_gpu.cuda(extra["norm_w"]) if gate else None, stream=stream)
    kda.kda_check_device_error(stream)
    return out, fin, cs


CASES = [
    # lengths, H, d, io, segment, init, conv, gate
    ([1000], 4, 128, torch.bfloat16, 256, False, False, False),
    ([0, 1, 130, 64, 700, 0, 65, 300, 2], 4, 128, torch.bfloat16, 192, True, True, True),
    ([3, 517, 64, 129], 2, 128, torch.bfloat16, 64, True, True, False),
    ([0, 5, 200, 64, 129], 2, 16, torch.float32, 64, True, True, True),
    ([0, 5, 200, 64, 129], 2, 16, torch.bfloat16, 128, True, True, False),
]


@pytest.mark.parametrize("lengths,H,d,io,seg,init,conv,gate", CASES)
def test_host_stream_equals_the_device_path_bitwise(lengths, H, d, io, seg, init, conv, gate):
    p = kda.params(H=H, d=d, io_dtype=io)
    pin, extra = _case(lengths, H, d, io, seed=40 + len(lengths), init=init, conv=conv,
                       gate=gate)
    ref_out, ref_fin, ref_cs = _device_path(p, pin, extra, gate)
    out, fin, cs = _host_path(p, pin, extra, gate, seg)
    assert torch.equal(out, ref_out)
    assert torch.equal(fin, ref_fin)
    if conv:
        assert torch.equal(cs, ref_cs)
    # a second call over the same buffers (workspace and copy streams reused) is unchanged
    out2, fin2, _ = _host_path(p, pin, extra, gate, seg)
    assert torch.equal(out2, ref_out) and torch.equal(fin2, ref_fin)


def test_host_stream_matches_the_oracle_and_its_conv_tails():
    lengths, H, d = [0, 70, 300, 1, 191], 2, 128
    io = torch.bfloat16
    p = kda.params(H=H, d=d, io_dtype=io)
    pin, extra = _case(lengths, H, d, io, seed=77, init=True, conv=True, gate=True)
    out, fin, cs = _host_path(p, pin, extra, True, 128, stream=torch.cuda.Stream())
    T = pin["x"].shape[0]
    pr = oracle.prologue(pin["x"], pin["conv_w"], pin["cu_seqlens"], H, d,
                         conv_state=pin["conv_state"], beta_logit=pin["beta_logit"])
    # q, k, v are stored in bf16 between the two kernels, as the oracle's fp64 y rounded to
    # nearest even; the recurrence then normalises q, k and clamps the raw log-retention
    y = torch.from_numpy(pr["y"].reshape(T, 3, H, d)).to(io)
    ref = oracle.kda_forward(y[:, 0], y[:, 1], y[:, 2], pin["g_raw"],
                             pr["beta"].astype(np.float32), pin["cu_seqlens"],
                             init_state=extra["init_state"], gate=extra["gate"],
                             norm_w=extra["norm_w"], qk_l2norm=True)
    assert out_error(out, ref["out"], io) <= 1e-2
    assert max_err_rel_rms(fin, ref["final_state"]) <= 1e-3
    assert np.array_equal(cs.view(torch.int16).numpy().view(np.uint16),
                          np.asarray(pr["conv_state"]).view(np.uint16))


def test_host_stream_with_no_tokens_returns_the_initial_states():
    H, d = 2, 16
    p = kda.params(H=H, d=d, io_dtype=torch.float32)
    pin, extra = _case([0, 0], H, d, torch.float32, seed=5, init=True, conv=True, gate=False)
    out, fin, cs = _host_path(p, pin, extra, False, 64)
    assert out.numel() == 0
    assert torch.equal(fin, extra["init_state"])
    assert torch.equal(cs, pin["conv_state"])
