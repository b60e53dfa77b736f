"""Runs the library's entry points on cuda:0 for the tests (marshalling through the binding)."""
import torch

from hybrid_linear_attention_gb300 import build as kbuild
from hybrid_linear_attention_gb300 import kda

_built = False


def lib():
    global _built
    if not _built:
        kbuild.build()
        _built = True
    return kda.load()


def cuda(x):
    return None if x is None else x.to("cuda").contiguous()


def prefill(inp, p, *, gate=False, want_final=True, stream=None):
    """inp: dict from inputs.kda_inputs (any device).  Returns (out, final_state) on cuda."""
    lib()
    q, k, v = cuda(inp["q"]), cuda(inp["k"]), cuda(inp["v"])
    g, beta, cu = cuda(inp["g"]), cuda(inp["beta"]), cuda(inp["cu_seqlens"])
    T, H, d = q.shape
    N = cu.numel() - 1
    init = cuda(inp.get("init_state"))
    out = torch.empty((T, H, d), dtype=p.io_torch, device="cuda")
    fin = torch.empty((N, H, d, d), dtype=p.state_torch, device="cuda") if want_final else None
    ws_n = kda.kda_prefill_workspace_size(p, N, T)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda") if ws_n else None
    kda.kda_prefill(p, q, k, v, g, beta, cu, out, init_state=init, final_state=fin,
                    gate_logit=cuda(inp.get("gate")) if gate else None,
                    norm_w=cuda(inp.get("norm_w")) if gate else None, workspace=ws,
                    stream=stream)
    return out, fin
