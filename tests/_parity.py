"""Error metrics shared by the parity tests.

max_err_rel_rms:       max_i |gpu_i - ref_i| / RMS(ref)        -- the tolerance's own form.
excess_over_half_ulp:  max_i (|gpu_i - ref_i| - ulp_bf16(gpu_i) / 2)+ / RMS(ref)
                       for results stored in bf16.  A bf16 result is the kernel's own value x'
                       rounded to nearest, so |gpu - x'| <= ulp_bf16(gpu) / 2 (rounding never
                       leaves the binade downwards, so the stored value's ulp is the larger);
                       what is left, |x' - ref| >= |gpu - ref| - ulp_bf16(gpu) / 2, is the
                       computation error the observation proves, and that is what the
                       tolerance bounds.  Exact rounding of the exact result passes with 0.
"""
import numpy as np
import torch


def to64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().double().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def rms(x):
    x = to64(x)
    return float(np.sqrt((x * x).mean())) if x.size else 0.0


def max_err_rel_rms(gpu, ref):
    g, r = to64(gpu), to64(ref)
    if r.size == 0:
        return 0.0
    return float(np.abs(g - r).max() / max(rms(r), 1e-300))


def ulp_bf16(x):
    """One bf16 ulp at |x| (8 significant bits); 0 at 0."""
    a = np.abs(to64(x))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 0.0)


def excess_over_half_ulp(gpu, ref):
    g, r = to64(gpu), to64(ref)
    if r.size == 0:
        return 0.0
    ex = np.maximum(np.abs(g - r) - 0.5 * ulp_bf16(g), 0.0)
    return float(ex.max() / max(rms(r), 1e-300))


def out_error(gpu, ref, io_dtype):
    """The output metric used against the tolerance for this output storage type."""
    if io_dtype == torch.bfloat16:
        return excess_over_half_ulp(gpu, ref)
    return max_err_rel_rms(gpu, ref)
