"""The tensor-core prefill's precision design, checked on the CPU with a numerical model of
its operand roundings (tests/_kernel_numerics.py) against the fp64 oracle.

Bounds (the workload definition's, in the forms the GPU tests use): bf16-stored output within
1e-2 of RMS beyond half a bf16 ulp, final fp32 state within 1e-3 of RMS.  The model without
rounding is the recurrence itself; with the kernel's roundings (bf16 hi + lo A/P operands on
the band, tf32 elsewhere, hi + lo Y, three-term bf16 state update, the state operand truncated
to tf32) it meets the bounds; with every operand in a single bf16 it does not, which is why
the kernel splits operands at all.
"""
import numpy as np
import pytest

import oracle
from hybrid_linear_attention_gb300 import inputs
from tests._kernel_numerics import prefill_head
from tests._parity import excess_over_half_ulp, max_err_rel_rms

D = 128


def _run(T, H, seed, scheme, *, gate, init=None):
    inp = inputs.kda_inputs([T], H, D, seed=seed, gate=gate, init_state=init)
    s0 = inp.get("init_state")
    ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                             inp["cu_seqlens"], init_state=s0,
                             gate=inp.get("gate") if gate else None,
                             norm_w=inp.get("norm_w") if gate else None)
    eo = es = 0.0
    for h in range(H):
        def f(x):
            return x[:, h].float().numpy()
        out, S = prefill_head(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["g"]),
                              inp["beta"][:, h].numpy(),
                              s0[0, h].numpy() if s0 is not None else np.zeros((D, D)),
                              scheme, gate=f(inp["gate"]) if gate else None)
        ro, rs = ref["out"][:, h], ref["final_state"][0, h]
        eo = max(eo, max_err_rel_rms(out, ro) if scheme == "exact" else excess_over_half_ulp(out, ro))
        es = max(es, max_err_rel_rms(S, rs))
    return eo, es


@pytest.mark.parametrize("gate", [False, True])
def test_model_without_rounding_is_the_recurrence(gate):
    eo, es = _run(192, 1, 5, "exact", gate=gate, init="all")
    assert eo < 1e-10 and es < 1e-10


@pytest.mark.parametrize("scheme", ["kernel", "kernel_1cta"])
@pytest.mark.parametrize("seed", [300, 301, 302])
def test_kernel_roundings_meet_the_bounds(seed, scheme):
    """Both kernel forms (the pair's inverse by distance, the one-CTA form's by halves)."""
    eo, es = _run(512, 2, seed, scheme, gate=False, init="all")
    assert eo <= 1e-2 and es <= 1e-3, (eo, es)
    eo_g, _ = _run(512, 2, seed, scheme, gate=True)
    assert eo_g <= 1e-2, eo_g


def test_inverse_orders_agree():
    """The two block orders of the inverse are the same matrix up to the tf32 rounding of their
    products, and each is (I + A)^-1 to that rounding."""
    from tests import _kernel_numerics as kn
    rng = np.random.default_rng(7)
    k = rng.standard_normal((64, 128))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    A = np.tril(0.5 * (k @ k.T), -1).astype(np.float32)
    exact = np.linalg.inv(np.eye(64) + A.astype(np.float64))
    t_d = kn._inverse(A, kn.SCHEMES["kernel"])
    t_h = kn._inverse(A, kn.SCHEMES["kernel_1cta"])
    scale = np.abs(exact).max()
    assert np.abs(t_d - exact).max() <= 1e-3 * scale
    assert np.abs(t_h - exact).max() <= 1e-3 * scale
    assert np.abs(t_d - t_h).max() <= 1e-3 * scale
    assert np.array_equal(np.triu(t_h, 1), np.zeros_like(t_h))


def test_single_bf16_operands_miss_the_state_bound():
    _, es = _run(512, 2, 300, "all_bf16", gate=False)
    assert es > 1e-3, es


# Each split the kernel pays for is needed: dropping any one of them misses a bound (the
# model's values at these sizes are in the comments; the bounds are 1e-2 and 1e-3).
CHEAPER = [
    # name, change to the kernel's scheme, tokens, metric that fails
    ("lo terms on the own block only", dict(band="own"), 1024, "gated"),      # 1.8e-2
    ("query rows (P) without lo terms", dict(split_q=False), 512, "gated"),   # 4.1e-2
    ("A and P from bf16 hi alone", dict(band=False), 512, "gated"),            # 4.1e-2
    ("Y as one tf32 operand", dict(y_split=False), 512, "state"),              # 2.0e-3
    ("update without u's lo term", dict(upd="bf16x2k"), 512, "state"),         # 2.3e-2
    ("update without Kbar's lo term", dict(upd="bf16x2u"), 512, "state"),      # 1.5e-2
]


@pytest.mark.parametrize("name,change,T,metric", CHEAPER, ids=[c[0] for c in CHEAPER])
def test_every_split_of_the_kernel_is_needed(name, change, T, metric):
    from tests import _kernel_numerics as kn
    key = "cheaper: " + name
    kn.SCHEMES[key] = dict(kn.SCHEMES["kernel"], **change)
    try:
        if metric == "gated":
            err, _ = _run(T, 2, 300, key, gate=True, init="all")
            assert err > 1e-2, err
        else:
            _, err = _run(T, 2, 300, key, gate=False, init="all")
            assert err > 1e-3, err
    finally:
        del kn.SCHEMES[key]


def test_device_fp8_model_differs_from_the_definition_only_at_rounding_boundaries():
    """The tests-side model of the kernels' fp32 quantiser against the oracle's fp64
    definition: the same scales up to fp32 rounding, and codes that differ, if at all, by
    one E4M3 step and only where x / scale lies within fp32 rounding of a code boundary."""
    from tests._kernel_numerics import fp8_quantize_groups_device

    rng = np.random.default_rng(5)
    x = (rng.standard_normal((400, 256)) * np.exp2(rng.uniform(-8, 8, (400, 1)))).astype(np.float32)
    c_ref, s_ref = oracle.fp8_quantize_groups(x, 128)
    c_dev, s_dev = fp8_quantize_groups_device(x, 128)
    np.testing.assert_allclose(s_dev, s_ref, rtol=2 ** -23)
    v_ref = oracle.fp8_e4m3_decode(c_ref)
    v_dev = oracle.fp8_e4m3_decode(c_dev)
    diff = c_ref != c_dev
    assert diff.mean() < 1e-3
    y = np.abs(x.astype(np.float64).reshape(400, 2, 128) / s_ref[..., None]).reshape(400, 256)
    # where they differ, both codes are neighbours of y (one step apart)
    lo, hi = np.minimum(np.abs(v_ref), np.abs(v_dev)), np.maximum(np.abs(v_ref), np.abs(v_dev))
    assert ((lo[diff] <= y[diff] * (1 + 2 ** -20)) & (y[diff] <= hi[diff] * (1 + 2 ** -20))).all()


def test_query_rows_need_the_split_read_of_the_state():
    """The query rows' read of the state: as one tf32 product (the state truncated, Q Gamma
    rounded) one draw of the gated workload misses the bound (model: 1.96e-2, seed 8, four
    heads, T = 1024); as the kernel takes it, three bf16 products of the split state and the
    split Q Gamma, the same draw stays at ~1.3e-3."""
    from tests import _kernel_numerics as kn
    key = "cheaper: one tf32 read"
    kn.SCHEMES[key] = dict(kn.SCHEMES["kernel"], xq=None)
    try:
        err_one, _ = _run(1024, 4, 8, key, gate=True)
    finally:
        del kn.SCHEMES[key]
    err_kernel, _ = _run(1024, 4, 8, "kernel", gate=True)
    assert err_one > 1e-2, err_one
    assert err_kernel < 3e-3, err_kernel
