"""A numerical model of the tensor-core prefill's precision design, in numpy (tests only).

The chunk algebra is the one in tests/_chunk_form.py; what this model adds is where the
tensor-core kernel rounds.  Each dense product of the kernel takes its operands in a narrow
type, so the model rounds each operand exactly there and accumulates in fp32:

  * A = K~ K^T and P = Q~ K^T (bf16 tensor-core product): rows relative to their own 16-token
    block, K~_r = k_r 2^(gam_r - gam_R0), Q~_r likewise, columns K^_s = k_s 2^(gam_R0 - gam_s)
    times the decay between block starts; operands split into bf16 hi + lo, with hi*hi over
    every column and hi*lo + lo*hi over the band (the row's own block and the one before);
  * T = (I + A)^-1: diagonal 16 x 16 blocks in fp32, off-diagonal blocks from tf32 products;
    T and P' stored as tf32 (round half away, as the kernel rounds on the bit pattern);
  * X = [K Gamma; Q Gamma] S as three bf16 products (hi*hi + hi*lo + lo*hi) of [K Gamma;
    Q Gamma] and of the state, both split into bf16 hi + lo (~2^-16): the query rows' read
    can nearly cancel against P u, and one product serves both row sets;
  * u = T Y with Y = beta (V - K Gamma S) split into tf32 hi + lo; O = X_q + P' tf32(u);
  * S <- Gamma_C S + Kbar^T u as three bf16 products (hi*hi + hi*lo + lo*hi).

The "exact" scheme rounds nothing and computes in fp64, and must reproduce the oracle; the
"all_bf16" scheme puts every operand in one bf16 (no hi/lo splits, no tf32), the cheapest
design the tensor cores allow, for comparison.
"""
import numpy as np

LOG2E = 1.4426950408889634


def bf16(x):
    """fp32 -> bf16 value, round to nearest even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def tf32(x):
    """fp32 -> tf32 value, round half away from zero on the bit pattern."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((b + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def tf32_trunc(x):
    """fp32 -> tf32 value by dropping the low 13 mantissa bits (the state operand)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (b & np.uint32(0xFFFFE000)).view(np.float32)


def _ident(x):
    return x


SCHEMES = {
    # band: True = hi*lo + lo*hi on the row's own block and the one before; "own" = its own
    # block only; "all" = every block.  split_q False: the query rows (P) take hi*hi only
    "kernel": dict(dt=np.float32, split_ap=True, band=True, p=tf32, inv=tf32, t=tf32,
                   x=tf32, s=tf32_trunc, xq="bf16x3", xk="bf16x3", y_split=True, y=tf32,
                   u=tf32, upd="bf16x3"),
    # the one-CTA form: the same roundings, the inverse's off-diagonal blocks by halves
    "kernel_1cta": dict(dt=np.float32, split_ap=True, band=True, p=tf32, inv=tf32, t=tf32,
                        x=tf32, s=tf32_trunc, xq="bf16x3", xk="bf16x3", y_split=True, y=tf32,
                        u=tf32, upd="bf16x3", inv_form="halves"),
    "all_bf16": dict(dt=np.float32, split_ap=False, band=False, p=bf16, inv=bf16, t=bf16,
                     x=bf16, s=bf16, y_split=False, y=bf16, u=bf16, upd="bf16"),
    "exact": dict(dt=np.float64, split_ap=False, band=False, p=_ident, inv=_ident, t=_ident,
                  x=_ident, s=_ident, y_split=False, y=_ident, u=_ident, upd="exact"),
}


def _prod(a, b, sc, band):
    """a @ b.T with the A/P product's operand splits."""
    if sc["dt"] == np.float64:
        return a @ b.T
    if not sc["split_ap"]:
        return bf16(a) @ bf16(b).T
    ah, bh = bf16(a), bf16(b)
    r = ah @ bh.T
    if band:
        al, bl = bf16(a - ah), bf16(b - bh)
        r = r + ah @ bl.T + al @ bh.T
    return r


def _inverse(A, sc):
    """(I + A)^-1 by 16 x 16 blocks: diagonal blocks exact in the working type, off-diagonal
    blocks from products of rounded operands, in one of the kernel's two orders:
    "distance" (the cluster pair's producer): block (R, S) = -T_RR sum_Q A_RQ T_QS by distance
    R - S; "halves" (the one-CTA form): a 2 x 2 block inverse of the 32 x 32 halves, whose
    diagonal halves are 2 x 2 block inverses of their 16 x 16 blocks."""
    dt, rnd = sc["dt"], sc["inv"]
    n = A.shape[0]
    T = np.zeros_like(A)
    blk = [slice(16 * R, 16 * R + 16) for R in range(n // 16)]
    for b in blk:
        T[b, b] = np.linalg.inv(np.eye(16) + A[b, b].astype(np.float64)).astype(dt)
    if sc.get("inv_form", "distance") == "halves":
        assert n == 64
        for R in (1, 3):  # T_R,R-1 = -T_RR (A_R,R-1 T_R-1,R-1)
            M = rnd(A[blk[R], blk[R - 1]]) @ rnd(T[blk[R - 1], blk[R - 1]])
            T[blk[R], blk[R - 1]] = -(rnd(T[blk[R], blk[R]]) @ rnd(M))
        X = {}
        for R in (2, 3):  # X_RS = sum_{Q = S..1} A_RQ T_QS
            for S_ in (0, 1):
                M = np.zeros((16, 16), dtype=dt)
                for Q in range(S_, 2):
                    M = M + rnd(A[blk[R], blk[Q]]) @ rnd(T[blk[Q], blk[S_]])
                X[R, S_] = M
        for R in (2, 3):  # T_RS = -sum_{Q = 2..R} T_RQ X_QS
            for S_ in (0, 1):
                M = np.zeros((16, 16), dtype=dt)
                for Q in range(2, R + 1):
                    M = M + rnd(T[blk[R], blk[Q]]) @ rnd(X[Q, S_])
                T[blk[R], blk[S_]] = -M
        return T
    for dist in range(1, n // 16):
        for R in range(dist, n // 16):
            S_ = R - dist
            rb, sb = blk[R], blk[S_]
            M = np.zeros((16, 16), dtype=dt)
            for Q in range(S_, R):
                M = M + rnd(A[rb, blk[Q]]) @ rnd(T[blk[Q], sb])
            T[rb, sb] = -(rnd(T[rb, rb]) @ rnd(M))
    return T


def prefill_head(q, k, v, g, beta, S0, scheme, *, gate=None, norm_w=None, g_min=-5.0,
                 l2_eps=1e-6, norm_eps=1e-6, C=64):
    """One head, one sequence of a multiple of 64 tokens.  q, k, v [T, d] (bf16 values),
    g [T, d] raw log-retention, beta [T], S0 [d, d]; gate [T, d] logits or None.
    Returns (out as stored: bf16 values in fp32, final state)."""
    sc = SCHEMES[scheme]
    dt = sc["dt"]
    q, k, v, g, beta = (np.asarray(x, dtype=dt) for x in (q, k, v, g, beta))
    S = np.asarray(S0, dtype=dt).copy()
    T_, d = q.shape
    assert T_ % C == 0
    out = np.zeros((T_, d), dtype=np.float64)
    rq = (1 / np.sqrt((q * q).sum(1) + dt(l2_eps))).astype(dt)
    rk = (1 / np.sqrt((k * k).sum(1) + dt(l2_eps))).astype(dt)
    pd_all = (q * k).sum(1) * rq * rk
    blk = np.arange(C) // 16
    for c0 in range(0, T_, C):
        sl = slice(c0, c0 + C)
        qc, kc, vc, bc = q[sl], k[sl], v[sl], beta[sl]
        rqc, rkc = rq[sl][:, None], rk[sl][:, None]
        gam = np.cumsum(np.maximum(g[sl], dt(g_min)) * dt(LOG2E), axis=0, dtype=dt)
        g0 = np.concatenate([np.zeros((1, d), dtype=dt), gam[15:C - 1:16]], axis=0)  # [4, d]
        rel = gam - g0[blk]
        Kt, Qt = kc * rkc * np.exp2(rel), qc * rqc * np.exp2(rel)
        Kh_own = kc * rkc * np.exp2(-rel)
        Dk = np.zeros((C, C), dtype=dt)
        Dq = np.zeros((C, C), dtype=dt)
        for R in range(4):
            rb = slice(16 * R, 16 * R + 16)
            for Rs in range(R + 1):
                cb = slice(16 * Rs, 16 * Rs + 16)
                Kh = Kh_own[cb] if Rs == R else Kh_own[cb] * np.exp2(g0[R] - g0[Rs])
                band = sc["band"] == "all" or (sc["band"] == "own" and R == Rs) or (
                    sc["band"] is True and R - Rs <= 1)
                Dk[rb, cb] = _prod(Kt[rb], Kh, sc, band)
                Dq[rb, cb] = _prod(Qt[rb], Kh, sc, band and sc.get("split_q", True))
        low = np.tril(np.ones((C, C), dtype=bool), -1)
        A = np.where(low, bc[:, None] * Dk, 0).astype(dt)
        P = np.where(low, sc["p"](Dq), 0).astype(dt)
        Tm = sc["t"](_inverse(A, sc))
        G = np.exp2(gam)
        KG, QG = sc["x"](kc * rkc * G), sc["x"](qc * rqc * G)
        St = sc["s"](S)
        Xk, Xq = KG @ St, QG @ St
        if sc.get("xq") == "bf16x3":  # the query rows: three bf16 products of split operands
            QGe = (qc * rqc * G).astype(dt)
            Qh, Sh = bf16(QGe), bf16(S)
            Xq = Qh @ Sh + bf16(QGe - Qh) @ Sh + Qh @ bf16(S - Sh)
        if sc.get("xk") == "bf16x3":  # the key rows likewise
            KGe = (kc * rkc * G).astype(dt)
            Kh, Sh = bf16(KGe), bf16(S)
            Xk = Kh @ Sh + bf16(KGe - Kh) @ Sh + Kh @ bf16(S - Sh)
        Y = bc[:, None] * (vc - Xk)
        if sc["y_split"]:
            Yh = sc["y"](Y)
            Ye = Yh + sc["y"](Y - Yh)
        else:
            Ye = sc["y"](Y)
        u = (Tm @ Ye).astype(dt)
        o = Xq + P @ sc["u"](u) + pd_all[sl][:, None] * u
        Kb = kc * rkc * np.exp2(gam[-1] - gam)
        if sc["upd"] == "bf16x3":
            Kbh, uh = bf16(Kb), bf16(u)
            upd = Kbh.T @ uh + bf16(Kb - Kbh).T @ uh + Kbh.T @ bf16(u - uh)
        elif sc["upd"] == "bf16x2k":  # hi*hi + lo*hi (the key's residual only)
            Kbh = bf16(Kb)
            upd = Kbh.T @ bf16(u) + bf16(Kb - Kbh).T @ bf16(u)
        elif sc["upd"] == "bf16x2u":  # hi*hi + hi*lo (the write's residual only)
            Kbh, uh = bf16(Kb), bf16(u)
            upd = Kbh.T @ uh + Kbh.T @ bf16(u - uh)
        elif sc["upd"] == "bf16":
            upd = bf16(Kb).T @ bf16(u)
        else:
            upd = Kb.T @ u
        S = (np.exp2(gam[-1])[:, None] * S + upd).astype(dt)
        if gate is not None:
            gt = np.asarray(gate[sl], dtype=np.float64)
            w = np.ones(d) if norm_w is None else np.asarray(norm_w, dtype=np.float64)
            o64 = o.astype(np.float64)
            o = o64 / np.sqrt((o64 * o64).mean(1, keepdims=True) + norm_eps) * w / (1 + np.exp(-gt))
        out[sl] = o
    stored = out if dt == np.float64 else bf16(out.astype(np.float32)).astype(np.float64)
    return stored, S.astype(np.float64)


# ---------------------------------------------------------------------------------------
# The FP8 output quantiser as the kernels round it (a model of the device, not the oracle):
# the group's amax clamped at 1e-10, the scale amax / 448 and the factor 448 / amax each
# divided once in IEEE fp32 (round to nearest), every value multiplied by that factor in
# fp32, then converted to E4M3 (nearest even, saturated).  The oracle's quantiser is the
# fp64 definition code = E4M3(x / scale); the two differ only where the fp32 product lands
# on the other side of an E4M3 rounding boundary than the exact quotient.
# ---------------------------------------------------------------------------------------

def fp8_quantize_groups_device(x, group=128):
    from oracle import FP8_EPS, FP8_MAX, fp8_e4m3_encode

    x = np.asarray(x, dtype=np.float32)
    shp = x.shape
    xg = x.reshape(shp[:-1] + (shp[-1] // group, group))
    a = np.maximum(np.abs(xg).max(axis=-1), np.float32(FP8_EPS)).astype(np.float32)
    scale = (a / np.float32(FP8_MAX)).astype(np.float32)
    inv = (np.float32(FP8_MAX) / a).astype(np.float32)
    codes = fp8_e4m3_encode((xg * inv[..., None]).astype(np.float32))
    return codes.reshape(shp), scale
