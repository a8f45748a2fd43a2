"""Per-element error bounds for the attention backward's 16-bit arithmetic.

The gradients follow the chain of "FlashAttention: Why Tiling Attention
Makes Transformers Fast Without Changing the Result", section "The backward
pass: recompute instead of storing" (per head, visible pairs only):

    P_ij  = exp(scale q_i . k_j - lse_i)          dP_ij = dO_i . v_j
    delta_i = sum_j P_ij dP_ij (= dO_i . O_i)     dS_ij = P_ij (dP_ij - delta_i)
    dV_j = sum_i P_ij dO_i    dQ_i = scale sum_j dS_ij k_j    dK_j = scale sum_i dS_ij q_i

The kernels compute S and dP with fp32 accumulation, round P and dS to the
16-bit input type (unit roundoff u: 2^-8 for bf16, 2^-11 for fp16) before the
products that use them, accumulate the gradients in fp32 and round each
gradient once.  delta is taken as dO_i . O_i from the O the forward stored in
16 bits.  To first order, each gradient element then differs from the exact
one by

  * a coherent term from delta's error d_delta_i = dO_i . (O_stored_i - O_i):
    it enters every dS_ij of row i as -P_ij d_delta_i, so dQ_i gains
    -scale d_delta_i sum_j P_ij k_j and dK_j gains -scale sum_i P_ij d_delta_i q_i
    (these are computed here from the stored O, signed, then taken in
    absolute value);
  * relative errors of each term: P's rounding and dS's rounding (u each),
    the forward's lse error (measured, per row), the fp32 rounding of the
    exponent's argument, the fp32 accumulation of S, dP and the gradients
    (at most n 2^-24 of the sum of |terms| for n additions); these are
    bounded term by term (worst case, no averaging);
  * for fp16, absolute errors of subnormal P and dS codes (half the
    subnormal spacing, 2^-25);
  * the final rounding of the gradient, u |G|.

Every bound here is a sum of absolute values, so it is an upper bound on the
first-order error whatever the signs; a mistake in the chain (a dropped term,
a wrong operand or index) changes gradients by the order of |G| itself.  The
quantities P, dP, delta are evaluated in float64 from the exact lse the
oracle returns; they weight the bound and are not the values compared.
"""
from __future__ import annotations

import numpy as np

BF16 = "bf16"
FP16 = "fp16"


def unit_roundoff(dtype: str) -> float:
    """Half the spacing of the 16-bit type at 1: 2^-8 (bf16, 8 significant
    bits) or 2^-11 (fp16, 11 significant bits)."""
    return 2.0 ** -8 if dtype == BF16 else 2.0 ** -11


def _visible(i0: int, i1: int, Sk: int, mask: str, window: int) -> np.ndarray:
    """[i1 - i0, Sk] booleans: key j visible to query row i (causal top-left,
    window = the W keys ending at the diagonal)."""
    i = np.arange(i0, i1)[:, None]
    j = np.arange(Sk)[None, :]
    vis = np.ones((i1 - i0, Sk), dtype=bool)
    if mask != "none":
        vis &= j <= i
    if mask == "window":
        vis &= j > i - window
    return vis


def gradient_bounds(qf, kf, vf, dof, o_stored, lse_stored, o_ref, lse_ref, scale: float,
                    mask: str, window: int, dtype: str, g_ref, row_block: int = 1024):
    """Elementwise bounds (dq, dk, dv) on |G - G_ref| for the kernels'
    arithmetic.  qf, dof, o_* are [B, H, Sq, d]; kf, vf [B, Hkv, Sk, d];
    lse_* [B, H, Sq]; g_ref = the exact (dq, dk, dv)."""
    B, H, Sq, d = qf.shape
    Hkv, Sk = kf.shape[1], kf.shape[2]
    g = H // Hkv
    u = unit_roundoff(dtype)
    # fp32 accumulation: at most n additions per gradient element or score
    acc = (Sk + Sq * g + d) * 2.0 ** -23
    sub = 2.0 ** -25 if dtype == FP16 else 0.0   # subnormal 16-bit codes (absolute)
    bq = np.zeros_like(qf)
    bk = np.zeros_like(kf)
    bv = np.zeros_like(vf)
    ck = np.zeros_like(kf)       # coherent dK term, signed, summed over rows and heads
    for b in range(B):
        for h in range(H):
            kv = h // g
            K, V = kf[b, kv], vf[b, kv]
            aK, aV = np.abs(K), np.abs(V)
            for i0 in range(0, Sq, row_block):
                i1 = min(Sq, i0 + row_block)
                Q, dO = qf[b, h, i0:i1], dof[b, h, i0:i1]
                aQ, adO = np.abs(Q), np.abs(dO)
                lr = lse_ref[b, h, i0:i1]
                fin = np.isfinite(lr)
                vis = _visible(i0, i1, Sk, mask, window) & fin[:, None]
                lr0 = np.where(fin, lr, 0.0)
                S = scale * (Q @ K.T)
                with np.errstate(over="ignore", invalid="ignore"):
                    P = np.where(vis, np.exp(np.where(vis, S - lr0[:, None], 0.0)), 0.0)
                dP = dO @ V.T
                delta = (P * dP).sum(axis=1)
                # delta from the stored O: coherent part and its fp32 evaluation
                d_delta = (dO * (o_stored[b, h, i0:i1] - o_ref[b, h, i0:i1])).sum(axis=1)
                e_delta = 2.0 * d * 2.0 ** -23 * (adO * np.abs(o_stored[b, h, i0:i1])).sum(axis=1)
                ls = lse_stored[b, h, i0:i1]
                d_lse = np.where(fin, np.abs(np.where(fin, ls, 0.0) - lr0), 0.0)
                # relative error of one P element: P's rounding, the lse the
                # forward returned, the fp32 score (d products) and argument,
                # and the exponent instruction
                r_p = (u + d_lse[:, None] + d * 2.0 ** -23 * scale * (aQ @ aK.T)
                       + 2.0 ** -22 * (np.abs(S) + np.abs(lr0)[:, None]) + 2.0 ** -20)
                r_s = r_p + u + acc              # plus dS's rounding and the accumulation
                # |dP - delta| with the fp32 errors of dP (d products) and of the
                # subtraction
                G = (np.abs(dP - delta[:, None]) + d * 2.0 ** -23 * (adO @ aV.T)
                     + 2.0 ** -22 * (np.abs(dP) + np.abs(delta)[:, None]))
                W = P * (r_s * (G + np.abs(d_delta)[:, None]) + e_delta[:, None])
                if sub:
                    W = W + vis * sub * (G + np.abs(d_delta)[:, None] + 1.0)
                bq[b, h, i0:i1] += scale * (W @ aK + np.abs(d_delta)[:, None] * np.abs(P @ K))
                bk[b, kv] += scale * (W.T @ aQ)
                ck[b, kv] += scale * ((P * d_delta[:, None]).T @ Q)
                Wv = P * (r_p + acc)
                if sub:
                    Wv = Wv + vis * sub
                bv[b, kv] += Wv.T @ adO
    bk += np.abs(ck)
    out = []
    for inner, ref in zip((bq, bk, bv), g_ref):
        out.append(inner * (1.0 + u) + u * np.abs(ref) + 2.0 ** -24)
    return tuple(out)


def check_gradients(got, ref, bounds, names=("dq", "dk", "dv")):
    """Asserts |got - ref| <= bound elementwise; returns per-tensor stats
    (max and mean error, the reference's scale, the worst error/bound)."""
    stats = {}
    for name, gv, rv, bd in zip(names, got, ref, bounds):
        assert np.all(np.isfinite(gv)), f"{name}: non-finite values"
        err = np.abs(gv - rv)
        ratio = err / bd
        st = dict(max=float(err.max()), mean=float(err.mean()), ref_max=float(np.abs(rv).max()),
                  ref_mean=float(np.abs(rv).mean()), worst_ratio=float(ratio.max()),
                  bound_mean=float(bd.mean()))
        stats[name] = st
        bad = ratio > 1.0
        assert not bad.any(), (name, st, int(bad.sum()), np.argwhere(bad)[:4].tolist())
    return stats
