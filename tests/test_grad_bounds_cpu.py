"""CPU checks of the backward's per-element error bound (tests/grad_bounds.py).

Two directions, so that the bound is neither too tight nor vacuous:
  * a float32 emulation of the kernels' arithmetic (P and dS rounded to the
    16-bit type, delta from the 16-bit O, fp32 products, one rounding of each
    gradient) stays inside it on small cases with every mask, grouped K/V
    heads and spiky keys, for both 16-bit types;
  * every planted mistake in the oracle's backward (the mutations of the pin
    suite) produces gradients that break it.
"""
import numpy as np
import pytest

import oracle
from exact_io_aware_30_gb300 import inputs

import grad_bounds

LOG2E = 1.4426950408889634


def _r16(x, dtype):
    return inputs.round_to_dtype(np.asarray(x, dtype=np.float32), dtype)


def emulate_kernel_bwd(qf, kf, vf, dof, o_stored, lse, scale, mask, window, dtype):
    """The kernels' roundings, in numpy float32 (test-only model)."""
    B, H, Sq, d = qf.shape
    Hkv, Sk = kf.shape[1], kf.shape[2]
    g = H // Hkv
    f = np.float32
    dq = np.zeros(qf.shape, np.float64)
    dk = np.zeros(kf.shape, np.float64)
    dv = np.zeros(vf.shape, np.float64)
    dk32 = np.zeros(kf.shape, f)
    dv32 = np.zeros(vf.shape, f)
    c = f(scale * LOG2E)
    for b in range(B):
        for h in range(H):
            kv = h // g
            Q, K, V, dO = (x.astype(f) for x in (qf[b, h], kf[b, kv], vf[b, kv], dof[b, h]))
            vis = grad_bounds._visible(0, Sq, Sk, mask, window)
            l2 = (lse[b, h] * LOG2E).astype(f)
            fin = np.isfinite(l2)
            vis &= fin[:, None]
            S = Q @ K.T
            with np.errstate(invalid="ignore", over="ignore"):
                arg = np.where(vis, S * c - np.where(fin, l2, f(0))[:, None], f(-np.inf))
                P = _r16(np.exp2(arg), dtype).astype(f)
            dP = dO @ V.T
            delta = (dO * o_stored[b, h].astype(f)).sum(axis=1, dtype=f)
            dS = _r16(P * (dP - delta[:, None]), dtype).astype(f)
            dq[b, h] = _r16(f(scale) * (dS @ K), dtype)
            dk32[b, kv] += dS.T @ Q
            dv32[b, kv] += P.T @ dO
    for b in range(B):
        for kv in range(Hkv):
            dk[b, kv] = _r16(f(scale) * dk32[b, kv], dtype)
            dv[b, kv] = _r16(dv32[b, kv], dtype)
    return dq, dk, dv


CASES = [
    # B, H, Hkv, Sq, Sk, d, mask, window, spiky
    (1, 2, 2, 130, 130, 64, "none", 0, False),
    (1, 2, 2, 200, 173, 64, "causal", 0, False),
    (2, 4, 2, 150, 190, 128, "window", 37, False),
    (1, 2, 1, 257, 257, 128, "causal", 0, True),
    (1, 1, 1, 180, 180, 256, "none", 0, True),
    (1, 2, 2, 120, 30, 64, "window", 9, False),     # rows with no visible key
]


def _case(B, H, Hkv, Sq, Sk, d, mask, window, spiky, dtype, seed):
    inp = inputs.custom(B, H, Sq, Sk, d, dtype, mask, window, seed=seed, spiky_keys=spiky,
                        Hkv=Hkv if Hkv != H else 0)
    qf, kf, vf = inp.f64()
    dof = inputs.bits_to_f64(inputs.grad_output(inp.workload), dtype)
    sc = inp.workload.scale
    o_ref, lse_ref = oracle.attention(qf, kf, vf, sc, mask, window)
    o_stored = np.where(np.isfinite(lse_ref)[..., None], _r16(o_ref, dtype), 0.0)
    lse_stored = lse_ref.astype(np.float32).astype(np.float64)
    ref = oracle.attention_bwd(qf, kf, vf, dof, sc, mask, window)
    bounds = grad_bounds.gradient_bounds(qf, kf, vf, dof, o_stored, lse_stored, o_ref, lse_ref,
                                         sc, mask, window, dtype, ref)
    return qf, kf, vf, dof, o_stored, lse_stored, sc, ref, bounds


@pytest.mark.parametrize("dtype", [inputs.BF16, inputs.FP16])
@pytest.mark.parametrize("case", CASES, ids=[f"{c[6]}-d{c[5]}-{c[3]}x{c[4]}" for c in CASES])
def test_emulated_kernel_arithmetic_is_inside_the_bound(case, dtype):
    B, H, Hkv, Sq, Sk, d, mask, window, spiky = case
    qf, kf, vf, dof, o_st, l_st, sc, ref, bounds = _case(*case, dtype, seed=900 + CASES.index(case))
    got = emulate_kernel_bwd(qf, kf, vf, dof, o_st, l_st, sc, mask, window, dtype)
    stats = grad_bounds.check_gradients(got, ref, bounds)
    print(case, dtype, {n: (round(st["worst_ratio"], 3), round(st["bound_mean"] / st["ref_mean"], 4))
                        for n, st in stats.items()})


BWD_MUTATIONS = [
    ("Jacobian row term dropped (dQ pass)", "const double ds = P[j] * (dP[j] - rowdot);",
     "const double ds = P[j] * dP[j];"),
    ("Jacobian row term sign (dK/dV pass)",
     "const double ds = Pij * (orc_dot(doi, vj, d) - rt[r]);",
     "const double ds = Pij * (orc_dot(doi, vj, d) + rt[r]);"),
    ("dK without scale", "dkj[c] += scale * ds * qi[c];", "dkj[c] += ds * qi[c];"),
    ("dQ from q", "dqi[c] += scale * ds * kj[c];", "dqi[c] += scale * ds * qi[c];"),
    ("dV from dS", "dvj[c] += Pij * doi[c];", "dvj[c] += ds * doi[c];"),
    ("unnormalised P (dQ pass)", "P[j] /= l;\n            double rowdot",
     "P[j] /= 1.0;\n            double rowdot"),
    ("P without the row sum (dK/dV pass)", "- rm[r]) / rl[r];", "- rm[r]);"),
    ("dP against k", "dP[j] = orc_dot(doi, vh + j * (int64_t)d, d);",
     "dP[j] = orc_dot(doi, kh + j * (int64_t)d, d);"),
    ("key pass skips the causal mask",
     "if (rl[r] == 0.0 || !orc_visible(mask_kind, window, i, j))", "if (rl[r] == 0.0)"),
]


@pytest.mark.parametrize("name,old,new", BWD_MUTATIONS, ids=[m[0] for m in BWD_MUTATIONS])
def test_planted_backward_mistakes_break_the_bound(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert old in src, f"mutation anchor for '{name}' not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    orc = oracle.OracleLib(oracle.compile_source(str(mutated), str(tmp_path / "libmutant.so")))
    caught = 0
    for case in (CASES[1], CASES[3]):
        B, H, Hkv, Sq, Sk, d, mask, window, spiky = case
        qf, kf, vf, dof, _, _, sc, ref, bounds = _case(*case, inputs.BF16, seed=77)
        with np.errstate(all="ignore"):
            wrong = orc.attention_bwd(qf, kf, vf, dof, sc, mask, window)
        wrong = tuple(_r16(x, inputs.BF16) for x in wrong)
        try:
            grad_bounds.check_gradients(wrong, ref, bounds)
        except AssertionError:
            caught += 1
    assert caught == 2, f"the bound let the planted mistake '{name}' through"
