"""GPU parity of the 8-bit forward (fa_fwd_fp8) against the fp64 oracle on
the dequantised inputs.

Tolerance, from the arithmetic: S is exact up to fp32 accumulation of
products of e4m3 values, and the only roundings on the way to O are those of
the weights to e4m3 and of O to bf16.  The kernel keeps a reference max m at
most 2^4 below the row's running max (so the largest weight is in [1, 2^4]
and the row sum l >= 1) and stores each weight p times 2^4.  An e4m3 code
carries a relative error of at most 2^-4 (3 mantissa bits) when normal and an
absolute one of at most 2^-10 (half the subnormal spacing) otherwise, so
|p_hat - p| <= 2^-4 p + 2^-14, and per element
  |O - O_ref| <= 2^-4 sum_j P_ij |v_jc| + 2^-14 sum_{j visible} |v_jc|
               + 2^-8 |O_ref| + 1e-6,
where sum_j P_ij |v_jc| is the oracle's attention over |V|.  The lse is
computed from unrounded weights: |lse - lse_ref| <= 1e-3 as in the 16-bit
forward.
"""
import numpy as np
import pytest

import oracle
from exact_io_aware_30_gb300 import fa, inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from exact_io_aware_30_gb300 import build
    build.build()
    fa.load()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK


def run_gpu(inp):
    w = inp.workload
    q, k, vt = (torch.from_numpy(np.ascontiguousarray(b)).cuda()
                for b in (inp.q_bits, inp.k_bits, inp.vt_bits))
    o, lse = fa.forward_fp8(q, k, vt, inp.q_descale, inp.k_descale, inp.v_descale, scale=w.scale,
                            mask=w.mask, window=w.window)
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _visible_abs_sum(w, vf, rows):
    """sum over the keys row i sees of |v_jc|, per row: [rows, d] or [B,H,Sq,d]."""
    av = np.abs(vf)                                 # [B, Hkv, Sk, d]
    csum = np.concatenate([np.zeros_like(av[:, :, :1]), np.cumsum(av, axis=2)], axis=2)
    g = w.H // w.Hkv
    flat = np.arange(w.B * w.H * w.Sq) if rows is None else np.asarray(rows)
    b, h, i = flat // (w.H * w.Sq), (flat // w.Sq) % w.H, flat % w.Sq
    hi = np.full(i.shape, w.Sk) if w.mask == "none" else np.minimum(i + 1, w.Sk)
    lo = np.maximum(0, i - w.window + 1) if w.mask == "window" else np.zeros_like(i)
    lo = np.minimum(lo, hi)
    out = csum[b, h // g, hi] - csum[b, h // g, lo]
    return out if rows is not None else out.reshape(w.B, w.H, w.Sq, w.d)


def check(inp, rows=None):
    w = inp.workload
    o, lse = run_gpu(inp)
    qf, kf, vf = inp.f64()
    o_ref, lse_ref = oracle.attention(qf, kf, vf, w.scale, w.mask, w.window, rows=rows)
    pv_abs, _ = oracle.attention(qf, kf, np.abs(vf), w.scale, w.mask, w.window, rows=rows)
    if rows is not None:
        o, lse = o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows]
    assert np.all(np.isfinite(o))
    bound = (2.0 ** -4 * pv_abs + 2.0 ** -14 * _visible_abs_sum(w, vf, rows)
             + 2.0 ** -8 * np.abs(o_ref) + 1e-6)
    err = np.abs(o - o_ref)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse))
    stats = dict(max=float(err.max()), mean=float(err.mean()),
                 worst_ratio=float((err / bound).max()),
                 lse=float(np.abs(lse[fin] - lse_ref[fin]).max()) if fin.any() else 0.0)
    assert np.all(err <= bound), stats
    assert stats["lse"] <= 1e-3, stats
    return stats


SHAPES = [(1, 16), (7, 32), (127, 128), (128, 128), (129, 144), (300, 304), (300, 176),
          (173, 304), (700, 704)]


DIMS = [64, 128, 256]


@pytest.mark.parametrize("d", DIMS)
@pytest.mark.parametrize("mask,window", [("none", 0), ("causal", 0), ("window", 1), ("window", 77)])
def test_fp8_parity_small(mask, window, d):
    for i, (Sq, Sk) in enumerate(SHAPES):
        w = inputs.Fp8Workload("t", 1, 2, 2, Sq, Sk, d, mask, window, seed=40 + i + d)
        print(Sq, Sk, check(inputs.generate_fp8(w)))


@pytest.mark.parametrize("d", DIMS)
@pytest.mark.parametrize("H,Hkv", [(4, 4), (8, 2), (6, 1)])
def test_fp8_heads_batches_and_groups(H, Hkv, d):
    w = inputs.Fp8Workload("t", 2, H, Hkv, 400, 512, d, "causal", seed=50 + H + Hkv + d)
    print(check(inputs.generate_fp8(w)))


@pytest.mark.parametrize("d", [64, 256])
def test_fp8_long_rows(d):
    """Many key tiles per row (both S buffers cycle many times at d = 256),
    with large logits so that the reference max moves and O is rescaled."""
    w = inputs.Fp8Workload("t", 1, 2, 1, 1100, 2048, d, "none", seed=70 + d)
    inp = inputs.generate_fp8(w)
    print(check(inp))
    hot = inputs.Fp8Inputs(w, inp.q_bits, inp.k_bits, inp.vt_bits, inp.q_descale * 4.0,
                           inp.k_descale * 4.0, inp.v_descale)
    print(check(hot))


@pytest.mark.parametrize("d", DIMS)
def test_fp8_rows_without_keys(d):
    w = inputs.Fp8Workload("t", 1, 2, 2, 300, 48, d, "window", 17, seed=55)
    inp = inputs.generate_fp8(w)
    check(inp)
    o, lse = run_gpu(inp)
    empty = np.arange(300) >= 48 + 16
    assert np.all(o[:, :, empty] == 0) and np.all(np.isneginf(lse[:, :, empty]))


def test_fp8_refusals():
    q = torch.zeros(1, 1, 8, 96, dtype=torch.uint8, device="cuda")
    vt = torch.zeros(1, 1, 96, 16, dtype=torch.uint8, device="cuda")
    k = torch.zeros(1, 1, 16, 96, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.forward_fp8(q, k, vt, 1.0, 1.0, 1.0)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED  # d = 96
    q = torch.zeros(1, 1, 8, 128, dtype=torch.uint8, device="cuda")
    k = torch.zeros(1, 1, 20, 128, dtype=torch.uint8, device="cuda")
    vt = torch.zeros(1, 1, 128, 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.forward_fp8(q, k, vt, 1.0, 1.0, 1.0)
    assert e.value.status == fa.FA_ERR_INVALID_ARG  # Sk not a multiple of 16
    k = torch.zeros(1, 1, 32, 128, dtype=torch.uint8, device="cuda")
    vt = torch.zeros(1, 1, 128, 32, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.forward_fp8(q, k, vt, 1.0, 0.0, 1.0)
    assert e.value.status == fa.FA_ERR_INVALID_ARG  # descale must be positive


@pytest.mark.parametrize("wi", range(len(inputs.FP8_WORKLOADS)))
def test_fp8_full_size_sampled(wi):
    w = inputs.FP8_WORKLOADS[wi]
    inp = inputs.generate_fp8(w)
    rng = np.random.default_rng(33)
    rows = np.unique(np.concatenate([rng.integers(0, w.B * w.H * w.Sq, 256),
                                     [0, 127, 128, w.Sq - 1, w.B * w.H * w.Sq - 1]]))
    print(w.name, check(inp, rows=rows))
