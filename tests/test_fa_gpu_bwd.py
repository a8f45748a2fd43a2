"""GPU parity of the attention backward (fa_bwd) against the fp64 oracle.

The GPU forward produces O and lse, the GPU backward takes them with dO and
returns dQ, dK, dV; the oracle differentiates the exact attention of the same
16-bit inputs.  Tolerance: a per-element bound derived from the kernels'
arithmetic (tests/grad_bounds.py): P and dS rounded to the 16-bit type, fp32
products and accumulation, each gradient rounded once, and the coherent term
that delta = dO . O carries from the O the forward stored (computed here from
the stored O against the oracle's).  The bound is checked on the CPU against
an emulation of that arithmetic and against the planted backward mistakes
(tests/test_grad_bounds_cpu.py).
"""
import numpy as np
import pytest

import oracle
from exact_io_aware_30_gb300 import fa, inputs

import grad_bounds

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


def _dev(bits, dtype):
    tdt = torch.bfloat16 if dtype == inputs.BF16 else torch.float16
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt).cuda()


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu_bwd(inp, dout_bits):
    """GPU forward then backward; returns (dq, dk, dv) and the forward's (O, lse)."""
    w = inp.workload
    q, k, v, do = (_dev(b, w.dtype) for b in (inp.q_bits, inp.k_bits, inp.v_bits, dout_bits))
    o, lse = fa.forward(q, k, v, scale=w.scale, mask=w.mask, window=w.window)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, scale=w.scale, mask=w.mask, window=w.window)
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK
    return (_np(dq), _np(dk), _np(dv)), (_np(o), lse.cpu().numpy().astype(np.float64))


def check_case(got, fwd, qf, kf, vf, dof, scale, mask, window, dtype):
    """Oracle gradients and forward of these inputs, then the per-element bound."""
    ref = oracle.attention_bwd(qf, kf, vf, dof, scale, mask, window)
    o_ref, lse_ref = oracle.attention(qf, kf, vf, scale, mask, window)
    bounds = grad_bounds.gradient_bounds(qf, kf, vf, dof, fwd[0], fwd[1], o_ref, lse_ref, scale,
                                         mask, window, dtype, ref)
    return grad_bounds.check_gradients(got, ref, bounds), ref


def bwd_case(B, H, Sq, Sk, d, dtype, mask, window=0, seed=0, Hkv=0, spiky=False):
    inp = inputs.custom(B, H, Sq, Sk, d, dtype, mask, window, seed=seed, Hkv=Hkv,
                        spiky_keys=spiky)
    dob = inputs.grad_output(inp.workload)
    got, fwd = run_gpu_bwd(inp, dob)
    qf, kf, vf = inp.f64()
    stats, ref = check_case(got, fwd, qf, kf, vf, inputs.bits_to_f64(dob, dtype),
                            inp.workload.scale, mask, window, dtype)
    return stats, got, ref


SHAPES = [(1, 1), (64, 64), (127, 127), (128, 128), (129, 129), (300, 300), (300, 173),
          (173, 300), (700, 700)]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("dtype", [inputs.BF16, inputs.FP16])
@pytest.mark.parametrize("mask,window", [("none", 0), ("causal", 0), ("window", 1),
                                         ("window", 77), ("window", 300)])
def test_bwd_parity_small(d, dtype, mask, window):
    for i, (Sq, Sk) in enumerate(SHAPES):
        stats, _, _ = bwd_case(1, 2, Sq, Sk, d, dtype, mask, window, seed=50 + i)
        print(Sq, Sk, stats)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_bwd_many_units_heads_and_batches(d):
    bwd_case(3, 5, 400, 400, d, inputs.BF16, "causal", seed=60 + d)
    bwd_case(2, 4, 333, 517, d, inputs.BF16, "none", seed=61 + d)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (6, 1), (8, 8)])
def test_bwd_grouped_query_heads(d, H, Hkv):
    bwd_case(2, H, 300, 260, d, inputs.BF16, "causal", seed=70 + H + Hkv, Hkv=Hkv)
    bwd_case(1, H, 200, 333, d, inputs.FP16, "window", 90, seed=71 + H + Hkv, Hkv=Hkv)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_bwd_spiky_keys(d):
    bwd_case(1, 2, 600, 600, d, inputs.BF16, "none", seed=80 + d, spiky=True)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_bwd_rows_without_keys_get_zero_dq(d):
    # window with Sq > Sk: rows i >= Sk + W - 1 see no key, and keys past the
    # last row's window are seen by nobody
    _, got, ref = bwd_case(1, 2, 400, 40, d, inputs.BF16, "window", 17, seed=90 + d)
    dq = got[0]
    assert np.all(dq[:, :, 40 + 16:] == 0.0)


def test_bwd_keys_seen_by_no_row_get_zero():
    # causal with Sk > Sq: keys j >= Sq are hidden from every row
    _, got, _ = bwd_case(1, 2, 100, 300, 128, inputs.BF16, "causal", seed=95)
    assert np.all(got[1][:, :, 100:] == 0.0) and np.all(got[2][:, :, 100:] == 0.0)


def test_bwd_deterministic():
    inp = inputs.custom(2, 3, 500, 500, 128, inputs.BF16, "causal", seed=96)
    dob = inputs.grad_output(inp.workload)
    a = run_gpu_bwd(inp, dob)[0]
    b = run_gpu_bwd(inp, dob)[0]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_bwd_empty_query_zeroes_dk_dv():
    k = torch.randn(1, 2, 50, 64, device="cuda").to(torch.bfloat16)
    q = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 2, 0, dtype=torch.float32, device="cuda")
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(k, 7.0)
    fa.backward(q, k, k, q, lse, q, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0


def test_bwd_unsupported_head_dim_is_refused():
    q = torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 8, dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.backward(q, q, q, q, lse, q)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED


def test_bwd_d256_keys_seen_by_no_row_get_zero():
    _, got, _ = bwd_case(1, 2, 100, 300, 256, inputs.BF16, "causal", seed=97)
    assert np.all(got[1][:, :, 100:] == 0.0) and np.all(got[2][:, :, 100:] == 0.0)


BWD_FULL = inputs.Workload("bwd_b1h32_s8192_d128_fp16_causal", 1, 32, 8192, 8192, 128,
                           inputs.FP16, "causal", seed=1003)


def test_bwd_full_size_two_heads():
    # the benchmark's backward workload (8k tokens x 32 heads, causal, fp16),
    # run whole on the GPU; the oracle differentiates heads 0 and 31, which
    # are independent of the others
    w = BWD_FULL
    inp = inputs.generate(w)
    dob = inputs.grad_output(w)
    (dq, dk, dv), (o, lse) = run_gpu_bwd(inp, dob)
    qf, kf, vf = inp.f64()
    dof = inputs.bits_to_f64(dob, w.dtype)
    for h in (0, w.H - 1):
        sl = slice(h, h + 1)
        stats, _ = check_case((dq[:, sl], dk[:, sl], dv[:, sl]), (o[:, sl], lse[:, sl]),
                              qf[:, sl], kf[:, sl], vf[:, sl], dof[:, sl], w.scale, w.mask, 0,
                              w.dtype)
        print(f"{w.name} head {h}: {stats}")


@pytest.mark.parametrize("d", [128, 256])
def test_bwd_under_cuda_graph_capture(d):
    # The backward runs dQ on a library stream forked from and joined back to
    # the caller's with events (and at d = 256 its dK/dV kernel as clusters
    # of two): captured into a CUDA graph and replayed, it gives the bits of
    # a direct call (and the replay depends on nothing enqueued outside the
    # graph).
    inp = inputs.custom(1, 4, 700, 700, d, inputs.BF16, "causal", 0, seed=98)
    w = inp.workload
    q, k, v, do = (_dev(b, w.dtype)
                   for b in (inp.q_bits, inp.k_bits, inp.v_bits, inputs.grad_output(w)))
    o, lse = fa.forward(q, k, v, scale=w.scale, mask=w.mask)
    ref = fa.backward(q, k, v, o, lse, do, scale=w.scale, mask=w.mask)
    torch.cuda.synchronize()
    dq, dk, dv = (torch.empty_like(x) for x in (q, k, v))
    st, ws_bytes = fa.bwd_workspace_query(1, 4, 4, 700, 700, d, "causal", 0, fa.DTYPE_BF16)
    assert st == fa.FA_OK
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # a call outside the capture on the capture's stream first
        fa.backward(q, k, v, o, lse, do, scale=w.scale, mask=w.mask, dq=dq, dk=dk, dv=dv,
                    workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.backward(q, k, v, o, lse, do, scale=w.scale, mask=w.mask, dq=dq, dk=dk, dv=dv,
                    workspace=ws)
    for x in (dq, dk, dv):
        x.fill_(7.0)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK
    for a, b in zip((dq, dk, dv), ref):
        assert torch.equal(a, b)


def test_bwd_calls_from_two_threads_on_two_streams():
    # Two host threads call the backward at once, each on its own stream:
    # the library serialises the enqueue of its shared dQ stream and events,
    # and each call's results are the bits of the same call made alone.
    import threading
    cases = []
    for i, (S, mask) in enumerate(((600, "causal"), (900, "none"))):
        inp = inputs.custom(1, 4, S, S, 128, inputs.BF16, mask, 0, seed=120 + i)
        w = inp.workload
        q, k, v, do = (_dev(b, w.dtype)
                       for b in (inp.q_bits, inp.k_bits, inp.v_bits, inputs.grad_output(w)))
        o, lse = fa.forward(q, k, v, scale=w.scale, mask=mask)
        ref = fa.backward(q, k, v, o, lse, do, scale=w.scale, mask=mask)
        cases.append((q, k, v, o, lse, do, w.scale, mask, ref))
    torch.cuda.synchronize()
    results = [None, None]
    errors = []

    def run(idx):
        try:
            q, k, v, o, lse, do, scale, mask, _ = cases[idx]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(3):
                    results[idx] = fa.backward(q, k, v, o, lse, do, scale=scale, mask=mask, stream=s)
            s.synchronize()
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK
    for idx in range(2):
        for a, b in zip(results[idx], cases[idx][8]):
            assert torch.equal(a, b)
