"""fa_bwd_noalloc (the backward with the library's fixed workspace) against
fa_bwd with a caller workspace: two calls in a row on different problems
must give the very bits fa_bwd gives.  Kept in its own file, collected last,
and independent of the other tests' state: the first call on the device does
the workspace lookup, whether or not other tests ran before it."""
import numpy as np
import pytest

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


def _problem(B, H, Hkv, S, d, dtype, mask, window, seed):
    inp = inputs.custom(B, H, S, S, d, dtype, mask, window, seed=seed, Hkv=Hkv)
    tdt = torch.bfloat16 if dtype == inputs.BF16 else torch.float16
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(tdt).cuda()
    q, k, v = dev(inp.q_bits), dev(inp.k_bits), dev(inp.v_bits)
    do = dev(inputs.grad_output(inp.workload))
    o, lse = fa.forward(q, k, v, scale=inp.workload.scale, mask=mask, window=window)
    return dict(q=q, k=k, v=v, o=o, lse=lse, do=do, B=B, H=H, Hkv=Hkv, S=S, d=d,
                scale=inp.workload.scale, mask=fa.mask_code(mask), window=window,
                dt=fa.DTYPE_BF16 if dtype == inputs.BF16 else fa.DTYPE_FP16)


def _noalloc(p):
    dq, dk, dv = torch.empty_like(p["q"]), torch.empty_like(p["k"]), torch.empty_like(p["v"])
    st = fa.bwd_noalloc_raw(p["q"].data_ptr(), p["k"].data_ptr(), p["v"].data_ptr(),
                            p["o"].data_ptr(), p["lse"].data_ptr(), p["do"].data_ptr(),
                            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), p["B"], p["H"], p["Hkv"],
                            p["S"], p["S"], p["d"], p["scale"], p["mask"], p["window"],
                            torch.cuda.current_stream().cuda_stream, p["dt"])
    assert st == fa.FA_OK, fa.status_string(st)
    return dq, dk, dv


def _with_workspace(p):
    return fa.backward(p["q"], p["k"], p["v"], p["o"], p["lse"], p["do"], scale=p["scale"],
                       mask=p["mask"], window=p["window"])


def test_two_calls_in_a_row_match_fa_bwd():
    a = _problem(2, 4, 2, 333, 128, inputs.BF16, "causal", 0, seed=901)
    b = _problem(1, 3, 3, 517, 64, inputs.FP16, "window", 100, seed=902)
    got_a = _noalloc(a)
    got_b = _noalloc(b)  # reuses the same fixed workspace right after the first
    torch.cuda.synchronize()
    ref_a = _with_workspace(a)
    ref_b = _with_workspace(b)
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK
    for g, r in zip(got_a + got_b, ref_a + ref_b):
        assert torch.equal(g, r)


def test_sizes_over_the_limit_are_refused():
    # 32 MiB holds 4,194,304 padded rows; 33 heads x 128k rows is over it
    z = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(4, dtype=torch.float32, device="cuda")
    st = fa.bwd_noalloc_raw(z.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(),
                            lse.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(),
                            z.data_ptr(), 1, 33, 33, 131072, 131072, 128, 0.088, fa.MASK_CAUSAL,
                            0, 0, fa.DTYPE_BF16)
    assert st == fa.FA_ERR_INVALID_ARG


def test_a_problem_filling_the_whole_array_is_accepted_and_exact():
    # 32768 batches of one one-row head pad to 32768 x 128 = 4,194,304 rows:
    # exactly the 32 MiB array, so this call writes its last bytes
    a = _problem(32768, 1, 1, 1, 64, inputs.BF16, "none", 0, seed=903)
    got = _noalloc(a)
    torch.cuda.synchronize()
    ref = _with_workspace(a)
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK
    for g, r in zip(got, ref):
        assert torch.equal(g, r)
    # one more batch is over the limit
    z = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(4, dtype=torch.float32, device="cuda")
    st = fa.bwd_noalloc_raw(z.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(),
                            lse.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(),
                            z.data_ptr(), 32769, 1, 1, 1, 1, 64, 0.125, fa.MASK_NONE, 0, 0,
                            fa.DTYPE_BF16)
    assert st == fa.FA_ERR_INVALID_ARG
