"""GPU tests of the forward from host memory (fa_fwd_host): the library
copies Q, K, V in, runs the fused forward chunk by chunk (whole K/V heads per
chunk) and copies O and lse out.  Every unit of the forward computes the same
arithmetic whatever the chunking and scheduling, so the results must be
bitwise those of the device forward; they are also checked against the
fp64 oracle with the forward's tolerances."""
import numpy as np
import pytest

import oracle
from exact_io_aware_30_gb300 import fa, inputs

from test_fa_gpu import compare

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


def _host(bits, dtype):
    tdt = torch.bfloat16 if dtype == inputs.BF16 else torch.float16
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt).pin_memory()


CASES = [
    # B, H, Hkv, S, d, dtype, mask, window
    (1, 32, 32, 2048, 128, inputs.BF16, "causal", 0),      # 6 chunks of whole heads
    (2, 16, 4, 1500, 128, inputs.FP16, "window", 333),     # grouped K/V, chunks of K/V heads
    (1, 8, 8, 4100, 64, inputs.BF16, "none", 0),           # ragged tail in every head
    (2, 4, 4, 1000, 256, inputs.BF16, "causal", 0),        # d = 256
    (1, 2, 1, 300, 128, inputs.BF16, "causal", 0),         # one chunk
]


@pytest.mark.parametrize("case", CASES, ids=[f"h{c[1]}kv{c[2]}-s{c[3]}-d{c[4]}-{c[6]}" for c in CASES])
def test_host_forward_equals_device_forward_and_oracle(case):
    B, H, Hkv, S, d, dtype, mask, window = case
    inp = inputs.custom(B, H, S, S, d, dtype, mask, window, seed=1200 + S,
                        Hkv=Hkv if Hkv != H else 0)
    w = inp.workload
    qh, kh, vh = (_host(b, dtype) for b in (inp.q_bits, inp.k_bits, inp.v_bits))
    st, ws_bytes = fa.host_workspace_query(B, H, Hkv, S, S, d, mask, window,
                                           fa.DTYPE_BF16 if dtype == inputs.BF16 else fa.DTYPE_FP16)
    assert st == fa.FA_OK and ws_bytes > 0
    # two calls in a row into the same caller buffers and workspace
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    o_h = torch.empty(qh.shape, dtype=qh.dtype, pin_memory=True)
    l_h = torch.empty((B, H, S), dtype=torch.float32, pin_memory=True)
    for _ in range(2):
        o_h.fill_(7.0)
        fa.forward_host(qh, kh, vh, scale=w.scale, mask=mask, window=window, out=o_h, lse=l_h,
                        workspace=ws)
        assert fa.device_error() == fa.FA_OK
        o_d, l_d = fa.forward(qh.cuda(), kh.cuda(), vh.cuda(), scale=w.scale, mask=mask,
                              window=window)
        torch.cuda.synchronize()
        assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())
    qf, kf, vf = inp.f64()
    o_ref, lse_ref = oracle.attention(qf, kf, vf, w.scale, mask, window)
    compare(o_h.float().numpy().astype(np.float64), l_h.numpy().astype(np.float64), o_ref,
            lse_ref, dtype)


def test_host_forward_rejects_device_tensors():
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.forward_host(q, q, q)
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    # the raw entry point refuses device pointers itself
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    qh = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, pin_memory=True)
    lh = torch.zeros(1, 1, 8, dtype=torch.float32, pin_memory=True)
    st = fa.fwd_host_raw(q.data_ptr(), qh.data_ptr(), qh.data_ptr(), qh.data_ptr(), lh.data_ptr(),
                         ws.data_ptr(), ws.numel(), 1, 1, 1, 8, 8, 64, 0.125, fa.MASK_NONE, 0,
                         fa.DTYPE_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_ERR_INVALID_ARG


def test_host_forward_empty_query_is_a_noop():
    q = torch.zeros(1, 2, 0, 128, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 5, 128, dtype=torch.bfloat16)
    o, lse = fa.forward_host(q, k, k)
    assert o.numel() == 0 and lse.numel() == 0


def test_host_forward_with_as_many_chunks_as_heads():
    # 8 K/V heads of 8.4 MB each make 8 chunks; with the half-weight first and
    # last chunks the first one is empty and skipped.  Bitwise the device
    # forward (itself checked against the oracle elsewhere).
    B, H, S, d = 1, 8, 11000, 128
    inp = inputs.custom(B, H, S, S, d, inputs.BF16, "causal", 0, seed=1299)
    w = inp.workload
    qh, kh, vh = (_host(b, inputs.BF16) for b in (inp.q_bits, inp.k_bits, inp.v_bits))
    o_h, l_h = fa.forward_host(qh, kh, vh, scale=w.scale, mask="causal")
    assert fa.device_error() == fa.FA_OK
    o_d, l_d = fa.forward(qh.cuda(), kh.cuda(), vh.cuda(), scale=w.scale, mask="causal")
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())
