"""Bounded pipeline waits on the GPU: a wait that runs out sets the device
status word, the kernel winds down without a fault, and the context stays
usable.  The wait is made to run out with FA_DEBUG_STALL_MS, which points the
first softmax wait of the launch at a barrier nothing completes."""
import time

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


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("d", [64, 128, 256])
def test_timed_out_wait_is_reported_and_context_recovers(monkeypatch, d):
    inp = inputs.custom(1, 3, 300, 300, d, inputs.BF16, "causal", seed=31)
    q, k, v = (_dev(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits))
    assert fa.device_error() == fa.FA_OK

    monkeypatch.setenv("FA_DEBUG_STALL_MS", "50")
    t0 = time.time()
    fa.forward(q, k, v, scale=inp.workload.scale, mask="causal")
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert fa.device_error() == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.device_error() == fa.FA_OK  # reading clears it
    assert elapsed < 10.0

    monkeypatch.delenv("FA_DEBUG_STALL_MS")
    o, lse = fa.forward(q, k, v, scale=inp.workload.scale, mask="causal")
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK
    qf, kf, vf = inp.f64()
    o_ref, lse_ref = oracle.attention(qf, kf, vf, inp.workload.scale, "causal")
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    assert np.abs(o - o_ref).mean() <= 1e-3
    assert np.abs(lse - lse_ref).max() <= 1e-3
