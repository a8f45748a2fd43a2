"""Bounded pipeline waits on the GPU: a wait that runs out sets the device
status word, the kernel winds down without a fault, and the context stays
usable.  The wait is made to run out with the test hook fa_set_debug_stall_ms,
which points the first softmax (or compute-warp) wait of each launch at a
barrier nothing completes, for the forward, the backward, paged decoding and
the 8-bit forward."""
import time

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


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("d", [64, 128, 256])
def test_timed_out_wait_is_reported_and_context_recovers(d):
    inp = inputs.custom(1, 3, 300, 300, d, inputs.BF16, "causal", seed=31)
    q, k, v = (_dev(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits))
    assert fa.device_error() == fa.FA_OK

    fa.set_debug_stall_ms(50)
    t0 = time.time()
    fa.forward(q, k, v, scale=inp.workload.scale, mask="causal")
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert fa.device_error() == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.device_error() == fa.FA_OK  # reading clears it
    assert elapsed < 10.0

    fa.set_debug_stall_ms(0)
    o, lse = fa.forward(q, k, v, scale=inp.workload.scale, mask="causal")
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK
    qf, kf, vf = inp.f64()
    o_ref, lse_ref = oracle.attention(qf, kf, vf, inp.workload.scale, "causal")
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    assert np.abs(o - o_ref).mean() <= 1e-3
    assert np.abs(lse - lse_ref).max() <= 1e-3


def _check_recovers(run, check):
    """run() under the stall hook must report the timeout within 10 s, and the
    same call afterwards must be right (check)."""
    assert fa.device_error() == fa.FA_OK
    fa.set_debug_stall_ms(50)
    try:
        t0 = time.time()
        run()
        torch.cuda.synchronize()
        elapsed = time.time() - t0
    finally:
        fa.set_debug_stall_ms(0)
    assert fa.device_error() == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.device_error() == fa.FA_OK
    assert elapsed < 10.0
    out = run()
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK
    check(out)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_timeout_is_reported_and_context_recovers(d):
    inp = inputs.custom(1, 2, 300, 300, d, inputs.BF16, "causal", seed=32)
    q, k, v = (_dev(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits))
    dob = inputs.grad_output(inp.workload)
    do = _dev(dob)
    o, lse = fa.forward(q, k, v, scale=inp.workload.scale, mask="causal")
    torch.cuda.synchronize()

    def run():
        return fa.backward(q, k, v, o, lse, do, scale=inp.workload.scale, mask="causal")

    def check(grads):
        qf, kf, vf = inp.f64()
        refs = oracle.attention_bwd(qf, kf, vf, inputs.bits_to_f64(dob, inputs.BF16),
                                    inp.workload.scale, "causal")
        o_ref, lse_ref = oracle.attention(qf, kf, vf, inp.workload.scale, "causal")
        bounds = grad_bounds.gradient_bounds(
            qf, kf, vf, inputs.bits_to_f64(dob, inputs.BF16), o.float().cpu().numpy().astype(np.float64),
            lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, inp.workload.scale, "causal", 0,
            inputs.BF16, refs)
        grad_bounds.check_gradients(tuple(g.float().cpu().numpy().astype(np.float64) for g in grads),
                                    refs, bounds)

    _check_recovers(run, check)


@pytest.mark.parametrize("kernel", ["cuda_cores", "tensor_cores"])
def test_decode_timeout_is_reported_and_context_recovers(kernel):
    # 2 rows per K/V head: either kernel serves
    inp = inputs.custom_paged(3, 4, 2, 1, 128, 16, 400, inputs.BF16, "causal", seed=33)
    q, kc, vc = (_dev(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits))
    table = torch.from_numpy(inp.block_table).cuda()
    lens = torch.from_numpy(inp.seq_lens).cuda()

    def run():
        return fa.decode_paged(q, kc, vc, table, lens, 400, mask="causal", kernel=kernel)

    def check(out):
        qf, kf, vf = inp.f64()
        o_ref, _ = oracle.attention_paged(qf, kf, vf, inp.block_table, inp.seq_lens,
                                          inp.workload.scale, "causal")
        assert np.abs(out[0].float().cpu().numpy().astype(np.float64) - o_ref).mean() <= 1e-3

    _check_recovers(run, check)


def test_fp8_timeout_is_reported_and_context_recovers():
    w = inputs.Fp8Workload("t", 1, 2, 2, 300, 304, 128, "causal", seed=34)
    inp = inputs.generate_fp8(w)
    q, k, vt = (torch.from_numpy(np.ascontiguousarray(b)).cuda()
                for b in (inp.q_bits, inp.k_bits, inp.vt_bits))

    def run():
        return fa.forward_fp8(q, k, vt, inp.q_descale, inp.k_descale, inp.v_descale, mask="causal")

    def check(out):
        qf, kf, vf = inp.f64()
        o_ref, _ = oracle.attention(qf, kf, vf, w.scale, "causal")
        assert np.abs(out[0].float().cpu().numpy().astype(np.float64) - o_ref).mean() <= 1e-2

    _check_recovers(run, check)
