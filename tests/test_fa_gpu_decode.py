"""GPU parity of the paged-cache decoding attention (fa_decode_paged) against
the fp64 oracle, with the forward's tolerances: max |O - O_ref| <= 1e-2 (less
half an ulp of O_ref for bf16 outputs), mean <= 1e-3, |lse - lse_ref| <= 1e-3."""
import numpy as np
import pytest

import oracle
from exact_io_aware_30_gb300 import fa, inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

MAX_TOL = 1e-2
MEAN_TOL = 1e-3
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from exact_io_aware_30_gb300 import build
    build.build()
    fa.load()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK


_KERNEL = {"which": "auto"}


@pytest.fixture(autouse=True, params=["auto", "tensor_cores"])
def kernel(request):
    """Every test runs twice: with the library's own choice of kernel (the
    CUDA-core one for at most 2 rows per K/V head, else the tensor-core one)
    and with the tensor-core kernel forced (fa_decode_paged's kernel
    argument)."""
    _KERNEL["which"] = request.param
    yield request.param
    _KERNEL["which"] = "auto"


def _dev16(bits, dtype):
    tdt = torch.bfloat16 if dtype == inputs.BF16 else torch.float16
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt).cuda()


def _ulp(x, dtype):
    mant = 7 if dtype == inputs.BF16 else 10
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126 if dtype == inputs.BF16 else -14)
    return np.ldexp(1.0, (e - mant).astype(np.int64))


def run_gpu(inp, k_bits=None, v_bits=None):
    w = inp.workload
    q = _dev16(inp.q_bits, w.dtype)
    kc = _dev16(inp.k_bits if k_bits is None else k_bits, w.dtype)
    vc = _dev16(inp.v_bits if v_bits is None else v_bits, w.dtype)
    table = torch.from_numpy(inp.block_table).cuda()
    lens = torch.from_numpy(inp.seq_lens).cuda()
    o, lse = fa.decode_paged(q, kc, vc, table, lens, w.max_seq_len, scale=w.scale, mask=w.mask,
                             kernel=_KERNEL["which"])
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def check(inp):
    w = inp.workload
    o, lse = run_gpu(inp)
    qf, kf, vf = inp.f64()
    o_ref, lse_ref = oracle.attention_paged(qf, kf, vf, inp.block_table, inp.seq_lens, w.scale,
                                            w.mask)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    err = np.abs(o - o_ref)
    adj = np.maximum(err - 0.5 * _ulp(o_ref, w.dtype), 0.0)
    stats = dict(max=float(err.max()), max_adj=float(adj.max()), mean=float(err.mean()),
                 lse=float(np.abs(lse - lse_ref).max()))
    assert adj.max() <= MAX_TOL, stats
    if w.dtype == inputs.FP16:
        assert err.max() <= MAX_TOL, stats
    assert err.mean() <= MEAN_TOL, stats
    assert stats["lse"] <= LSE_TOL, stats
    return stats


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("dtype", [inputs.BF16, inputs.FP16])
@pytest.mark.parametrize("block_size", [16, 32, 64, 128])
@pytest.mark.parametrize("mask", ["none", "causal"])
def test_decode_one_row(d, dtype, block_size, mask):
    inp = inputs.custom_paged(5, 4, 2, 1, d, block_size, 700, dtype, mask, seed=block_size + d)
    print(check(inp))


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("H,Hkv,Sq", [(8, 8, 1), (8, 2, 4), (32, 1, 4), (16, 4, 3), (6, 3, 7)])
def test_decode_groups_and_several_rows(d, H, Hkv, Sq):
    # up to 128 packed rows per K/V head (32 heads x 4 rows on one K/V head)
    inp = inputs.custom_paged(3, H, Hkv, Sq, d, 16, 500, inputs.BF16, "causal", seed=H * Sq)
    print(check(inp))


def test_decode_many_key_ranges_and_short_requests():
    # one request, one K/V head, 4k tokens: one key range per 128-key tile;
    # the short requests of the second case leave most ranges empty
    print(check(inputs.custom_paged(1, 2, 1, 1, 128, 16, 4096, inputs.BF16, "causal", seed=3)))
    print(check(inputs.custom_paged(4, 4, 4, 2, 128, 64, 6000, inputs.FP16, "none", min_seq_len=2,
                                    seed=4)))


def test_decode_lengths_at_block_edges():
    for L in (1, 15, 16, 17, 127, 128, 129):
        inp = inputs.custom_paged(2, 2, 2, 1, 64, 16, L, inputs.BF16, "causal", min_seq_len=L,
                                  seed=L)
        assert np.all(inp.seq_lens == L)
        check(inp)


@pytest.mark.parametrize("d", [128, 256])
def test_decode_junk_in_unused_cache_slots_never_leaks(d):
    inp = inputs.custom_paged(3, 4, 4, 2, d, 16, 333, inputs.BF16, "causal", seed=7)
    o1, l1 = run_gpu(inp)
    kb, vb = inp.k_bits.copy(), inp.v_bits.copy()
    nan = np.uint16(0x7FC0)
    inf = np.uint16(0x7F80)
    used = {}
    for b, L in enumerate(inp.seq_lens):
        n = -(-int(L) // 16)
        for t in range(n):
            used[int(inp.block_table[b, t])] = (L - 16 * t) if t == n - 1 else 16
    for blk in range(kb.shape[0]):
        fill = used.get(blk, 0)
        kb[blk, :, fill:] = nan
        vb[blk, :, fill:] = inf
    o2, l2 = run_gpu(inp, kb, vb)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("bad", [-1, "past"])
def test_decode_out_of_range_table_entry_reads_zeros(bad):
    """A table entry outside [0, num_blocks) inside a request's blocks reads
    as a block of zeros: the result equals the oracle's on a pool with an
    all-zero block at that entry."""
    inp = inputs.custom_paged(3, 4, 2, 1, 128, 16, 300, inputs.BF16, "causal", min_seq_len=200,
                              seed=12)
    nb = inp.k_bits.shape[0]
    table = inp.block_table.copy()
    table[1, 2] = -1 if bad == -1 else nb + 5
    w = inp.workload
    q = _dev16(inp.q_bits, w.dtype)
    kc, vc = _dev16(inp.k_bits, w.dtype), _dev16(inp.v_bits, w.dtype)
    o, lse = fa.decode_paged(q, kc, vc, torch.from_numpy(table).cuda(),
                             torch.from_numpy(inp.seq_lens).cuda(), w.max_seq_len, scale=w.scale,
                             mask=w.mask, kernel=_KERNEL["which"])
    torch.cuda.synchronize()
    assert fa.device_error() == fa.FA_OK
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    # the same attention on a valid table: the entry points at an added zero block
    qf, kf, vf = inp.f64()
    zeros = np.zeros_like(kf[:1])
    kz, vz = np.concatenate([kf, zeros]), np.concatenate([vf, zeros])
    table_ref = inp.block_table.copy()
    table_ref[1, 2] = nb
    o_ref, lse_ref = oracle.attention_paged(qf, kz, vz, table_ref, inp.seq_lens, w.scale, w.mask)
    err = np.abs(o - o_ref)
    assert np.maximum(err - 0.5 * _ulp(o_ref, w.dtype), 0.0).max() <= MAX_TOL
    assert err.mean() <= MEAN_TOL and np.abs(lse - lse_ref).max() <= LSE_TOL


def test_decode_is_deterministic():
    inp = inputs.custom_paged(4, 8, 2, 1, 128, 32, 900, inputs.BF16, "causal", seed=8)
    a, b = run_gpu(inp), run_gpu(inp)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_decode_unsupported_requests_raise():
    t = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    ln = torch.ones(1, dtype=torch.int32, device="cuda")
    q = torch.zeros(1, 2, 1, 96, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 2, 16, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.decode_paged(q, kc, kc, t, ln, 16, kernel=_KERNEL["which"])
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    q = torch.zeros(1, 2, 1, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 2, 24, 128, dtype=torch.bfloat16, device="cuda")  # block of 24 tokens
    with pytest.raises(fa.FAError) as e:
        fa.decode_paged(q, kc, kc, t, ln, 16, kernel=_KERNEL["which"])
    assert e.value.status == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("idx", [0, 1])
def test_decode_workload_full_size(idx):
    w = inputs.PAGED_WORKLOADS[idx]
    inp = inputs.generate_paged(w)
    print(w.name, check(inp))
