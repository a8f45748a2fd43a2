"""The C-ABI library builds, loads and exports what include/fa.h declares, and
rejects invalid calls synchronously -- all without a GPU (no compute call is
made: every call here fails validation before touching the device)."""
import os
import re

import pytest

from exact_io_aware_30_gb300 import build, fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_documented_entry_points():
    assert _declared_functions() == sorted(fa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_library_is_sm103a_only():
    # one -gencode, sm_103a; the oracle is never linked into it
    assert build.ARCH_FLAGS == ["-gencode", "arch=compute_103a,code=sm_103a"]
    with open(build.LIB_PATH, "rb") as f:
        blob = f.read()
    assert b"oracle_attn" not in blob


def test_status_strings(lib):
    for code in range(6):
        s = fa.status_string(code)
        assert s.startswith("FA_")
    assert fa.status_string(99) == "FA_ERR_UNKNOWN"


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("mask", ["none", "causal", "window"])
@pytest.mark.parametrize("dtype", [fa.DTYPE_BF16, fa.DTYPE_FP16])
def test_describe_names_the_kernel(lib, d, mask, dtype):
    s = fa.describe(d, mask, dtype)
    assert f"d={d}" in s and "tcgen05" in s
    assert ("fp16" if dtype == fa.DTYPE_FP16 else "bf16") in s


def test_describe_rejects_unsupported(lib):
    with pytest.raises(fa.FAError) as e:
        fa.describe(96, "none")
    assert e.value.status == fa.FA_ERR_UNSUPPORTED


FAKE = 0x7F0000001000  # 16-byte aligned, never dereferenced: validation fails first


def _fwd(**kw):
    a = dict(q_ptr=FAKE, k_ptr=FAKE + (1 << 30), v_ptr=FAKE + (2 << 30), o_ptr=FAKE + (3 << 30),
             lse_ptr=FAKE + (4 << 30), B=1, H=1, Sq=128, Sk=128, d=128, scale=0.088,
             mask_kind=fa.MASK_NONE, window=0, stream=0, dtype=fa.DTYPE_BF16)
    a.update(kw)
    return fa.fwd_raw(**a)


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(d=512), fa.FA_ERR_UNSUPPORTED),
    (dict(mask_kind=3), fa.FA_ERR_UNSUPPORTED),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=-1), fa.FA_ERR_INVALID_ARG),
    (dict(Sk=0), fa.FA_ERR_INVALID_ARG),
    (dict(Sq=-1), fa.FA_ERR_INVALID_ARG),
    (dict(mask_kind=fa.MASK_SLIDING_WINDOW, window=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-0.5), fa.FA_ERR_INVALID_ARG),
    (dict(q_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(q_ptr=FAKE + 8), fa.FA_ERR_MISALIGNED),
    (dict(o_ptr=FAKE + (3 << 30) + 2), fa.FA_ERR_MISALIGNED),
    (dict(lse_ptr=FAKE + (4 << 30) + 2), fa.FA_ERR_MISALIGNED),
    (dict(o_ptr=FAKE + 64), fa.FA_ERR_INVALID_ARG),                # o overlaps q
    (dict(lse_ptr=FAKE + (3 << 30) + 1024), fa.FA_ERR_INVALID_ARG),  # lse inside o
    (dict(B=1 << 16, H=1 << 16), fa.FA_ERR_INVALID_ARG),             # unit count overflows
])
def test_invalid_calls_are_rejected_before_launch(lib, kw, status):
    for dt in (fa.DTYPE_BF16, fa.DTYPE_FP16):
        kw2 = dict(kw)
        kw2.setdefault("dtype", dt)
        assert _fwd(**kw2) == status


def _fwd_gqa(**kw):
    a = dict(q_ptr=FAKE, k_ptr=FAKE + (1 << 30), v_ptr=FAKE + (2 << 30), o_ptr=FAKE + (3 << 30),
             lse_ptr=FAKE + (4 << 30), B=1, H=4, H_kv=2, Sq=128, Sk=128, d=128, scale=0.088,
             mask_kind=fa.MASK_NONE, window=0, stream=0, dtype=fa.DTYPE_BF16)
    a.update(kw)
    return fa.fwd_gqa_raw(**a)


@pytest.mark.parametrize("kw,status", [
    (dict(H=3, H_kv=2), fa.FA_ERR_INVALID_ARG),      # H_kv must divide H
    (dict(H_kv=0), fa.FA_ERR_INVALID_ARG),
    (dict(H_kv=-2), fa.FA_ERR_INVALID_ARG),
    (dict(H=2, H_kv=4), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=2), fa.FA_ERR_UNSUPPORTED),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(mask_kind=fa.MASK_SLIDING_WINDOW, window=0), fa.FA_ERR_INVALID_ARG),
    (dict(k_ptr=FAKE + (1 << 30) + 8), fa.FA_ERR_MISALIGNED),
    # o overlaps the (smaller) K block: [B, H_kv, Sk, d] = 64 KiB from k_ptr
    (dict(o_ptr=FAKE + (1 << 30) + 65536 - 16), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
])
def test_gqa_invalid_calls_are_rejected_before_launch(lib, kw, status):
    assert _fwd_gqa(**kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Sk=0), fa.FA_ERR_INVALID_ARG),
    (dict(q_ptr=FAKE + 8), fa.FA_ERR_MISALIGNED),
    (dict(o_ptr=FAKE + 64), fa.FA_ERR_INVALID_ARG),
])
def test_gqa_entry_with_equal_heads_validates_like_fa_fwd(lib, kw, status):
    for dt in (fa.DTYPE_BF16, fa.DTYPE_FP16):
        kw2 = dict(kw, dtype=dt)
        assert _fwd(**kw2) == status
        assert _fwd_gqa(H=1, H_kv=1, **kw2) == status


@pytest.mark.parametrize("args,status", [
    ((1, 1, 128, 128, 96, "none", 0, 0), fa.FA_ERR_UNSUPPORTED),
    ((1, 1, 128, 128, 128, "none", 0, 5), fa.FA_ERR_UNSUPPORTED),
    ((0, 1, 128, 128, 128, "none", 0, 0), fa.FA_ERR_INVALID_ARG),
    ((1, 1, 128, 128, 128, "window", 0, 0), fa.FA_ERR_INVALID_ARG),
])
def test_workspace_query_matches_fwd_status(lib, args, status):
    st, nbytes = fa.workspace_query(*args)
    assert st == status
    assert nbytes == 0
    B, H, Sq, Sk, d, mask, window, dtype = args
    if dtype not in (fa.DTYPE_BF16, fa.DTYPE_FP16):
        return  # the dtype is implied by the fa_fwd / fa_fwd_fp16 symbol
    assert _fwd(B=B, H=H, Sq=Sq, Sk=Sk, d=d, mask_kind=fa.mask_code(mask), window=window,
                dtype=dtype) == status


def test_python_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(fa.FAError):
        fa.forward(q, q, q)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(fa.FAError):
        fa.load(str(tmp_path / "libfa.so"))


def _bwd(**kw):
    g = 1 << 30
    a = dict(q_ptr=FAKE, k_ptr=FAKE + g, v_ptr=FAKE + 2 * g, o_ptr=FAKE + 3 * g,
             lse_ptr=FAKE + 4 * g, do_ptr=FAKE + 5 * g, dq_ptr=FAKE + 6 * g, dk_ptr=FAKE + 7 * g,
             dv_ptr=FAKE + 8 * g, ws_ptr=FAKE + 9 * g, ws_bytes=1 << 20, B=1, H=4, H_kv=2,
             Sq=128, Sk=128, d=128, scale=0.088, mask_kind=fa.MASK_CAUSAL, window=0, stream=0,
             dtype=fa.DTYPE_BF16)
    a.update(kw)
    return fa.bwd_raw(**a)


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=512), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=3), fa.FA_ERR_UNSUPPORTED),
    (dict(mask_kind=4), fa.FA_ERR_UNSUPPORTED),
    (dict(H=3, H_kv=2), fa.FA_ERR_INVALID_ARG),
    (dict(H_kv=0), fa.FA_ERR_INVALID_ARG),
    (dict(Sk=0), fa.FA_ERR_INVALID_ARG),
    (dict(mask_kind=fa.MASK_SLIDING_WINDOW, window=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(ws_bytes=2 * 4 * 4 * 128 - 4), fa.FA_ERR_INVALID_ARG),   # one float short
    (dict(ws_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(dq_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws_ptr=FAKE + 9 * (1 << 30) + 16), fa.FA_ERR_MISALIGNED),  # workspace wants 256 B
    (dict(do_ptr=FAKE + 5 * (1 << 30) + 8), fa.FA_ERR_MISALIGNED),
    (dict(lse_ptr=FAKE + 4 * (1 << 30) + 2), fa.FA_ERR_MISALIGNED),
    (dict(dq_ptr=FAKE + 64), fa.FA_ERR_INVALID_ARG),                 # dq overlaps q
    (dict(dv_ptr=FAKE + 7 * (1 << 30) + 4096), fa.FA_ERR_INVALID_ARG),  # dv overlaps dk
    (dict(ws_ptr=FAKE + 8 * (1 << 30)), fa.FA_ERR_INVALID_ARG),       # workspace on dv
])
def test_bwd_invalid_calls_are_rejected_before_launch(lib, kw, status):
    assert _bwd(**kw) == status


def test_bwd_workspace_query_sizes(lib):
    # rejected sizes report their status and 0 bytes, before any device query
    assert fa.bwd_workspace_query(1, 4, 2, 128, 128, 96) == (fa.FA_ERR_UNSUPPORTED, 0)
    assert fa.bwd_workspace_query(1, 3, 2, 128, 128, 128) == (fa.FA_ERR_INVALID_ARG, 0)
    assert fa.bwd_workspace_query(1, 4, 2, 128, 128, 128, "window", 0) == (fa.FA_ERR_INVALID_ARG, 0)


def _dec(**kw):
    g = 1 << 30
    a = dict(q_ptr=FAKE, k_ptr=FAKE + g, v_ptr=FAKE + 2 * g, table_ptr=FAKE + 3 * g,
             lens_ptr=FAKE + 4 * g, o_ptr=FAKE + 5 * g, lse_ptr=FAKE + 6 * g, ws_ptr=FAKE + 7 * g,
             ws_bytes=1 << 24, B=2, H=8, H_kv=2, Sq=1, d=128, block_size=16, max_blocks=64,
             num_blocks=128, max_seq_len=1024, scale=0.088, mask_kind=fa.MASK_CAUSAL,
             dtype=fa.DTYPE_BF16, stream=0)
    a.update(kw)
    return fa.decode_raw(**a)


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=2), fa.FA_ERR_UNSUPPORTED),
    (dict(mask_kind=fa.MASK_SLIDING_WINDOW), fa.FA_ERR_UNSUPPORTED),  # decode: none or causal
    (dict(block_size=24), fa.FA_ERR_UNSUPPORTED),
    (dict(block_size=256, max_blocks=4), fa.FA_ERR_UNSUPPORTED),
    (dict(H=64, H_kv=1, Sq=4), fa.FA_ERR_UNSUPPORTED),                # 256 packed rows > 128
    (dict(H=3, H_kv=2), fa.FA_ERR_INVALID_ARG),
    (dict(Sq=0), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(num_blocks=0), fa.FA_ERR_INVALID_ARG),
    (dict(max_seq_len=64 * 16 + 1), fa.FA_ERR_INVALID_ARG),            # beyond the table
    (dict(Sq=2, max_seq_len=1), fa.FA_ERR_INVALID_ARG),                # fewer tokens than rows
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(table_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(q_ptr=FAKE + 8), fa.FA_ERR_MISALIGNED),
    (dict(lens_ptr=FAKE + 4 * (1 << 30) + 2), fa.FA_ERR_MISALIGNED),
    (dict(ws_ptr=FAKE + 7 * (1 << 30) + 16), fa.FA_ERR_MISALIGNED),     # workspace wants 256 B
])
def test_decode_invalid_calls_are_rejected_before_launch(lib, kw, status):
    assert _dec(**kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(kernel=7), fa.FA_ERR_UNSUPPORTED),                         # no such kernel choice
    (dict(kernel=-1), fa.FA_ERR_UNSUPPORTED),
    (dict(kernel=fa.DECODE_CUDA_CORES), fa.FA_ERR_UNSUPPORTED),      # 4 rows per K/V head > 2
])
def test_decode_kernel_choice_is_checked(lib, kw, status):
    assert _dec(**kw) == status


def test_decode_workspace_query_sizes(lib):
    # rejected sizes report their status and 0 bytes, before any device query
    q = fa.decode_workspace_query
    assert q(2, 8, 2, 1, 96, 16, 64, 128, 1024) == (fa.FA_ERR_UNSUPPORTED, 0)
    assert q(2, 8, 2, 1, 128, 24, 64, 128, 1024) == (fa.FA_ERR_UNSUPPORTED, 0)
    assert q(2, 64, 1, 4, 128, 16, 64, 128, 1024) == (fa.FA_ERR_UNSUPPORTED, 0)
    assert q(2, 3, 2, 1, 128, 16, 64, 128, 1024) == (fa.FA_ERR_INVALID_ARG, 0)
    assert q(2, 8, 2, 1, 128, 16, 64, 128, 2048) == (fa.FA_ERR_INVALID_ARG, 0)


def _fp8(**kw):
    g = 1 << 30
    a = dict(q_ptr=FAKE, k_ptr=FAKE + g, vt_ptr=FAKE + 2 * g, o_ptr=FAKE + 3 * g,
             lse_ptr=FAKE + 4 * g, B=1, H=4, H_kv=2, Sq=256, Sk=256, d=128, scale=0.088,
             q_descale=1.0, k_descale=1.0, v_descale=1.0, mask_kind=fa.MASK_CAUSAL, window=0,
             stream=0)
    a.update(kw)
    return fa.fwd_fp8_raw(**a)


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=512), fa.FA_ERR_UNSUPPORTED),
    (dict(mask_kind=3), fa.FA_ERR_UNSUPPORTED),
    (dict(H=3, H_kv=2), fa.FA_ERR_INVALID_ARG),
    (dict(Sk=0), fa.FA_ERR_INVALID_ARG),
    (dict(Sk=200), fa.FA_ERR_INVALID_ARG),                              # V^T rows: 16-byte multiples
    (dict(mask_kind=fa.MASK_SLIDING_WINDOW, window=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(k_descale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(v_descale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(q_descale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(vt_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(q_ptr=FAKE + 8), fa.FA_ERR_MISALIGNED),
    (dict(lse_ptr=FAKE + 4 * (1 << 30) + 2), fa.FA_ERR_MISALIGNED),
    (dict(o_ptr=FAKE + 64), fa.FA_ERR_INVALID_ARG),                     # o overlaps q
    (dict(Sq=0, q_ptr=0, o_ptr=0), fa.FA_OK),                          # no rows: nothing to do
])
def test_fp8_invalid_calls_are_rejected_before_launch(lib, kw, status):
    assert _fp8(**kw) == status


def _host(**kw):
    g = 1 << 30
    a = dict(q_ptr=FAKE, k_ptr=FAKE + g, v_ptr=FAKE + 2 * g, o_ptr=FAKE + 3 * g,
             lse_ptr=FAKE + 4 * g, ws_ptr=FAKE + 5 * g, ws_bytes=1 << 30, B=1, H=4, H_kv=2,
             Sq=300, Sk=300, d=128, scale=0.088, mask_code_=fa.MASK_CAUSAL, window=0,
             dtype=fa.DTYPE_BF16, stream_ptr=0)
    a.update(kw)
    return fa.fwd_host_raw(**a)


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=2), fa.FA_ERR_UNSUPPORTED),
    (dict(mask_code_=5), fa.FA_ERR_UNSUPPORTED),
    (dict(H=3), fa.FA_ERR_INVALID_ARG),                       # H_kv does not divide H
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Sk=0), fa.FA_ERR_INVALID_ARG),
    (dict(mask_code_=fa.MASK_SLIDING_WINDOW, window=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(q_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws_ptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws_bytes=1000), fa.FA_ERR_INVALID_ARG),              # workspace too small
    (dict(ws_ptr=FAKE + 5 * (1 << 30) + 128), fa.FA_ERR_MISALIGNED),
    (dict(Sq=0, q_ptr=0, ws_ptr=0), fa.FA_OK),                 # nothing to do
])
def test_host_invalid_calls_are_rejected_before_any_copy(lib, kw, status):
    assert _host(**kw) == status


def test_host_workspace_query_sizes(lib):
    # Q, K, V, O and lse, each rounded up to 256 bytes; rejected sizes give 0
    assert fa.host_workspace_query(1, 4, 2, 300, 300, 96) == (fa.FA_ERR_UNSUPPORTED, 0)
    assert fa.host_workspace_query(1, 3, 2, 300, 300, 128) == (fa.FA_ERR_INVALID_ARG, 0)


def test_debug_stall_hook_range(lib):
    # the test hook is set explicitly (no environment variable); off by default
    assert lib.fa_set_debug_stall_ms(-1) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_set_debug_stall_ms(10001) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_set_debug_stall_ms(0) == fa.FA_OK
