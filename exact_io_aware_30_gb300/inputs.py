"""Seeded synthetic inputs shared by the GPU path's tests/bench and the oracle.

This module holds no attention arithmetic: it draws Q, K, V, rounds them to
the 16-bit storage type and hands out both the raw 16-bit patterns (for the
GPU library) and the exactly widened float64 values (for the CPU oracle).

Recipe (the same for every workload):
  * numpy ``Generator(PCG64(seed))``; Q, then K, then V drawn in that order
    with ``standard_normal(shape, dtype=float32)``, shape [B, H, S, d] (K and
    V: [B, Hkv, Sk, d], Hkv = H unless the workload shares K/V heads);
  * round-to-nearest-even to bf16 (or fp16 for the fp16 workload);
  * the "spiky keys" workload then picks, per (b, K/V head), round(0.01 * Sk)
    distinct key rows with ``rng.choice(Sk, n, replace=False)`` and multiplies
    them by 8 (a power of two: exact in both 16-bit types);
  * scale = 1/sqrt(d) as float32.

The five named workloads mirror the cases the pages discuss: a tiny
single-head case, a batched causal case, 8k tokens x 32 heads ("FlashAttention:
IO-aware attention kernels", section "Why you'd care"), an 18 000-token
document with d = 128 ("Flash attention and memory-efficient attention
variants", section "The wall you hit is not the one you expect"), and a
d = 256 case with rare large keys that force running-max jumps.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BF16 = "bf16"
FP16 = "fp16"


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Sk: int
    d: int
    dtype: str
    mask: str          # "none" | "causal" | "window"
    window: int = 0
    spiky_keys: bool = False
    seed: int = 0
    Hkv: int = 0       # K/V heads (grouped-query attention); 0 = H
    notes: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return float(np.float32(1.0) / np.sqrt(np.float32(self.d)))

    def shape_q(self):
        return (self.B, self.H, self.Sq, self.d)

    @property
    def kv_heads(self) -> int:
        return self.Hkv if self.Hkv > 0 else self.H

    def shape_kv(self):
        return (self.B, self.kv_heads, self.Sk, self.d)


# The five workloads, indexed 0..4; seed = 1001 + index.
WORKLOADS = [
    Workload("tiny_b1h1_s256_d64_bf16_nomask", 1, 1, 256, 256, 64, BF16, "none", seed=1001),
    Workload("b4h16_s2048_d128_bf16_causal", 4, 16, 2048, 2048, 128, BF16, "causal", seed=1002),
    Workload("b1h32_s8192_d128_fp16_causal", 1, 32, 8192, 8192, 128, FP16, "causal", seed=1003),
    Workload("b1h16_s18000_d128_bf16_window4096", 1, 16, 18000, 18000, 128, BF16, "window",
             window=4096, seed=1004),
    Workload("b2h8_s4096_d256_bf16_nomask_spikykeys", 2, 8, 4096, 4096, 256, BF16, "none",
             spiky_keys=True, seed=1005),
]


# Further forward workloads, by name: the 8k x 32-head causal case in bf16
# (the same draws as the fp16 one, rounded to bf16), and a d = 64 case with
# the same flops (twice the heads at half the head dimension).
EXTRA_WORKLOADS = [
    Workload("b1h32_s8192_d128_bf16_causal", 1, 32, 8192, 8192, 128, BF16, "causal", seed=1003),
    Workload("b1h64_s8192_d64_bf16_causal", 1, 64, 8192, 8192, 64, BF16, "causal", seed=1006),
]


def workload(index_or_name) -> Workload:
    if isinstance(index_or_name, int):
        return WORKLOADS[index_or_name]
    for w in WORKLOADS + EXTRA_WORKLOADS:
        if w.name == index_or_name:
            return w
    raise KeyError(index_or_name)


def with_dtype(w: Workload, dtype: str) -> Workload:
    """The same workload (same seed, so the same draws) rounded to another
    16-bit type; the name's type tag follows."""
    if dtype == w.dtype:
        return w
    name = w.name.replace(f"_{w.dtype}_", f"_{dtype}_")
    if name == w.name:
        name = f"{w.name}_{dtype}"
    return Workload(name, w.B, w.H, w.Sq, w.Sk, w.d, dtype, w.mask, w.window, w.spiky_keys,
                    w.seed, w.Hkv)


# ----------------------------------------------------------------------------
# 16-bit encodings (storage conversions only)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    rounded = b + np.uint32(0x7FFF) + lsb
    out = (rounded >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f32_to_fp16_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def fp16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == BF16 else f32_to_fp16_bits(x)


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f64(bits) if dtype == BF16 else fp16_bits_to_f64(bits)


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 values of x after rounding to the 16-bit type."""
    return bits_to_f64(to_bits(np.asarray(x, dtype=np.float32), dtype), dtype)


# ----------------------------------------------------------------------------
# Generators
# ----------------------------------------------------------------------------

@dataclass
class Inputs:
    workload: Workload
    q_bits: np.ndarray   # uint16 [B,H,Sq,d]
    k_bits: np.ndarray   # uint16 [B,Hkv,Sk,d]
    v_bits: np.ndarray   # uint16 [B,Hkv,Sk,d]

    def f64(self):
        dt = self.workload.dtype
        return (bits_to_f64(self.q_bits, dt), bits_to_f64(self.k_bits, dt),
                bits_to_f64(self.v_bits, dt))


def generate(w: Workload, seed: int | None = None) -> Inputs:
    """Draw one workload's Q, K, V by the recipe in the module docstring."""
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    q = rng.standard_normal(w.shape_q(), dtype=np.float32)
    k = rng.standard_normal(w.shape_kv(), dtype=np.float32)
    v = rng.standard_normal(w.shape_kv(), dtype=np.float32)
    qb, kb, vb = to_bits(q, w.dtype), to_bits(k, w.dtype), to_bits(v, w.dtype)
    del q, k, v
    if w.spiky_keys:
        n = int(round(0.01 * w.Sk))
        kf = bits_to_f64(kb, w.dtype)
        for b in range(w.B):
            for h in range(w.kv_heads):
                rows = rng.choice(w.Sk, n, replace=False)
                kf[b, h, rows, :] *= 8.0
        kb = to_bits(kf.astype(np.float32), w.dtype)
    return Inputs(w, qb, kb, vb)


def grad_output(w: Workload, seed: int | None = None) -> np.ndarray:
    """dO for the backward, [B, H, Sq, d]: standard normal float32 from
    ``PCG64(seed + 500)`` (seed = the workload's), rounded to the 16-bit type;
    returns the 16-bit patterns."""
    rng = np.random.Generator(np.random.PCG64((w.seed if seed is None else seed) + 500))
    return to_bits(rng.standard_normal(w.shape_q(), dtype=np.float32), w.dtype)


def custom(B, H, Sq, Sk, d, dtype=BF16, mask="none", window=0, seed=0, spiky_keys=False,
           name="custom", Hkv=0) -> Inputs:
    """An ad-hoc shape drawn by the same recipe (Hkv > 0: K/V with Hkv heads)."""
    w = Workload(name, B, H, Sq, Sk, d, dtype, mask, window, spiky_keys, seed, Hkv)
    return generate(w)


# ----------------------------------------------------------------------------
# Paged K/V cache (decoding)
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class PagedWorkload:
    """Decoding over a paged cache: B requests, each with seq_len cached tokens
    in blocks of block_size tokens (the last Sq of them the new rows')."""
    name: str
    B: int
    H: int
    Hkv: int
    Sq: int
    d: int
    block_size: int
    max_seq_len: int
    dtype: str
    mask: str = "causal"
    min_seq_len: int = 1
    seed: int = 0
    spare_blocks: int = 8   # blocks in the pool that no request uses

    @property
    def scale(self) -> float:
        return float(np.float32(1.0) / np.sqrt(np.float32(self.d)))


# Decoding for a 13B model shaped like OPT-13B (40 heads x 128 = hidden 5120,
# fp16), cache blocks of 16 tokens and a 2,048-token context window, as the
# paged-cache section of "Flash attention and memory-efficient attention
# variants" describes it; 128 concurrent requests with lengths spread
# uniformly over the window.
PAGED_WORKLOADS = [
    PagedWorkload("decode_b128_h40_d128_bs16_ctx2048_fp16", 128, 40, 40, 1, 128, 16, 2048, FP16,
                  seed=2001),
    PagedWorkload("decode_b64_h32kv8_d128_bs64_ctx8192_bf16", 64, 32, 8, 1, 128, 64, 8192, BF16,
                  seed=2002),
]


@dataclass
class PagedInputs:
    workload: PagedWorkload
    q_bits: np.ndarray        # uint16 [B, H, Sq, d]
    k_bits: np.ndarray        # uint16 [num_blocks, Hkv, block_size, d]
    v_bits: np.ndarray        # uint16 [num_blocks, Hkv, block_size, d]
    block_table: np.ndarray   # int32 [B, max_blocks]
    seq_lens: np.ndarray      # int32 [B]

    def f64(self):
        dt = self.workload.dtype
        return (bits_to_f64(self.q_bits, dt), bits_to_f64(self.k_bits, dt),
                bits_to_f64(self.v_bits, dt))


def generate_paged(w: PagedWorkload) -> PagedInputs:
    """Seeded paged-cache inputs: lengths uniform in [max(Sq, min_seq_len),
    max_seq_len] (the first request gets max_seq_len), each request's blocks
    a random set of physical blocks (a permutation of the pool), table
    entries past a request's blocks set to -1; then Q, K cache, V cache drawn
    N(0, 1) float32 and rounded to the 16-bit type."""
    rng = np.random.Generator(np.random.PCG64(w.seed))
    lo = max(w.Sq, w.min_seq_len)
    lens = rng.integers(lo, w.max_seq_len + 1, size=w.B).astype(np.int32)
    lens[0] = w.max_seq_len
    max_blocks = -(-w.max_seq_len // w.block_size)
    need = [-(-int(L) // w.block_size) for L in lens]
    num_blocks = sum(need) + w.spare_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    table = np.full((w.B, max_blocks), -1, np.int32)
    used = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[used:used + n]
        used += n
    q = to_bits(rng.standard_normal((w.B, w.H, w.Sq, w.d), dtype=np.float32), w.dtype)
    shape = (num_blocks, w.Hkv, w.block_size, w.d)
    k = to_bits(rng.standard_normal(shape, dtype=np.float32), w.dtype)
    v = to_bits(rng.standard_normal(shape, dtype=np.float32), w.dtype)
    return PagedInputs(w, q, k, v, table, lens)


def custom_paged(B, H, Hkv, Sq, d, block_size, max_seq_len, dtype=BF16, mask="causal",
                 min_seq_len=1, seed=0) -> PagedInputs:
    return generate_paged(PagedWorkload("custom_paged", B, H, Hkv, Sq, d, block_size,
                                        max_seq_len, dtype, mask, min_seq_len, seed))


# ----------------------------------------------------------------------------
# 8-bit (e4m3) inputs
# ----------------------------------------------------------------------------

def e4m3_table() -> np.ndarray:
    """float64 value of every e4m3 code (1 sign, 4 exponent bits with bias 7,
    3 mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448)."""
    codes = np.arange(256)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e = (codes >> 3) & 0xF
    m = codes & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    val = sign * val
    val[(e == 15) & (m == 7)] = np.nan
    return val


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to the even code), saturating
    at +-448; uint8 codes."""
    tab = e4m3_table()
    pos = tab[:0x7F]                  # codes 0x00 .. 0x7E: 0 .. 448, increasing
    a = np.minimum(np.abs(np.asarray(x, dtype=np.float64)), 448.0)
    hi = np.clip(np.searchsorted(pos, a, side="left"), 1, len(pos) - 1)
    lo = hi - 1
    dlo, dhi = a - pos[lo], pos[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a == pos[hi], hi, pick)
    code = pick.astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def e4m3_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return e4m3_table()[np.asarray(bits, dtype=np.uint8)]


@dataclass(frozen=True)
class Fp8Workload:
    name: str
    B: int
    H: int
    Hkv: int
    Sq: int
    Sk: int
    d: int
    mask: str
    window: int = 0
    seed: int = 0

    @property
    def scale(self) -> float:
        return float(np.float32(1.0) / np.sqrt(np.float32(self.d)))


@dataclass
class Fp8Inputs:
    workload: Fp8Workload
    q_bits: np.ndarray    # uint8 e4m3 [B, H, Sq, d]
    k_bits: np.ndarray    # uint8 e4m3 [B, Hkv, Sk, d]
    vt_bits: np.ndarray   # uint8 e4m3 [B, Hkv, d, Sk] (V transposed)
    q_descale: float
    k_descale: float
    v_descale: float

    def f64(self):
        """Dequantised q, k, v (v as [B, Hkv, Sk, d])."""
        q = e4m3_bits_to_f64(self.q_bits) * self.q_descale
        k = e4m3_bits_to_f64(self.k_bits) * self.k_descale
        v = e4m3_bits_to_f64(self.vt_bits).transpose(0, 1, 3, 2) * self.v_descale
        return q, k, np.ascontiguousarray(v)


def generate_fp8(w: Fp8Workload) -> Fp8Inputs:
    """Q, then K, then V drawn N(0, 1) float32 from PCG64(seed); each tensor
    quantised to e4m3 with one factor, descale = max|x| / 448 (a power of two
    above it, so that the factor is exact); V stored transposed."""
    rng = np.random.Generator(np.random.PCG64(w.seed))
    out = []
    for shape in ((w.B, w.H, w.Sq, w.d), (w.B, w.Hkv, w.Sk, w.d), (w.B, w.Hkv, w.Sk, w.d)):
        x = rng.standard_normal(shape, dtype=np.float32)
        amax = float(np.abs(x).max()) if x.size else 1.0
        descale = float(2.0 ** np.ceil(np.log2(max(amax, 1e-30) / 448.0)))
        out.append((f32_to_e4m3_bits(x / descale), descale))
    (qb, qs), (kb, ks), (vb, vs) = out
    vt = np.ascontiguousarray(vb.transpose(0, 1, 3, 2))
    return Fp8Inputs(w, qb, kb, vt, qs, ks, vs)


# The 8k-token causal shape in 8 bits; heads x d fixed at 4096 across the
# three head dimensions, so the three do the same number of flops.
FP8_WORKLOADS = [
    Fp8Workload("fp8_b1h32_s8192_d128_causal", 1, 32, 32, 8192, 8192, 128, "causal", seed=3001),
    Fp8Workload("fp8_b1h64_s8192_d64_causal", 1, 64, 64, 8192, 8192, 64, "causal", seed=3002),
    Fp8Workload("fp8_b1h16_s8192_d256_causal", 1, 16, 16, 8192, 8192, 256, "causal", seed=3003),
]
