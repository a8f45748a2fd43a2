// fa_fp8_kernel.cuh -- the fused attention forward with 8-bit (e4m3) inputs,
// for sm_103a (GB300): the low-precision path that "FlashAttention: IO-aware
// attention kernels" (section "Concept") names as a later variant.  The
// arithmetic is that of the tiled forward pass ("FlashAttention: Why Tiling
// Attention Makes Transformers Fast Without Changing the Result", sections
// "Online softmax: correct as you go" and "The tiled forward pass").
//
// Inputs are e4m3 codes with one dequantisation factor per tensor: the value
// of a stored code x is x * q_descale (k_descale, v_descale).  The kernel
// computes S = Q K^T on the 8-bit tensor path (kind::f8f6f4, fp32
// accumulation) with the factors and 1/sqrt(d)-type scale folded into the
// exponent's multiplier, keeps a running reference max, sum and unnormalised
// O per row, and stores P as e4m3 for O += P V on the same 8-bit path.  The
// reference moves (and O is rescaled) only when a tile's max exceeds it by
// more than 2^4, as the forward defers rescaling; weights, at most 2^4, are
// stored times 2^4 (at most 256, inside e4m3's range of 448).  O is written
// as bf16, lse in fp32.
//
// V is taken transposed, [B, H_kv, d, Sk]: both tile products then read
// K-major operands (keys contiguous for V^T), the operand layout every 8-bit
// tcgen05 form accepts.
//
// One CTA per 128-row query tile (longest first); warps 0-3 softmax and
// epilogue (one row per thread), warp 4 issues the MMAs, warp 5 the TMA
// copies (Q once, K and V^T tiles through rings).  The tile width, the
// number of S buffers in tensor memory and so the CTAs per SM are chosen per
// head dimension (Fp8Pick below).
#pragma once

#include <math.h>
#include <stdint.h>

#include "fa_bwd_kernel.cuh"

namespace fa {

struct Fp8Params {
    CUtensorMap tm_q;   // e4m3 [B, H, Sq, d], box {min(d, 128), 128 rows}
    CUtensorMap tm_k;   // e4m3 [B, Hkv, Sk, d], box {min(d, 128), BN keys}
    CUtensorMap tm_vt;  // e4m3 [B, Hkv, d, Sk], box {BN keys, d rows}
    void *o;            // bf16 [B, H, Sq, d]
    float *lse;         // fp32 [B, H, Sq]
    int B, H, Hkv, kv_group, Sq, Sk;
    int mask_kind, window;
    float c;            // scale * q_descale * k_descale * log2(e), kept positive
    float o_mul;        // v_descale (the weights' stored factor cancels in O / l)
    int n_qtiles;
    uint64_t wait_limit_ns;
    int stall_test;     // test only: the softmax's first wait is on a barrier nothing completes
};

// Shared-memory descriptor of a K-major operand whose rows are 64 bytes,
// stored with the 64-byte swizzle (8-row atoms of 512 bytes).
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(512 >> 4) << 32) |
           (1ull << 46) | (4ull << 61);
}

// Tiling, for head dimension D, BN keys per tile and NS S buffers:
//  - Q and K rows are split into column chunks of at most 128 bytes (one
//    swizzle atom row): d = 64 one 64-byte chunk (64-byte swizzle), d = 128
//    one chunk, d = 256 two chunks stored one after the other.  V^T rows are
//    BN keys (BN bytes) wide, with the swizzle of that width;
//  - tensor memory holds NS S buffers of BN columns, then O (D columns); P
//    (BN keys of e4m3, BN/4 columns) is written over the first columns of
//    its tile's S buffer once the softmax has read S.  A CTA whose layout
//    fits 256 columns shares its SM with a second CTA; otherwise it takes
//    all 512;
//  - with two S buffers, S of tile t+1 is issued before P V of tile t, so
//    the tensor core works while the softmax runs; with one, a CTA's next S
//    waits for its P V and only the other CTA on the SM fills the gap.
template <int D_, int BN_, int NS_>
struct Fp8Cfg {
    static constexpr int D = D_;
    static constexpr int BN = BN_;
    static constexpr int NS = NS_;
    static_assert(D == 64 || D == 128 || D == 256, "d = 64, 128 or 256");
    static_assert(BN == 64 || BN == 128, "64- or 128-key tiles");
    static_assert(NS == 1 || NS == 2, "one or two S buffers");
    static constexpr int CHUNK = D < 128 ? D : 128;          // bytes of a Q/K row in one chunk
    static constexpr int NCHUNK = D / CHUNK;
    static constexpr int Q_CHUNK_BYTES = 128 * CHUNK;          // one 128-row Q chunk
    static constexpr int K_CHUNK_BYTES = BN * CHUNK;           // one BN-row K chunk
    static constexpr int Q_BYTES = 128 * D;
    static constexpr int TILE_BYTES = BN * D;  // K tile, or V^T tile (d rows x BN keys)
    static constexpr uint32_t TMEM_COLS = (NS * BN + D <= 256) ? 256 : 512;
    static constexpr int CTAS_PER_SM = TMEM_COLS == 256 ? 2 : 1;
    static constexpr int KST = TILE_BYTES >= 16384 ? 3 : 4;
    static constexpr int VST = TILE_BYTES >= 16384 ? 2 : (BN == 128 ? 3 : 4);
    static constexpr int NUM_SOFTMAX = 128;
    static constexpr int MMA_WARP = 4;
    static constexpr int TMA_WARP = 5;
    static constexpr int NUM_THREADS = 192;
    static constexpr uint32_t S_COL = 0;  // buffer b at S_COL + b * BN
    static constexpr uint32_t O_COL = NS * BN;
    static constexpr int B_QFULL = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_KEMPTY = B_KFULL + KST;
    static constexpr int B_VFULL = B_KEMPTY + KST;
    static constexpr int B_VEMPTY = B_VFULL + VST;
    static constexpr int B_SFULL = B_VEMPTY + VST;  // per S buffer
    static constexpr int B_PFULL = B_SFULL + NS;    // per S buffer
    static constexpr int B_PFREE = B_PFULL + NS;    // per S buffer: P V done, the buffer is free again
    static constexpr int B_OFINAL = B_PFREE + NS;
    static constexpr int B_DRAIN = B_OFINAL + 1;
    static constexpr int B_NEVER = B_DRAIN + 1;  // no arrivals (the stall test's wait)
    static constexpr int NUM_BARS = B_NEVER + 1;
    static constexpr int SMEM_TILES = Q_BYTES + (KST + VST) * TILE_BYTES;
    static constexpr int SMEM_BYTES = 1024 + SMEM_TILES + NUM_BARS * 8 + 32;
    static constexpr float TAU = 4.f;     // log2 of the stale-reference slack
    static constexpr float P_LOG2 = 4.f;  // weights are stored times 2^P_LOG2 (<= 2^8)
    static_assert(CTAS_PER_SM * (SMEM_BYTES + 1024) <= 233472, "CTAs per SM");
    static_assert(O_COL + D <= TMEM_COLS, "O fits");

    // Q/K operand descriptor at byte address a (a chunk's base, plus the K step).
    static __device__ __forceinline__ uint64_t qk_desc(uint32_t a) {
        if constexpr (CHUNK == 64) return smem_desc_sw64(a);
        else return smem_desc(a, 16);
    }
    // V^T operand descriptor (rows of BN bytes).
    static __device__ __forceinline__ uint64_t vt_desc(uint32_t a) {
        if constexpr (BN == 64) return smem_desc_sw64(a);
        else return smem_desc(a, 16);
    }
};

// The tile choice per head dimension.
template <int D> struct Fp8Pick;
template <> struct Fp8Pick<64> { using C = Fp8Cfg<64, 64, 2>; };
template <> struct Fp8Pick<128> { using C = Fp8Cfg<128, 64, 2>; };
template <> struct Fp8Pick<256> { using C = Fp8Cfg<256, 128, 2>; };

struct Fp8Unit {
    int b, h, kvh, i0, lo, n;  // key tiles lo .. lo + n (BN keys each)
};

template <int BN>
__device__ __forceinline__ Fp8Unit decode_fp8_unit(const Fp8Params &p) {
    Fp8Unit u;
    const int BH = p.B * p.H;
    const int g = p.n_qtiles - 1 - (int)blockIdx.x / BH;  // longest query tiles first
    const int bh = (int)blockIdx.x % BH;
    u.b = bh / p.H;
    u.h = bh - u.b * p.H;
    u.kvh = u.h / p.kv_group;
    u.i0 = g * 128;
    const int row_end = min(u.i0 + 128, p.Sq);
    int key_end = p.Sk;
    if (p.mask_kind != kMaskNone) key_end = min(p.Sk, row_end);
    int key_beg = 0;
    if (p.mask_kind == kMaskWindow) key_beg = max(0, u.i0 - p.window + 1);
    if (key_beg < key_end) {
        u.lo = key_beg / BN;
        u.n = (key_end + BN - 1) / BN - u.lo;
    } else {
        u.lo = 0;
        u.n = 0;
    }
    return u;
}

template <class C>
__device__ void fp8_tma_role(const Fp8Params &p, const Fp8Unit &un, uint8_t *sQ, uint8_t *sK, uint8_t *sV,
                             uint32_t bars, Ctl *ctl) {
    const bool leader = ptx::lane_id() == 0;
    const uint64_t pol_kv = ptx::policy_evict_last();
    if (un.n == 0) return;
    if (leader) {
        const uint32_t fb = bar_addr(bars, C::B_QFULL);
        ptx::mbar_arrive_expect_tx(fb, C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCHUNK; ++c)
            ptx::tma_load_4d(ptx::smem_addr(sQ + c * C::Q_CHUNK_BYTES), &p.tm_q, fb, c * C::CHUNK, un.i0, un.h,
                             un.b, ptx::policy_evict_first());
    }
    int k_issued = 0, v_issued = 0;
    bool ok = true;
    for (int t = 0; t < un.n && ok; ++t) {
        const int k0 = (un.lo + t) * C::BN;
        const int ks = t % C::KST, vs = t % C::VST;
        if (!wait_warp_backoff(bar_addr(bars, C::B_KEMPTY + ks), ((t / C::KST) & 1) ^ 1, ctl, 61)) {
            ok = false;
            break;
        }
        if (leader) {
            const uint32_t fb = bar_addr(bars, C::B_KFULL + ks);
            ptx::mbar_arrive_expect_tx(fb, C::TILE_BYTES);
#pragma unroll
            for (int c = 0; c < C::NCHUNK; ++c)
                ptx::tma_load_4d(ptx::smem_addr(sK + ks * C::TILE_BYTES + c * C::K_CHUNK_BYTES), &p.tm_k, fb,
                                 c * C::CHUNK, k0, un.kvh, un.b, pol_kv);
        }
        __syncwarp();
        ++k_issued;
        if (!wait_warp_backoff(bar_addr(bars, C::B_VEMPTY + vs), ((t / C::VST) & 1) ^ 1, ctl, 62)) {
            ok = false;
            break;
        }
        if (leader) {
            const uint32_t fb = bar_addr(bars, C::B_VFULL + vs);
            ptx::mbar_arrive_expect_tx(fb, C::TILE_BYTES);
            ptx::tma_load_4d(ptx::smem_addr(sV + vs * C::TILE_BYTES), &p.tm_vt, fb, k0, 0, un.kvh, un.b, pol_kv);
        }
        __syncwarp();
        ++v_issued;
    }
    wait_bar_drain(bar_addr(bars, C::B_QFULL), 0);
    if (!ok) {
        for (int t = k_issued - C::KST > 0 ? k_issued - C::KST : 0; t < k_issued; ++t)
            wait_bar_drain(bar_addr(bars, C::B_KFULL + t % C::KST), (t / C::KST) & 1);
        for (int t = v_issued - C::VST > 0 ? v_issued - C::VST : 0; t < v_issued; ++t)
            wait_bar_drain(bar_addr(bars, C::B_VFULL + t % C::VST), (t / C::VST) & 1);
    }
}

// Issue order: with one S buffer, S(t) then P V(t); with two, S(t) then
// P V(t-1), so the next tile's scores are on the tensor core while the
// softmax turns this tile's into weights.
template <class C>
__device__ void fp8_mma_role(const Fp8Params &p, const Fp8Unit &un, uint8_t *sQ, uint8_t *sK, uint8_t *sV,
                             uint32_t bars, uint32_t tmem, Ctl *ctl) {
    constexpr int LAG = C::NS - 1;
    // e4m3 x e4m3 -> fp32 (type code 0 for both), both operands K-major
    constexpr uint32_t kIdescS = make_idesc(128, C::BN, true, false);
    constexpr uint32_t kIdescO = make_idesc(128, C::D, true, false);
    const bool leader = ptx::lane_id() == 0;
    const uint32_t q_addr = ptx::smem_addr(sQ);
    bool ok = un.n == 0 || wait_warp(bar_addr(bars, C::B_QFULL), 0, ctl, 63);
    for (int t = 0; ok && t < un.n + LAG; ++t) {
        if (t < un.n) {
            const int ks = t % C::KST, b = t % C::NS;
            if (!wait_warp(bar_addr(bars, C::B_KFULL + ks), (t / C::KST) & 1, ctl, 64)) {
                ok = false;
                break;
            }
            // P V of tile t - NS has read P out of this S buffer
            if (t >= C::NS &&
                !wait_warp(bar_addr(bars, C::B_PFREE + b), ((t - C::NS) / C::NS) & 1, ctl, 65)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            if (leader) {
                const uint32_t k_addr = ptx::smem_addr(sK + ks * C::TILE_BYTES);
                // 32 elements (32 bytes) per instruction inside a chunk's row
#pragma unroll
                for (int kk = 0; kk < C::D / 32; ++kk) {
                    const int chunk = (kk * 32) / C::CHUNK, within = (kk * 32) % C::CHUNK;
                    ptx::mma_ss_f8(tmem + C::S_COL + b * C::BN,
                                   C::qk_desc(q_addr + (uint32_t)(chunk * C::Q_CHUNK_BYTES + within)),
                                   C::qk_desc(k_addr + (uint32_t)(chunk * C::K_CHUNK_BYTES + within)), kIdescS,
                                   kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(bar_addr(bars, C::B_SFULL + b));
                ptx::mma_commit(bar_addr(bars, C::B_KEMPTY + ks));
            }
            __syncwarp();
        }
        const int u = t - LAG;
        if (u < 0) continue;
        const int vs = u % C::VST, b = u % C::NS;
        if (!wait_warp(bar_addr(bars, C::B_VFULL + vs), (u / C::VST) & 1, ctl, 66) ||
            !wait_warp(bar_addr(bars, C::B_PFULL + b), (u / C::NS) & 1, ctl, 67)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        if (leader) {
            // V^T tile: N = d rows of BN keys (BN bytes), K-major
            const uint32_t v_addr = ptx::smem_addr(sV + vs * C::TILE_BYTES);
#pragma unroll
            for (int kk = 0; kk < C::BN / 32; ++kk)
                ptx::mma_ts_f8(tmem + C::O_COL, tmem + C::S_COL + b * C::BN + kk * 8,
                               C::vt_desc(v_addr + (uint32_t)(kk * 32)), kIdescO, (u > 0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(bar_addr(bars, C::B_PFREE + b));
            ptx::mma_commit(bar_addr(bars, C::B_VEMPTY + vs));
            if (u + 1 == un.n) ptx::mma_commit(bar_addr(bars, C::B_OFINAL));
        }
        __syncwarp();
    }
    if (leader) ptx::mma_commit(bar_addr(bars, C::B_DRAIN));
    __syncwarp();
    wait_bar_drain(bar_addr(bars, C::B_DRAIN), 0);
}

template <class C>
__device__ void fp8_softmax_role(const Fp8Params &p, const Fp8Unit &un, uint32_t bars, uint32_t tmem,
                                 Ctl *ctl) {
    const int r = (int)threadIdx.x;
    const int warp = r >> 5;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int i = un.i0 + r;  // query row
    const float c = p.c;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < un.n; ++t) {
        const int k0 = (un.lo + t) * C::BN;
        const int b = t % C::NS;
        const uint32_t s_col = C::S_COL + b * C::BN;
        if (!wait_warp(bar_addr(bars, (p.stall_test && t == 0) ? C::B_NEVER : C::B_SFULL + b), (t / C::NS) & 1,
                       ctl, 68)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        uint32_t s[C::BN];
        ptx::tmem_ld_x32<0>(lane_base + s_col, s);
        ptx::tmem_ld_x32<32>(lane_base + s_col + 32, s);
        if constexpr (C::BN == 128) {
            ptx::tmem_ld_x32<64>(lane_base + s_col + 64, s);
            ptx::tmem_ld_x32<96>(lane_base + s_col + 96, s);
        }
        ptx::tmem_wait_ld();
        ptx::reg_fence<C::BN>(s);

        // key k0 + e is visible to row i iff lo <= e < hi
        int lo = 0, hi = min(C::BN, p.Sk - k0);
        if (p.mask_kind != kMaskNone) hi = min(hi, i - k0 + 1);
        if (p.mask_kind == kMaskWindow) lo = max(0, i - p.window + 1 - k0);
        const bool masked = lo > 0 || hi < C::BN;
        if (masked) {
#pragma unroll
            for (int e = 0; e < C::BN; ++e)
                if (e < lo || e >= hi) s[e] = __float_as_uint(-INFINITY);
        }
        // tile max as four independent chains (the latency of one serial
        // chain of BN/2 three-way maxima would sit on every tile's path)
        static_assert(C::BN % 8 == 0, "tile max in groups of eight");
        float mx[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) mx[j] = fmaxf(__uint_as_float(s[j]), __uint_as_float(s[4 + j]));
#pragma unroll
        for (int e = 8; e + 8 <= C::BN; e += 8)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                mx[j] = ptx::max3(mx[j], __uint_as_float(s[e + j]), __uint_as_float(s[e + 4 + j]));
        const float smax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        // Deferred rescaling: the reference max moves only when the tile's max
        // exceeds it by more than 2^4, so weights stay below 2^4 (stored times
        // 2^4: at most 256, inside e4m3's range) and O is rescaled rarely.
        const float mt = smax * c;  // -inf when no key of the tile is visible
        const bool grow = mt > m + C::TAU;
        const float m_new = grow ? mt : m;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ptx::ex2_approx(m - m_use);  // 1 unless the reference moved
        const float shift = m_use - C::P_LOG2;           // weights carry the factor 2^P_LOG2
        const uint64_t c2 = ptx::f32x2(c, c), n2 = ptx::f32x2(-shift, -shift);
        uint64_t acc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] = ptx::f32x2(0.f, 0.f);
        uint32_t pw[C::BN / 4];
#pragma unroll
        for (int e = 0; e < C::BN; e += 4) {
            float x0, x1, x2, x3;
            ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), c2, n2),
                              x0, x1);
            ptx::unpack_f32x2(
                ptx::fma_f32x2(ptx::f32x2(__uint_as_float(s[e + 2]), __uint_as_float(s[e + 3])), c2, n2), x2, x3);
            const float p0 = ptx::ex2_approx(x0), p1 = ptx::ex2_approx(x1);
            const float p2 = ptx::ex2_approx(x2), p3 = ptx::ex2_approx(x3);
            const int j = (e / 4) & 1;  // four independent accumulator pairs
            acc[2 * j] = ptx::add_f32x2(acc[2 * j], ptx::f32x2(p0, p1));
            acc[2 * j + 1] = ptx::add_f32x2(acc[2 * j + 1], ptx::f32x2(p2, p3));
            pw[e / 4] = ptx::pack_e4m3x4(p0, p1, p2, p3);
        }
        float a[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) ptx::unpack_f32x2(acc[j], a[2 * j], a[2 * j + 1]);
        l = l * alpha + (((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7])));
        if (t >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
            // O must hold P V of every earlier tile.  With one S buffer, S of
            // this tile was issued after P V of the previous one had run; with
            // two, wait for that product here (its P was written before this
            // tile's, so the barrier is at most that one phase ahead).
            if (C::NS > 1 &&
                !wait_warp(bar_addr(bars, C::B_PFREE + (t - 1) % C::NS), ((t - 1) / C::NS) & 1, ctl, 69)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < C::D / 32; ++cc) {
                uint32_t o[32];
                ptx::tmem_ld_x32<0>(lane_base + C::O_COL + cc * 32, o);
                ptx::tmem_wait_ld();
                ptx::reg_fence<32>(o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                ptx::tmem_st_x32<0>(lane_base + C::O_COL + cc * 32, o);
            }
        }
        m = m_new;
        if constexpr (C::BN == 128) ptx::tmem_st_x32<0>(lane_base + s_col, pw);
        else ptx::tmem_st_x16<0>(lane_base + s_col, pw);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_addr(bars, C::B_PFULL + b));
    }

    // Epilogue (whole warps): O / l as bf16 and the row's lse.
    const bool row_ok = i < p.Sq;
    const size_t row = ((size_t)un.b * p.H + un.h) * (size_t)p.Sq + (size_t)(row_ok ? i : 0);
    uint8_t *orow = static_cast<uint8_t *>(p.o) + row * C::D * 2;
    if (un.n > 0) {
        if (!ok || !wait_warp(bar_addr(bars, C::B_OFINAL), 0, ctl, 70)) return;
        ptx::tc_fence_after();
    }
    const bool seen = un.n > 0 && l > 0.f;
    const float mul = seen ? p.o_mul / l : 0.f;
#pragma unroll
    for (int cc = 0; cc < C::D / 32; ++cc) {
        uint32_t o[32];
        if (un.n > 0) {
            ptx::tmem_ld_x32<0>(lane_base + C::O_COL + cc * 32, o);
            ptx::tmem_wait_ld();
            ptx::reg_fence<32>(o);
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (row_ok) store_row32<false>(orow + cc * 64, o, mul);
    }
    // l sums the weights times 2^P_LOG2 against the reference m
    if (row_ok) p.lse[row] = seen ? (m - C::P_LOG2 + __log2f(l)) * kLn2 : -INFINITY;
}

template <class C>
__global__ void __launch_bounds__(192, C::CTAS_PER_SM) fa_fwd_fp8_kernel(const __grid_constant__ Fp8Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem;
    uint8_t *sK = sQ + C::Q_BYTES;
    uint8_t *sV = sK + C::KST * C::TILE_BYTES;
    uint64_t *bar_mem = reinterpret_cast<uint64_t *>(smem + C::SMEM_TILES);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bar_mem + C::NUM_BARS);
    Ctl *ctl = reinterpret_cast<Ctl *>(tmem_holder + 2);
    const uint32_t bars = ptx::smem_addr(bar_mem);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_addr(bars, C::B_QFULL), 1);
        for (int s = 0; s < C::KST; ++s) {
            ptx::mbar_init(bar_addr(bars, C::B_KFULL + s), 1);
            ptx::mbar_init(bar_addr(bars, C::B_KEMPTY + s), 1);
        }
        for (int s = 0; s < C::VST; ++s) {
            ptx::mbar_init(bar_addr(bars, C::B_VFULL + s), 1);
            ptx::mbar_init(bar_addr(bars, C::B_VEMPTY + s), 1);
        }
        for (int s = 0; s < C::NS; ++s) {
            ptx::mbar_init(bar_addr(bars, C::B_SFULL + s), 1);
            ptx::mbar_init(bar_addr(bars, C::B_PFULL + s), C::NUM_SOFTMAX);
            ptx::mbar_init(bar_addr(bars, C::B_PFREE + s), 1);
        }
        ptx::mbar_init(bar_addr(bars, C::B_OFINAL), 1);
        ptx::mbar_init(bar_addr(bars, C::B_DRAIN), 1);
        ptx::mbar_init(bar_addr(bars, C::B_NEVER), 1);
        ctl->abort = 0;
        ctl->limit_ns = p.wait_limit_ns;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == C::MMA_WARP) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == C::TMA_WARP && ptx::lane_id() == 0) {
        ptx::prefetch_tensormap(&p.tm_q);
        ptx::prefetch_tensormap(&p.tm_k);
        ptx::prefetch_tensormap(&p.tm_vt);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const Fp8Unit un = decode_fp8_unit<C::BN>(p);

    if (warp < C::NUM_SOFTMAX / 32) {
        fp8_softmax_role<C>(p, un, bars, tmem, ctl);
    } else if (warp == C::MMA_WARP) {
        fp8_mma_role<C>(p, un, sQ, sK, sV, bars, tmem, ctl);
    } else {
        fp8_tma_role<C>(p, un, sQ, sK, sV, bars, ctl);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace fa
