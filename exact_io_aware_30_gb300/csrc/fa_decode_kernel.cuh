// fa_decode_kernel.cuh -- attention of a few new query rows per request over a
// paged K/V cache, for sm_103a (GB300).
//
// The cache lives in fixed-size physical blocks of block_size tokens, and a
// per-request block table maps logical block n (tokens n*block_size ..) to a
// physical block anywhere in the pool ("Flash attention and memory-efficient
// attention variants", sections "A different bottleneck: the KV cache during
// inference" and "PagedAttention: memory management borrowed from an
// operating system").  The kernel walks the table and gathers the blocks with
// TMA, and computes the exact attention of the tiled forward pass over them:
// running max and sum per row, one division at the end.
//
// Work split.  Decoding is bound by reading the cache, so every (request,
// K/V head) is cut into n_splits key ranges that run on different CTAs (the
// sequence-length split that "What FlashAttention-2 changed" describes, here
// along the keys); each CTA writes its rows' partial output O_s, normalised by
// its own sum, and partial lse_s.  fa_decode_combine_kernel then merges the
// partials of a row with the same rescaling the online softmax uses:
//   lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s.
//
// One CTA: the new rows of all query heads that share the K/V head are packed
// into one 128-row tile (row r = (h - kvh * group) * Sq + i; they are
// consecutive rows of q), so the cache is read once per K/V head.  Rows past
// the group's are computed and discarded.  The tensor core has ample slack:
// a 128 x 128 tile of S and of P V takes about 1,024 cycles while its 64 KB of
// K and V (d = 128) take about 2,400 cycles to arrive from HBM at the per-SM
// share of the bandwidth.
//   warps 0-3: softmax and epilogue, one row (TMEM lane) per thread;
//   warp 4:    MMA issuer (S = Q K^T into two S buffers, O += P V);
//   warp 5:    TMA: the Q tile once, then per key tile 128 / block_size block
//              loads of K and of V into rings of three slots each.
#pragma once

#include <math.h>
#include <stdint.h>

#include "fa_bwd_kernel.cuh"

namespace fa {

struct DecParams {
    CUtensorMap tm_q;  // q viewed as [B*H*Sq rows, d], box {64, 128}
    CUtensorMap tm_k;  // k_cache [num_blocks, Hkv, bs, d], box {64, bs, 1, 1}
    CUtensorMap tm_v;  // v_cache, same layout
    const int *block_table;  // [B, max_blocks]
    const int *seq_lens;     // [B]
    float *part_o;           // [n_splits, B*H*Sq, d] fp32, normalised per split
    float *part_lse;         // [n_splits, B*H*Sq] fp32, natural log; -inf: split saw no key
    const int *order;        // CTA x runs unit order[x] (longest first), or unit x when null
    int B, H, Hkv, kv_group, Sq, R;  // R = kv_group * Sq rows per CTA
    int bs, max_blocks, max_seq_len;
    int mask_kind;
    int n_splits, tiles_per_split;
    float scale_log2;
    uint64_t wait_limit_ns;
    int stall_test;          // test only: the softmax's first wait is on a barrier nothing completes
};

template <int D>
struct DecCfg {
    // d = 256 takes 64-key tiles, so that two S buffers, its 256-column O and
    // P fit in tensor memory and two-slot rings in shared memory.
    static constexpr int BN = (D == 256) ? 64 : 128;  // keys per tile
    static constexpr int KST = (D == 256) ? 2 : 3;
    static constexpr int VST = (D == 256) ? 2 : 3;
    static constexpr int Q_BOX = 128 * 128;
    static constexpr int KV_BOX = BN * 128;
    static constexpr int Q_BYTES = 128 * D * 2;
    static constexpr int TILE_BYTES = BN * D * 2;
    static constexpr int NUM_SOFTMAX = 128;
    static constexpr int MMA_WARP = 4;
    static constexpr int TMA_WARP = 5;
    static constexpr int NUM_THREADS = 192;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0;    // two S buffers, BN columns each
    static constexpr uint32_t O_COL = 2 * BN;
    static constexpr uint32_t P_COL = 384;  // BN / 2 columns of 16-bit pairs
    static constexpr int B_QFULL = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_KEMPTY = B_KFULL + KST;
    static constexpr int B_VFULL = B_KEMPTY + KST;
    static constexpr int B_VEMPTY = B_VFULL + VST;
    static constexpr int B_SFULL = B_VEMPTY + VST;  // [2]
    static constexpr int B_SFREE = B_SFULL + 2;     // [2]
    static constexpr int B_PFULL = B_SFREE + 2;
    static constexpr int B_PFREE = B_PFULL + 1;
    static constexpr int B_OFINAL = B_PFREE + 1;
    static constexpr int B_DRAIN = B_OFINAL + 1;
    static constexpr int B_NEVER = B_DRAIN + 1;  // no arrivals (the stall test's wait)
    static constexpr int NUM_BARS = B_NEVER + 1;
    static constexpr int SMEM_TILES = Q_BYTES + (KST + VST) * TILE_BYTES;
    static constexpr int SMEM_BYTES = 1024 + SMEM_TILES + NUM_BARS * 8 + 32;
    static_assert(O_COL + D <= P_COL && P_COL + BN / 2 <= TMEM_COLS, "tensor memory overflow");
    static_assert(SMEM_BYTES <= 232448, "shared memory overflow");
};

// One CTA's work: request b, K/V head kvh, keys [k_beg, k_end) in n tiles.
struct DecUnit {
    int b, kvh, split, L, k_beg, k_end, n;
};

template <int D>
__device__ __forceinline__ DecUnit decode_dec_unit(const DecParams &p) {
    DecUnit u;
    const int unit = p.order ? p.order[blockIdx.x] : (int)blockIdx.x;
    u.split = unit % p.n_splits;
    const int bk = unit / p.n_splits;
    u.b = bk / p.Hkv;
    u.kvh = bk - u.b * p.Hkv;
    // the caller guarantees Sq <= seq_lens[b] <= max_seq_len; clamp anyway so
    // that no index leaves the block table
    u.L = min(max(p.seq_lens[u.b], p.Sq), p.max_seq_len);
    constexpr int BN = DecCfg<D>::BN;
    u.k_beg = u.split * p.tiles_per_split * BN;
    u.k_end = min(u.k_beg + p.tiles_per_split * BN, u.L);
    u.n = u.k_end > u.k_beg ? (u.k_end - u.k_beg + BN - 1) / BN : 0;
    return u;
}

// Loads key tile t of the unit (BN keys) of one cache into a ring slot, as
// boxes of min(block_size, BN) rows (a box never crosses a block).  Boxes past
// the request's last block repeat its last block's first rows: the bytes still
// arrive (the barrier counts them) and the keys are masked.
template <int D>
__device__ __forceinline__ void dec_load_tile(const DecParams &p, const DecUnit &un, const CUtensorMap *tm,
                                              uint32_t dst, uint32_t fb, int t, uint64_t pol) {
    using C = DecCfg<D>;
    ptx::mbar_arrive_expect_tx(fb, C::TILE_BYTES);
    const int n_last = (un.L + p.bs - 1) / p.bs - 1;
    const int key0 = un.k_beg + t * C::BN;
    const int *row = p.block_table + (size_t)un.b * p.max_blocks;
    // (with 128-key tiles every supported block size divides the tile)
    if (C::BN >= 128 || p.bs <= C::BN) {  // whole blocks
        const int per_tile = C::BN / p.bs;
        const int n0 = key0 / p.bs;
        for (int blk = 0; blk < per_tile; ++blk) {
            const int phys = row[min(n0 + blk, n_last)];
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                ptx::tma_load_4d(dst + c * C::KV_BOX + blk * p.bs * 128, tm, fb, c * 64, 0, un.kvh, phys, pol);
        }
    } else {  // one BN-row box inside a larger block
        int n = key0 / p.bs, y = key0 % p.bs;
        if (n > n_last) {
            n = n_last;
            y = 0;
        }
        const int phys = row[n];
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
            ptx::tma_load_4d(dst + c * C::KV_BOX, tm, fb, c * 64, y, un.kvh, phys, pol);
    }
}

template <int D>
__device__ void dec_tma_role(const DecParams &p, const DecUnit &un, uint8_t *sQ, uint8_t *sK, uint8_t *sV,
                             uint32_t bars, Ctl *ctl) {
    using C = DecCfg<D>;
    const bool leader = ptx::lane_id() == 0;
    const uint64_t pol_stream = ptx::policy_evict_first();  // the cache is read once
    if (un.n == 0) return;
    if (leader) {
        const uint32_t fb = bar_addr(bars, C::B_QFULL);
        ptx::mbar_arrive_expect_tx(fb, C::Q_BYTES);
        const int row0 = (un.b * p.H + un.kvh * p.kv_group) * p.Sq;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
            ptx::tma_load_4d(ptx::smem_addr(sQ) + c * C::Q_BOX, &p.tm_q, fb, c * 64, row0, 0, 0,
                             ptx::policy_evict_last());
    }
    int k_issued = 0, v_issued = 0;
    bool ok = true;
    for (int t = 0; t < un.n && ok; ++t) {
        const int ks = t % C::KST, vs = t % C::VST;
        if (!wait_warp_backoff(bar_addr(bars, C::B_KEMPTY + ks), ((t / C::KST) & 1) ^ 1, ctl, 41)) {
            ok = false;
            break;
        }
        if (leader)
            dec_load_tile<D>(p, un, &p.tm_k, ptx::smem_addr(sK + ks * C::TILE_BYTES),
                             bar_addr(bars, C::B_KFULL + ks), t, pol_stream);
        __syncwarp();
        ++k_issued;
        if (!wait_warp_backoff(bar_addr(bars, C::B_VEMPTY + vs), ((t / C::VST) & 1) ^ 1, ctl, 42)) {
            ok = false;
            break;
        }
        if (leader)
            dec_load_tile<D>(p, un, &p.tm_v, ptx::smem_addr(sV + vs * C::TILE_BYTES),
                             bar_addr(bars, C::B_VFULL + vs), t, pol_stream);
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

template <int D, bool kFP16>
__device__ void dec_mma_role(const DecParams &p, const DecUnit &un, uint8_t *sQ, uint8_t *sK, uint8_t *sV,
                             uint32_t bars, uint32_t tmem, Ctl *ctl) {
    using C = DecCfg<D>;
    constexpr uint32_t kIdescS = make_idesc(128, C::BN, kFP16, false);
    constexpr uint32_t kIdescO = make_idesc(128, D, kFP16, true);
    const bool leader = ptx::lane_id() == 0;
    const uint64_t qd = smem_desc(ptx::smem_addr(sQ), 16);
    bool ok = un.n == 0 || wait_warp(bar_addr(bars, C::B_QFULL), 0, ctl, 43);
    for (int t = 0; ok && t <= un.n; ++t) {
        if (t < un.n) {
            const int ks = t % C::KST;
            const uint32_t b = (uint32_t)t & 1u;
            if (!wait_warp(bar_addr(bars, C::B_KFULL + ks), (t / C::KST) & 1, ctl, 44)) {
                ok = false;
                break;
            }
            // the softmax has read S of tile t-2 out of this buffer
            if (t >= 2 && !wait_warp(bar_addr(bars, C::B_SFREE + (int)b), ((t >> 1) - 1) & 1, ctl, 45)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            if (leader) {
                const uint64_t kd = smem_desc(ptx::smem_addr(sK + ks * C::TILE_BYTES), 16);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + C::S_COL + b * C::BN, qd + kmajor_step(kk, C::Q_BOX),
                                kd + kmajor_step(kk, C::KV_BOX), kIdescS, kk > 0 ? 1u : 0u);
                ptx::mma_commit(bar_addr(bars, C::B_SFULL + (int)b));
                ptx::mma_commit(bar_addr(bars, C::B_KEMPTY + ks));
            }
            __syncwarp();
        }
        if (t >= 1) {
            const int tp = t - 1, vs = tp % C::VST;
            if (!wait_warp(bar_addr(bars, C::B_VFULL + vs), (tp / C::VST) & 1, ctl, 46) ||
                !wait_warp(bar_addr(bars, C::B_PFULL), tp & 1, ctl, 47)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            if (leader) {
                const uint64_t vd = smem_desc(ptx::smem_addr(sV + vs * C::TILE_BYTES), C::KV_BOX);
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)
                    ptx::mma_ts(tmem + C::O_COL, tmem + C::P_COL + kk * 8, vd + (uint32_t)((kk * 2048) >> 4),
                                kIdescO, (tp > 0 || kk > 0) ? 1u : 0u);
                ptx::mma_commit(bar_addr(bars, C::B_PFREE));
                ptx::mma_commit(bar_addr(bars, C::B_VEMPTY + vs));
                if (tp + 1 == un.n) ptx::mma_commit(bar_addr(bars, C::B_OFINAL));
            }
            __syncwarp();
        }
    }
    if (leader) ptx::mma_commit(bar_addr(bars, C::B_DRAIN));
    __syncwarp();
    wait_bar_drain(bar_addr(bars, C::B_DRAIN), 0);
}

template <int D, bool kFP16>
__device__ void dec_softmax_role(const DecParams &p, const DecUnit &un, uint8_t *sV, uint32_t bars,
                                 uint32_t tmem, Ctl *ctl) {
    using C = DecCfg<D>;
    const int r = (int)threadIdx.x;  // packed row = TMEM lane
    const int warp = r >> 5;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int i = r % p.Sq;              // query row of its head
    // last key the row sees (rows past R are computed and discarded)
    const int last = (p.mask_kind == kMaskCausal) ? un.L - p.Sq + i : un.L - 1;
    const float c = p.scale_log2;
    float m = -INFINITY;  // running max of s * c (log2 units)
    float l = 0.f;        // running sum of 2^(s c - m)
    bool ok = true;
    for (int t = 0; t < un.n; ++t) {
        const uint32_t b = (uint32_t)t & 1u;
        const int k0 = un.k_beg + t * C::BN;
        if (!wait_warp(bar_addr(bars, (p.stall_test && t == 0) ? C::B_NEVER : C::B_SFULL + (int)b), (t >> 1) & 1,
                       ctl, 48)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        uint32_t s[C::BN];
        ptx::tmem_ld_x32<0>(lane_base + C::S_COL + b * C::BN, s);
        ptx::tmem_ld_x32<32>(lane_base + C::S_COL + b * C::BN + 32, s);
        if constexpr (C::BN == 128) {
            ptx::tmem_ld_x32<64>(lane_base + C::S_COL + b * C::BN + 64, s);
            ptx::tmem_ld_x32<96>(lane_base + C::S_COL + b * C::BN + 96, s);
        }
        ptx::tmem_wait_ld();
        ptx::reg_fence<C::BN>(s);
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_addr(bars, C::B_SFREE + (int)b));

        // scaled scores, hidden keys (past the row's last, or past the
        // request) replaced by -inf; a select, so junk in a hidden key's cache
        // row cannot leak in
        const int vis = last - k0 + 1;  // columns [0, vis) are visible
        float mt = -INFINITY;
#pragma unroll
        for (int e = 0; e < C::BN; ++e) {
            const float x = __uint_as_float(s[e]) * c;
            const float y = e < vis ? x : -INFINITY;
            s[e] = __float_as_uint(y);
            mt = fmaxf(mt, y);
        }
        const float m_new = fmaxf(m, mt);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // no visible key yet: all weights 0
        const float alpha = ptx::ex2_approx(m - m_use);           // 0 while m is -inf
        uint32_t pw[C::BN / 2];
        float ps = 0.f;
#pragma unroll
        for (int e = 0; e < C::BN; e += 2) {
            const float p0 = ptx::ex2_approx(__uint_as_float(s[e]) - m_use);
            const float p1 = ptx::ex2_approx(__uint_as_float(s[e + 1]) - m_use);
            ps += p0 + p1;
            pw[e / 2] = pack2b<kFP16>(p0, p1);
        }
        l = l * alpha + ps;
        // P V of tile t-1 has run: the P area is free and O is stable
        if (t >= 1 && !wait_warp(bar_addr(bars, C::B_PFREE), (t - 1) & 1, ctl, 49)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        if (t >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
            // rescale this warp's O rows to the new maximum
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
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
        ptx::tmem_st_x32<0>(lane_base + C::P_COL, pw);
        if constexpr (C::BN == 128) ptx::tmem_st_x32<32>(lane_base + C::P_COL + 32, pw);
        if (t + 1 == un.n && un.k_beg + (t + 1) * C::BN > un.L) {
            // last tile reaches past the request's keys: zero those V rows, so
            // that junk in an unused cache slot (even inf or NaN) meets P = 0
            // as an exact 0
            const int vs = t % C::VST;
            if (!wait_warp(bar_addr(bars, C::B_VFULL + vs), (t / C::VST) & 1, ctl, 50)) {
                ok = false;
                break;
            }
            if (r < C::BN && k0 + r >= un.L) {  // the tile's rows are its BN keys
                uint8_t *row = sV + vs * C::TILE_BYTES + r * 128;
#pragma unroll
                for (int cc = 0; cc < D / 64; ++cc)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        ptx::st_shared_v4(ptx::smem_addr(row + cc * C::KV_BOX + q * 16), 0u, 0u, 0u, 0u);
            }
            ptx::fence_proxy_async_smem();
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_addr(bars, C::B_PFULL));
    }

    // Epilogue: this split's normalised rows and their lse.  Whole warps run
    // it (tcgen05.ld is warp-collective); only rows below R are stored.
    if (32 * warp >= p.R) return;  // the warp holds no packed row
    if (un.n > 0) {
        if (!ok || !wait_warp(bar_addr(bars, C::B_OFINAL), 0, ctl, 51)) return;
        ptx::tc_fence_after();
    }
    const bool mine = r < p.R;
    const size_t row = (size_t)(un.b * p.H + un.kvh * p.kv_group) * p.Sq + (size_t)(mine ? r : 0);
    const size_t n_rows = (size_t)p.B * p.H * p.Sq;
    float *po = p.part_o + ((size_t)un.split * n_rows + row) * D;
    float *pl = p.part_lse + (size_t)un.split * n_rows + row;
    const bool seen = un.n > 0 && l > 0.f;
    const float inv = seen ? 1.f / l : 0.f;
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        if (un.n > 0) {
            ptx::tmem_ld_x32<0>(lane_base + C::O_COL + cc * 32, o);
            ptx::tmem_wait_ld();
            ptx::reg_fence<32>(o);
        }
        if (mine) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                float4 v;
                v.x = seen ? __uint_as_float(o[e]) * inv : 0.f;
                v.y = seen ? __uint_as_float(o[e + 1]) * inv : 0.f;
                v.z = seen ? __uint_as_float(o[e + 2]) * inv : 0.f;
                v.w = seen ? __uint_as_float(o[e + 3]) * inv : 0.f;
                *reinterpret_cast<float4 *>(po + cc * 32 + e) = v;
            }
        }
    }
    if (mine) *pl = seen ? (m + __log2f(l)) * kLn2 : -INFINITY;
}

template <int D, bool kFP16>
__global__ void __launch_bounds__(DecCfg<D>::NUM_THREADS, 1)
    fa_decode_kernel(const __grid_constant__ DecParams p) {
    using C = DecCfg<D>;
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
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_addr(bars, C::B_SFULL + b), 1);
            ptx::mbar_init(bar_addr(bars, C::B_SFREE + b), C::NUM_SOFTMAX);
        }
        ptx::mbar_init(bar_addr(bars, C::B_PFULL), C::NUM_SOFTMAX);
        ptx::mbar_init(bar_addr(bars, C::B_PFREE), 1);
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
        ptx::prefetch_tensormap(&p.tm_v);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const DecUnit un = decode_dec_unit<D>(p);

    if (warp < C::NUM_SOFTMAX / 32) {
        dec_softmax_role<D, kFP16>(p, un, sV, bars, tmem, ctl);
    } else if (warp == C::MMA_WARP) {
        dec_mma_role<D, kFP16>(p, un, sQ, sK, sV, bars, tmem, ctl);
    } else {
        dec_tma_role<D>(p, un, sQ, sK, sV, bars, ctl);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Longest-first order of the decode CTAs.  The host does not know the
// requests' lengths, so this one-CTA kernel counts the key tiles of every
// (request, K/V head, key range) unit -- the same ranges decode_dec_unit
// takes -- and lists the units by decreasing tile count (a counting sort on
// min(tiles, 255); the order within a count does not matter, since every
// unit writes its own partial slot).  CTA x of the decode kernel then runs
// unit order[x]: with one CTA per SM and lengths that differ by up to the
// whole context, the last wave otherwise leaves SMs idle behind a few long
// requests.
template <int BN>
__global__ void __launch_bounds__(1024)
    fa_decode_order_kernel(const int *__restrict__ seq_lens, int B, int Hkv, int Sq, int max_seq_len,
                           int n_splits, int tiles_per_split, int *__restrict__ order) {
    __shared__ int start[256];
    const int n = B * Hkv * n_splits;
    for (int i = (int)threadIdx.x; i < 256; i += (int)blockDim.x) start[i] = 0;
    __syncthreads();
    auto key = [&](int u) -> int {
        const int split = u % n_splits;
        const int b = u / n_splits / Hkv;
        const int L = min(max(seq_lens[b], Sq), max_seq_len);
        const int k_beg = split * tiles_per_split * BN;
        const int k_end = min(k_beg + tiles_per_split * BN, L);
        const int tiles = k_end > k_beg ? (k_end - k_beg + BN - 1) / BN : 0;
        return 255 - min(tiles, 255);  // ascending key = descending tile count
    };
    for (int u = (int)threadIdx.x; u < n; u += (int)blockDim.x) atomicAdd(&start[key(u)], 1);
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int i = 0; i < 256; ++i) {
            const int c = start[i];
            start[i] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int u = (int)threadIdx.x; u < n; u += (int)blockDim.x) order[atomicAdd(&start[key(u)], 1)] = u;
}

// Merges the n_splits partial rows: one warp per row, lanes over d.
template <int D, bool kFP16>
__global__ void __launch_bounds__(256)
    fa_decode_combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_lse,
                             void *__restrict__ o, float *__restrict__ lse, int n_rows, int n_splits) {
    const int row = (int)(blockIdx.x * 8 + (threadIdx.x >> 5));
    const int lane = (int)threadIdx.x & 31;
    if (row >= n_rows) return;  // whole warps leave together
    float mx = -INFINITY;
    for (int s = 0; s < n_splits; ++s) mx = fmaxf(mx, part_lse[(size_t)s * n_rows + row]);
    constexpr int PER = D / 32;  // values per lane
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    if (mx != -INFINITY) {
        for (int s = 0; s < n_splits; ++s) {
            const float ls = part_lse[(size_t)s * n_rows + row];
            if (ls == -INFINITY) continue;
            const float w = __expf(ls - mx);
            wsum += w;
            const float *src = part_o + ((size_t)s * n_rows + row) * D + lane * PER;
#pragma unroll
            for (int e = 0; e < PER; e += 2) {
                const float2 v = *reinterpret_cast<const float2 *>(src + e);
                acc[e] = fmaf(w, v.x, acc[e]);
                acc[e + 1] = fmaf(w, v.y, acc[e + 1]);
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint32_t w16[PER / 2];
#pragma unroll
    for (int e = 0; e < PER; e += 2) w16[e / 2] = pack2b<kFP16>(acc[e] * inv, acc[e + 1] * inv);
    uint8_t *dst = static_cast<uint8_t *>(o) + ((size_t)row * D + lane * PER) * 2;
    if constexpr (PER == 8) {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w16[0], w16[1], w16[2], w16[3]);
    } else if constexpr (PER == 4) {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w16[0], w16[1]);
    } else {
        *reinterpret_cast<uint32_t *>(dst) = w16[0];
    }
    if (lane == 0) lse[row] = wsum > 0.f ? mx + __logf(wsum) : -INFINITY;
}

}  // namespace fa
