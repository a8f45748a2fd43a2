// fa_fwd_kernel.cuh -- fused exact attention forward for sm_103a (GB300).
//
// What it computes: for every (batch, head) and query row i,
//   O_i = sum_j softmax_j(scale * q_i . k_j) v_j   over the keys j visible to i,
//   lse_i = ln sum_j exp(scale * q_i . k_j),
// by the tiled forward pass with the online softmax ("FlashAttention: Why
// Tiling Attention Makes Transformers Fast Without Changing the Result",
// sections "Online softmax: correct as you go" and "The tiled forward pass";
// "Flash attention and memory-efficient attention variants", section "Tiling
// and the running (online) softmax"): key/value tiles stream through shared
// memory, each query row keeps a running max m, a running sum l and an
// unnormalised accumulator rescaled by exp(m_old - m_new), and the row is
// divided by l once at the end.  Score and probability tiles live only in
// tensor memory.
//
// GB300 mapping (one CTA per SM, persistent over work units):
//   * a work unit is NQ query tiles of 128 rows of one (batch, head);
//     units are taken longest-first in a snake order over the CTAs;
//   * one TMA warp streams Q tiles and a ring of K / V tiles (128-byte
//     swizzled, 64 columns per box) into shared memory under mbarriers;
//   * one MMA warp (a single issuing lane) runs S = Q K^T (both operands in
//     shared memory) and O += P V (P read from tensor memory) as tcgen05
//     MMAs with fp32 accumulators in tensor memory;
//   * NQ softmax warpgroups own one query row per thread (= one TMEM lane):
//     they read a row of S, apply the mask on boundary tiles only, update the
//     running max / sum, write P (16-bit) back over S, rescale O in tensor
//     memory when the max grew enough, and run the epilogue (O / l, lse).
//   With NQ = 2 the two warpgroups ping-pong: the tensor core computes one
//   tile's MMAs while the other tile's softmax runs.
//
// Rescaling is deferred until the running max has grown by more than 2^8
// (log2 units).  Until then the accumulator and the sum both stay referenced
// to the same stale max, so the final O_acc / l is unchanged (the pages'
// remark that FlashAttention-2 "defers most rescaling"); the stale reference
// only lets unnormalised weights reach 2^8, far from fp32/bf16 limits.
#pragma once

#include <stdint.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBM = 128;  // query rows per tile = M of every MMA = TMEM lanes
constexpr int kMaskNone = 0;
constexpr int kMaskCausal = 1;
constexpr int kMaskWindow = 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a pipeline wait gives up after 2 s
constexpr float kRescaleLog2 = 8.0f;              // rescale O when the max grows > 2^8
constexpr float kRescaleBound = 256.0f;           // 2^kRescaleLog2
constexpr float kLn2 = 0.693147180559945309f;

// Device status word: 0 = fine; else 0x100 + the wait site that timed out.
// (This header is compiled into exactly one translation unit.)
__device__ int g_fa_status = 0;

struct Params {
    CUtensorMap tm_q;  // [B, H, Sq, d] 16-bit, box {64, 128, 1, 1}, 128-B swizzle
    CUtensorMap tm_k;  // [B, H, Sk, d], box {64, BN, 1, 1}
    CUtensorMap tm_v;  // [B, H, Sk, d], box {64, BN, 1, 1}
    void *o;           // [B, H, Sq, d] 16-bit
    float *lse;        // [B, H, Sq] fp32
    int B, H, Sq, Sk;
    int mask_kind, window;
    float scale_log2;  // scale * log2(e)
    int n_qtiles;      // ceil(Sq / 128)
    int n_groups;      // ceil(n_qtiles / NQ): units per (batch, head)
    int n_units;       // B * H * n_groups
};

template <int D>
struct Cfg {
    // One query tile per unit with two S buffers: the S MMA of key tile j+1
    // runs while the softmax works on tile j.  d = 256 uses 64-key tiles so
    // that two S buffers and its 256-column O fit in tensor memory and a
    // 5-deep K/V ring fits in shared memory.
    static constexpr int BN = (D == 256) ? 64 : 128;     // keys per K/V tile
    static constexpr int NQ = 1;                         // query tiles per unit
    static constexpr int SLOTS = (D == 64) ? 12 : (D == 128) ? 6 : 5;  // K/V ring depth (tiles)
    // Warps: NQ softmax warpgroups (warps 0 .. 4*NQ-1), then the MMA warp and
    // the TMA warp.
    static constexpr int NUM_WARPS = 4 * NQ + 2;
    static constexpr int NUM_THREADS = 32 * NUM_WARPS;
    static constexpr int MMA_WARP = 4 * NQ;
    static constexpr int TMA_WARP = 4 * NQ + 1;
    static constexpr int CHUNKS = D / 64;              // 64-column (128-byte) boxes per row
    static constexpr int Q_CHUNK = kBM * 128;          // bytes of one Q box
    static constexpr int KV_CHUNK = BN * 128;          // bytes of one K or V box
    static constexpr int Q_BYTES = kBM * D * 2;
    static constexpr int SLOT_BYTES = BN * D * 2;
    // Tensor memory: two S/P buffers per query tile (BN columns each) at
    // columns (2q + b) * BN, O accumulators (D columns each) from column 256.
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t O_COL0 = 256;
    // Barrier indices.
    static constexpr int B_QFULL = 0;
    static constexpr int B_QEMPTY = B_QFULL + NQ;
    static constexpr int B_KVFULL = B_QEMPTY + NQ;
    static constexpr int B_KVEMPTY = B_KVFULL + SLOTS;
    static constexpr int B_SFULL = B_KVEMPTY + SLOTS;   // [2 * NQ]: S buffer (q, b) computed
    static constexpr int B_PFULL = B_SFULL + 2 * NQ;    // [2 * NQ]: P buffer (q, b) written
    static constexpr int B_OFULL = B_PFULL + 2 * NQ;    // [NQ]: one phase per P V
    static constexpr int B_OFREE = B_OFULL + NQ;        // [NQ]: epilogue has read O
    static constexpr int B_DRAIN = B_OFREE + NQ;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int SMEM_TILES = NQ * Q_BYTES + SLOTS * SLOT_BYTES;
    static constexpr int SMEM_BYTES = 1024 + SMEM_TILES + NUM_BARS * 8 + 16;
    static_assert(O_COL0 + NQ * D <= TMEM_COLS, "tensor memory overflow");
    static_assert(2 * NQ * BN <= (int)O_COL0, "S buffers overlap O");
    static_assert(SMEM_BYTES <= 232448, "shared memory overflow");

    __device__ static constexpr uint32_t s_col(int q, int b) { return (uint32_t)((2 * q + b) * BN); }
};

// ---------------------------------------------------------------- helpers

// Shared-memory matrix descriptor, 128-byte swizzle, tcgen05 format.
// K-major operands: rows of 128 bytes, 8-row groups 1024 bytes apart (SBO);
// the leading offset is unused.  MN-major (V as the B operand of P V): 8-row
// groups along K 1024 bytes apart (SBO), 64-element column boxes `lbo` apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulate, A/B bf16 or fp16,
// A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool fp16, bool b_mn_major) {
    return (1u << 4) | ((fp16 ? 0u : 1u) << 7) | ((fp16 ? 0u : 1u) << 10) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + 8u * (uint32_t)i; }

// Bounded wait: gives up (and raises the abort flag and the device status
// word) after kWaitLimitNs, or as soon as another role has aborted.
__device__ __forceinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           int site) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicCAS(&g_fa_status, 0, 0x100 + site);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         int site) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, abort_flag, site);
}

// Wait used only while shutting down after an abort: ignores the abort flag.
__device__ __forceinline__ void wait_bar_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) return;
    }
}

// Unit k of this CTA in a snake order: even rounds left to right, odd rounds
// right to left, so that with units sorted longest-first each CTA's sum of
// work stays close to the others'.
__device__ __forceinline__ int unit_at(int k) {
    const int G = gridDim.x, c = blockIdx.x;
    return (k & 1) ? k * G + (G - 1 - c) : k * G + c;
}

template <int D>
struct Unit {
    int b, h;
    int i0[Cfg<D>::NQ];     // first query row of each tile
    int lo[Cfg<D>::NQ];     // K/V tile range [lo, hi) each tile must visit
    int hi[Cfg<D>::NQ];
    bool exists[Cfg<D>::NQ];  // tile has rows < Sq
    bool valid[Cfg<D>::NQ];   // exists and sees at least one key tile
    int ulo, uhi;             // union of the valid ranges
    bool any;
};

// Key tiles a query tile [i0, i0 + 128) has to visit: skip tiles the mask
// hides entirely (causal: keys past the last row; window: keys before the
// first row's window).
template <int D>
__device__ __forceinline__ void kv_range(int i0, const Params &p, int &lo, int &hi) {
    constexpr int BN = Cfg<D>::BN;
    const int row_end = min(i0 + kBM, p.Sq);
    int key_end = p.Sk;
    if (p.mask_kind != kMaskNone) key_end = min(p.Sk, row_end);
    int key_beg = 0;
    if (p.mask_kind == kMaskWindow) key_beg = max(0, i0 - p.window + 1);
    if (key_beg >= key_end) {
        lo = 0;
        hi = 0;
        return;
    }
    lo = key_beg / BN;
    hi = (key_end + BN - 1) / BN;
}

template <int D>
__device__ __forceinline__ void decode_unit(int u, const Params &p, Unit<D> &un) {
    constexpr int NQ = Cfg<D>::NQ;
    const int BH = p.B * p.H;
    const int gi = u / BH;
    const int bh = u - gi * BH;
    const int g = p.n_groups - 1 - gi;  // longest first (causal / window)
    un.b = bh / p.H;
    un.h = bh - un.b * p.H;
    un.ulo = 0x7fffffff;
    un.uhi = 0;
    un.any = false;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        const int i0 = (g * NQ + q) * kBM;
        un.i0[q] = i0;
        un.exists[q] = i0 < p.Sq;
        un.lo[q] = 0;
        un.hi[q] = 0;
        if (un.exists[q]) kv_range<D>(i0, p, un.lo[q], un.hi[q]);
        un.valid[q] = un.exists[q] && un.lo[q] < un.hi[q];
        if (un.valid[q]) {
            un.ulo = min(un.ulo, un.lo[q]);
            un.uhi = max(un.uhi, un.hi[q]);
            un.any = true;
        }
    }
}

// True if some (row, key) pair of this query tile x key tile is hidden.
template <int D>
__device__ __forceinline__ bool tile_needs_mask(int i0, int j, const Params &p) {
    constexpr int BN = Cfg<D>::BN;
    const int k0 = j * BN;
    if (k0 + BN > p.Sk) return true;
    if (p.mask_kind == kMaskNone) return false;
    if (k0 + BN - 1 > i0) return true;
    if (p.mask_kind == kMaskWindow && k0 <= i0 + kBM - 1 - p.window) return true;
    return false;
}

// ---------------------------------------------------------------- TMA role

template <int D>
__device__ void tma_role(const Params &p, uint8_t *sQ, uint8_t *sKV, uint32_t bars,
                         volatile int *abort_flag) {
    using C = Cfg<D>;
    const uint64_t pol_kv = ptx::policy_evict_last();
    const uint64_t pol_q = ptx::policy_evict_first();
    uint32_t kv_it = 0;
    uint32_t q_cnt[C::NQ];
#pragma unroll
    for (int q = 0; q < C::NQ; ++q) q_cnt[q] = 0;
    bool ok = true;

    for (int k = 0; ok; ++k) {
        const int u = unit_at(k);
        if (u >= p.n_units) break;
        Unit<D> un;
        decode_unit<D>(u, p, un);
        if (!un.any) continue;
#pragma unroll
        for (int q = 0; q < C::NQ; ++q) {
            if (!un.valid[q] || !ok) continue;
            if (!wait_bar(bar_addr(bars, C::B_QEMPTY + q), (q_cnt[q] & 1) ^ 1, abort_flag, 1)) {
                ok = false;
                break;
            }
            const uint32_t fb = bar_addr(bars, C::B_QFULL + q);
            ptx::mbar_arrive_expect_tx(fb, C::Q_BYTES);
            const uint32_t dst = ptx::smem_addr(sQ + q * C::Q_BYTES);
#pragma unroll
            for (int c = 0; c < C::CHUNKS; ++c)
                ptx::tma_load_4d(dst + c * C::Q_CHUNK, &p.tm_q, fb, c * 64, un.i0[q], un.h, un.b,
                                 pol_q);
            ++q_cnt[q];
        }
        for (int j = un.ulo; j < un.uhi && ok; ++j) {
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                const uint32_t slot = kv_it % C::SLOTS;
                if (!wait_bar(bar_addr(bars, C::B_KVEMPTY + slot), ((kv_it / C::SLOTS) & 1) ^ 1,
                              abort_flag, 2)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = bar_addr(bars, C::B_KVFULL + slot);
                ptx::mbar_arrive_expect_tx(fb, C::SLOT_BYTES);
                const uint32_t dst = ptx::smem_addr(sKV + slot * C::SLOT_BYTES);
                const CUtensorMap *m = kv ? &p.tm_v : &p.tm_k;
#pragma unroll
                for (int c = 0; c < C::CHUNKS; ++c)
                    ptx::tma_load_4d(dst + c * C::KV_CHUNK, m, fb, c * 64, j * C::BN, un.h, un.b,
                                     pol_kv);
                ++kv_it;
            }
        }
    }
    if (!ok) {
        // Let every copy already issued land before the CTA can exit.
        // Slot s has been filled ceil((kv_it - s) / SLOTS) times so far.
#pragma unroll
        for (int s = 0; s < C::SLOTS; ++s) {
            const uint32_t fills = kv_it > (uint32_t)s ? (kv_it - (uint32_t)s + C::SLOTS - 1) / C::SLOTS : 0u;
            if (fills) wait_bar_drain(bar_addr(bars, C::B_KVFULL + s), (fills - 1) & 1);
        }
#pragma unroll
        for (int q = 0; q < C::NQ; ++q)
            if (q_cnt[q]) wait_bar_drain(bar_addr(bars, C::B_QFULL + q), (q_cnt[q] - 1) & 1);
    }
}

// ---------------------------------------------------------------- MMA role

template <int D, bool kFP16>
__device__ void mma_role(const Params &p, uint8_t *sQ, uint8_t *sKV, uint32_t bars,
                         uint32_t tmem, volatile int *abort_flag) {
    using C = Cfg<D>;
    constexpr int NQ = C::NQ;
    constexpr int BN = C::BN;
    constexpr uint32_t kIdescS = make_idesc(kBM, BN, kFP16, false);
    constexpr uint32_t kIdescO = make_idesc(kBM, D, kFP16, true);

    uint32_t kv_it = 0;          // K/V ring fills consumed so far
    uint32_t q_cnt[NQ];          // Q tiles consumed per query slot
    uint32_t t_cnt[NQ];          // key tiles processed per query slot (S/P buffer = t & 1)
    uint32_t ofree_cnt[NQ];      // epilogues waited for per O accumulator
    bool o_used[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        q_cnt[q] = 0;
        t_cnt[q] = 0;
        ofree_cnt[q] = 0;
        o_used[q] = false;
    }
    bool ok = true;

    for (int k = 0; ok; ++k) {
        const int u = unit_at(k);
        if (u >= p.n_units) break;
        Unit<D> un;
        decode_unit<D>(u, p, un);
        if (!un.any) continue;
        const uint32_t kv_base = kv_it;
        auto kidx = [&](int j) -> uint32_t { return kv_base + 2u * (uint32_t)(j - un.ulo); };
        auto wait_kv = [&](uint32_t idx) -> bool {
            return wait_bar(bar_addr(bars, C::B_KVFULL + idx % C::SLOTS), (idx / C::SLOTS) & 1,
                            abort_flag, 3);
        };
        auto release_kv = [&](uint32_t idx) {
            ptx::mma_commit(bar_addr(bars, C::B_KVEMPTY + idx % C::SLOTS));
        };

#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            if (!un.valid[q] || !ok) continue;
            ok = wait_bar(bar_addr(bars, C::B_QFULL + q), q_cnt[q] & 1, abort_flag, 6);
        }
        if (!ok) break;

        // S_q(x) is issued one key tile ahead of P_q V: the softmax of tile j
        // overlaps the S MMA of tile j + 1 (two S buffers per query tile).
        int ns[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) ns[q] = un.lo[q];
        int k_ready = un.ulo - 1;  // highest key tile waited for
        int k_rel = un.ulo;        // next key tile to hand back to the TMA warp

        for (int j = un.ulo; j < un.uhi && ok; ++j) {
            // 1. every S of key tiles <= j + 1
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                if (!un.valid[q]) continue;
                while (ns[q] < un.hi[q] && ns[q] <= j + 1) {
                    const int x = ns[q];
                    if (x > k_ready) {
                        if (!wait_kv(kidx(x))) { ok = false; break; }
                        k_ready = x;
                    }
                    const int b = (int)((t_cnt[q] + (uint32_t)(x - un.lo[q])) & 1u);
                    const uint32_t a0 = ptx::smem_addr(sQ + q * C::Q_BYTES);
                    const uint32_t b0 = ptx::smem_addr(sKV + (kidx(x) % C::SLOTS) * C::SLOT_BYTES);
                    const uint32_t d_tmem = tmem + C::s_col(q, b);
                    const uint64_t da = smem_desc(a0, 16), db = smem_desc(b0, 16);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        // 16-column steps: 32 bytes inside a 128-byte box, then the next box.
                        const uint32_t off_a = (uint32_t)(((kk >> 2) * C::Q_CHUNK + (kk & 3) * 32) >> 4);
                        const uint32_t off_b = (uint32_t)(((kk >> 2) * C::KV_CHUNK + (kk & 3) * 32) >> 4);
                        ptx::mma_ss(d_tmem, da + off_a, db + off_b, kIdescS, kk > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar_addr(bars, C::B_SFULL + 2 * q + b));
                    ++ns[q];
                    if (ns[q] == un.hi[q]) {  // last read of this Q tile in the unit
                        ptx::mma_commit(bar_addr(bars, C::B_QEMPTY + q));
                        ++q_cnt[q];
                    }
                }
                if (!ok) break;
            }
            if (!ok) break;
            // every S that reads key tiles <= k_ready has been issued
            while (k_rel <= k_ready) {
                release_kv(kidx(k_rel));
                ++k_rel;
            }
            // 2. O_q (+)= P_q V_j for every query tile that sees key tile j
            bool v_ready = false;
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                if (!un.valid[q] || j < un.lo[q] || j >= un.hi[q]) continue;
                if (!v_ready) {
                    if (!wait_kv(kidx(j) + 1)) { ok = false; break; }
                    v_ready = true;
                }
                const uint32_t t = t_cnt[q] + (uint32_t)(j - un.lo[q]);
                const int b = (int)(t & 1u);
                if (!wait_bar(bar_addr(bars, C::B_PFULL + 2 * q + b), (t >> 1) & 1u, abort_flag, 4)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const bool first = (j == un.lo[q]);
                if (first && o_used[q]) {
                    if (!wait_bar(bar_addr(bars, C::B_OFREE + q), ofree_cnt[q] & 1, abort_flag, 5)) {
                        ok = false;
                        break;
                    }
                    ++ofree_cnt[q];
                    ptx::tc_fence_after();
                }
                const uint32_t v0 = ptx::smem_addr(sKV + ((kidx(j) + 1) % C::SLOTS) * C::SLOT_BYTES);
                const uint32_t d_tmem = tmem + C::O_COL0 + (uint32_t)q * D;
                const uint32_t p_tmem = tmem + C::s_col(q, b);
                const uint64_t dv = smem_desc(v0, C::KV_CHUNK);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // 16 keys = two 8-row groups (2048 bytes) per step; P: 8 columns.
                    ptx::mma_ts(d_tmem, p_tmem + kk * 8, dv + (uint32_t)((kk * 2048) >> 4),
                                kIdescO, (!first || kk > 0) ? 1u : 0u);
                }
                ptx::mma_commit(bar_addr(bars, C::B_OFULL + q));
            }
            if (!ok) break;
            release_kv(kidx(j) + 1);
        }
        if (!ok) break;
        kv_it = kv_base + 2u * (uint32_t)(un.uhi - un.ulo);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            if (!un.valid[q]) continue;
            t_cnt[q] += (uint32_t)(un.hi[q] - un.lo[q]);
            o_used[q] = true;
        }
    }
    // Every MMA issued must finish before tensor memory is released.
    ptx::mma_commit(bar_addr(bars, C::B_DRAIN));
    wait_bar_drain(bar_addr(bars, C::B_DRAIN), 0);
}

// ---------------------------------------------------------------- softmax role

// One thread's row of an S tile (BN fp32 columns) from tensor memory.
template <int BN>
__device__ __forceinline__ void load_s_row(uint32_t taddr, uint32_t (&r)[BN]) {
    ptx::tmem_ld_x32<0>(taddr, r);
    ptx::tmem_ld_x32<32>(taddr + 32, r);
    if constexpr (BN == 128) {
        ptx::tmem_ld_x32<64>(taddr + 64, r);
        ptx::tmem_ld_x32<96>(taddr + 96, r);
    }
}

// One thread's row of P (BN 16-bit values packed in BN/2 columns) to tensor memory.
template <int BN>
__device__ __forceinline__ void store_p_row(uint32_t taddr, const uint32_t (&r)[BN / 2]) {
    ptx::tmem_st_x32<0>(taddr, r);
    if constexpr (BN == 128) ptx::tmem_st_x32<32>(taddr + 32, r);
}

template <int D, bool kFP16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    return kFP16 ? ptx::pack_f16x2(lo, hi) : ptx::pack_bf16x2(lo, hi);
}

// Hidden keys of a boundary tile (columns outside [c_lo, c_hi]) become -inf.
template <int BN>
__device__ __forceinline__ void apply_mask(uint32_t (&sr)[BN], int c_lo, int c_hi) {
#pragma unroll
    for (int i = 0; i < BN; ++i)
        if (i < c_lo || i > c_hi) sr[i] = __float_as_uint(-INFINITY);
}

// Row max of one S tile (raw scores; scale >= 0 preserves the order).  With
// kMasked, columns outside [c_lo, c_hi] are first set to -inf.
template <int BN, bool kMasked>
__device__ __forceinline__ float tile_row_max(uint32_t (&sr)[BN], int c_lo, int c_hi) {
    if constexpr (kMasked) {
#pragma unroll
        for (int i = 0; i < BN; ++i)
            if (i < c_lo || i > c_hi) sr[i] = __float_as_uint(-INFINITY);
    }
    float mx0 = __uint_as_float(sr[0]), mx1 = __uint_as_float(sr[1]);
    float mx2 = __uint_as_float(sr[2]), mx3 = __uint_as_float(sr[3]);
#pragma unroll
    for (int i = 4; i < BN; i += 8) {
        mx0 = ptx::max3(mx0, __uint_as_float(sr[i]), __uint_as_float(sr[i + 1]));
        mx1 = ptx::max3(mx1, __uint_as_float(sr[i + 2]), __uint_as_float(sr[i + 3]));
        if (i + 4 < BN) {
            mx2 = ptx::max3(mx2, __uint_as_float(sr[i + 4]), __uint_as_float(sr[i + 5]));
            mx3 = ptx::max3(mx3, __uint_as_float(sr[i + 6]), __uint_as_float(sr[i + 7]));
        }
    }
    return fmaxf(ptx::max3(mx0, mx1, mx2), mx3);
}

// p = 2^(s*c - m) for one row of a tile, packed to 16 bits into pk; adds the
// exact fp32 sum of p to l_exact (for the logsumexp) and the sum of the
// rounded 16-bit p to l_round (the divisor of O, so that the weights the
// P V product uses sum exactly to what O is divided by).
template <int BN, bool kFP16, bool kMasked>
__device__ __forceinline__ void tile_row_exp(const uint32_t (&sr)[BN], float c, float neg,
                                             uint32_t (&pk)[BN / 2], float &l_exact,
                                             float &l_round) {
    const uint64_t c2 = ptx::f32x2(c, c), n2 = ptx::f32x2(neg, neg);
    uint64_t le0 = ptx::f32x2(0.f, 0.f), le1 = le0;
    float lr0 = 0.f, lr1 = 0.f, lr2 = 0.f, lr3 = 0.f;
#pragma unroll
    for (int i = 0; i < BN; i += 2) {
        const float x0 = __uint_as_float(sr[i]), x1 = __uint_as_float(sr[i + 1]);
        float y0, y1;
        ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(x0, x1), c2, n2), y0, y1);
        float e0 = ptx::ex2_approx(y0);
        float e1 = ptx::ex2_approx(y1);
        if constexpr (kMasked) {  // hidden keys weigh exactly 0 (also when scale == 0)
            e0 = (x0 == -INFINITY) ? 0.f : e0;
            e1 = (x1 == -INFINITY) ? 0.f : e1;
        }
        const uint32_t pw = kFP16 ? ptx::pack_f16x2(e0, e1) : ptx::pack_bf16x2(e0, e1);
        pk[i / 2] = pw;
        if ((i >> 1) & 1)
            le1 = ptx::add_f32x2(le1, ptx::f32x2(e0, e1));
        else
            le0 = ptx::add_f32x2(le0, ptx::f32x2(e0, e1));
        float &acc = ((i >> 1) & 3) == 0 ? lr0 : ((i >> 1) & 3) == 1 ? lr1 : ((i >> 1) & 3) == 2 ? lr2 : lr3;
        acc = kFP16 ? ptx::add_f16x2_to_f32(pw, acc) : ptx::add_bf16x2_to_f32(pw, acc);
    }
    float a0, a1;
    ptx::unpack_f32x2(ptx::add_f32x2(le0, le1), a0, a1);
    l_exact += a0 + a1;
    l_round += (lr0 + lr1) + (lr2 + lr3);
}

template <int D, bool kFP16>
__device__ void softmax_role(const Params &p, int wg, uint32_t bars, uint32_t tmem,
                             volatile int *abort_flag) {
    using C = Cfg<D>;
    constexpr int NQ = C::NQ;
    constexpr int BN = C::BN;
    const int tid = threadIdx.x - wg * 128;                // query row within the tile
    const uint32_t lane_off = (uint32_t)((tid >> 5) * 32) << 16;  // this warp's TMEM lanes
    const int q = (NQ == 2) ? wg : 0;
    const float c = p.scale_log2;
    uint32_t t_cnt = 0;  // key tiles processed by this warpgroup (S/P buffer = t & 1)
    bool ok = true;

    for (int k = 0; ok; ++k) {
        const int u = unit_at(k);
        if (u >= p.n_units) break;
        Unit<D> un;
        decode_unit<D>(u, p, un);
        if (!un.exists[q]) continue;
        const int row = un.i0[q] + tid;
        const bool row_ok = row < p.Sq;
        const size_t row_flat = ((size_t)(un.b * p.H + un.h)) * (size_t)p.Sq + (size_t)row;
        if (!un.valid[q]) {
            // No key visible to any row of this tile: guarded output.
            if (row_ok) {
                uint8_t *orow = reinterpret_cast<uint8_t *>(p.o) + row_flat * D * 2;
#pragma unroll
                for (int cc = 0; cc < D / 8; ++cc) ptx::st_global_v4(orow + cc * 16, 0, 0, 0, 0);
                p.lse[row_flat] = -INFINITY;
            }
            continue;
        }
        // Visible key columns of this row, as absolute key indices [key_lo, key_hi].
        const int key_hi = (p.mask_kind == kMaskNone) ? p.Sk - 1 : min(row, p.Sk - 1);
        const int key_lo = (p.mask_kind == kMaskWindow) ? row - p.window + 1 : 0;

        float m_ref = -INFINITY;  // max the accumulator and sums are referenced to (log2 units)
        float l = 0.f;            // sum of the rounded P actually multiplied into O
        float l_exact = 0.f;      // fp32 sum of P (for the logsumexp)
        const uint32_t o_tmem = tmem + lane_off + C::O_COL0 + (uint32_t)q * D;

        uint32_t t = 0;  // this warpgroup's tile counter at the current key tile
        for (int j = un.lo[q]; j < un.hi[q]; ++j) {
            t = t_cnt++;
            const int b = (int)(t & 1u);
            if (!wait_bar(bar_addr(bars, C::B_SFULL + 2 * q + b), (t >> 1) & 1u, abort_flag, 7)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t s_tmem = tmem + lane_off + C::s_col(q, b);

            uint32_t sr[BN];
            load_s_row<BN>(s_tmem, sr);
            ptx::tmem_wait_ld();
            ptx::reg_fence<BN>(sr);

            const bool masked = tile_needs_mask<D>(un.i0[q], j, p);
            if (masked) apply_mask<BN>(sr, key_lo - j * BN, key_hi - j * BN);

            // Fast path: exponentiate against the current reference max without
            // looking for this tile's max.  Weights above 2^8 (the max grew by
            // more than the deferral bound) always push the tile's sum above
            // 2^8, so a sum within the bound proves the reference is still
            // valid; otherwise (and on a row's first tile, when there is no
            // reference yet) the tile takes the slow path below.
            uint32_t pk[BN / 2];
            float le_t = 0.f, lr_t = 0.f;  // this tile's exact and rounded sums
            bool slow = (j == un.lo[q]) || (m_ref == -INFINITY);
            if (!slow) {
                if (masked)
                    tile_row_exp<BN, kFP16, true>(sr, c, -m_ref, pk, le_t, lr_t);
                else
                    tile_row_exp<BN, kFP16, false>(sr, c, -m_ref, pk, le_t, lr_t);
                slow = !(le_t <= kRescaleBound);  // also catches inf
            }
            float alpha = 1.f;
            bool rescale = false;
            if (slow) {
                const float mx = tile_row_max<BN, false>(sr, 0, 0);
                const float m_tile = (mx == -INFINITY) ? -INFINITY : mx * c;
                const float m_new = fmaxf(m_ref, m_tile);
                bool redo = true;
                if (j == un.lo[q]) {
                    m_ref = m_new;
                } else if (m_new > m_ref + kRescaleLog2) {
                    alpha = ptx::ex2_approx(m_ref - m_new);  // 0 while m_ref is -inf
                    m_ref = m_new;
                    rescale = true;
                } else {
                    redo = false;  // the fast-path weights are within the bound
                }
                if (redo) {
                    const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
                    le_t = 0.f;
                    lr_t = 0.f;
                    if (masked)
                        tile_row_exp<BN, kFP16, true>(sr, c, neg, pk, le_t, lr_t);
                    else
                        tile_row_exp<BN, kFP16, false>(sr, c, neg, pk, le_t, lr_t);
                }
            }
            // O-barrier phases (one per P V of this query slot, numbered like t)
            // are consumed in order: phase t-1 (P V of the previous key tile) is
            // waited for before P of this tile is released, i.e. before P V of
            // tile t can exist.  S of this tile implies P V of tile t-2 is done,
            // so the barrier is then at phase t-1 or t and a parity wait on t-1
            // is unambiguous.  The first tile of a unit has nothing to wait for:
            // the previous unit's epilogue consumed its last phase.
            if (__any_sync(0xffffffffu, rescale)) {
                // O may be touched only once the previous P V has finished.
                if (!wait_bar(bar_addr(bars, C::B_OFULL + q), (t - 1u) & 1u, abort_flag, 8)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t ov[32];
                    ptx::tmem_ld_x32<0>(o_tmem + cc * 32, ov);
                    ptx::tmem_wait_ld();
                    ptx::reg_fence<32>(ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    ptx::tmem_st_x32<0>(o_tmem + cc * 32, ov);
                }
            }
            l = alpha * l + lr_t;
            l_exact = alpha * l_exact + le_t;
            store_p_row<BN>(s_tmem, pk);
            if (j > un.lo[q] &&
                !wait_bar(bar_addr(bars, C::B_OFULL + q), (t - 1u) & 1u, abort_flag, 10)) {
                ok = false;
                break;
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_addr(bars, C::B_PFULL + 2 * q + b));
        }
        if (!ok) break;

        // Epilogue: wait for the last P V (phase t; phase t-1 was consumed
        // above), divide by l once, store O and lse.
        if (!wait_bar(bar_addr(bars, C::B_OFULL + q), t & 1u, abort_flag, 9)) { ok = false; break; }
        ptx::tc_fence_after();
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        uint8_t *orow = reinterpret_cast<uint8_t *>(p.o) + row_flat * D * 2;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            ptx::tmem_ld_x32<0>(o_tmem + cc * 32, ov);
            ptx::tmem_wait_ld();
            ptx::reg_fence<32>(ov);
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                w[i] = pack2<D, kFP16>(__uint_as_float(ov[2 * i]) * inv_l,
                                       __uint_as_float(ov[2 * i + 1]) * inv_l);
            if (row_ok) {
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    ptx::st_global_v4(orow + cc * 64 + v4 * 16, w[4 * v4], w[4 * v4 + 1],
                                      w[4 * v4 + 2], w[4 * v4 + 3]);
            }
        }
        if (row_ok) p.lse[row_flat] = (l_exact > 0.f) ? (m_ref + log2f(l_exact)) * kLn2 : -INFINITY;
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_addr(bars, C::B_OFREE + q));
    }
}

// ---------------------------------------------------------------- kernel

template <int D, bool kFP16>
__global__ void __launch_bounds__(Cfg<D>::NUM_THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ Params p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem;
    uint8_t *sKV = smem + C::NQ * C::Q_BYTES;
    uint64_t *bar_mem = reinterpret_cast<uint64_t *>(smem + C::SMEM_TILES);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bar_mem + C::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    const uint32_t bars = ptx::smem_addr(bar_mem);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const uint32_t lane = ptx::lane_id();

    if (threadIdx.x == 0) {
        for (int q = 0; q < C::NQ; ++q) {
            ptx::mbar_init(bar_addr(bars, C::B_QFULL + q), 1);
            ptx::mbar_init(bar_addr(bars, C::B_QEMPTY + q), 1);
            ptx::mbar_init(bar_addr(bars, C::B_OFULL + q), 1);
            ptx::mbar_init(bar_addr(bars, C::B_OFREE + q), 128);
        }
        for (int s = 0; s < C::SLOTS; ++s) {
            ptx::mbar_init(bar_addr(bars, C::B_KVFULL + s), 1);
            ptx::mbar_init(bar_addr(bars, C::B_KVEMPTY + s), 1);
        }
        for (int b = 0; b < 2 * C::NQ; ++b) {
            ptx::mbar_init(bar_addr(bars, C::B_SFULL + b), 1);
            ptx::mbar_init(bar_addr(bars, C::B_PFULL + b), 128);
        }
        ptx::mbar_init(bar_addr(bars, C::B_DRAIN), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == C::MMA_WARP) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == C::TMA_WARP && lane == 0) {
        ptx::prefetch_tensormap(&p.tm_q);
        ptx::prefetch_tensormap(&p.tm_k);
        ptx::prefetch_tensormap(&p.tm_v);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp < 4 * C::NQ) {
        softmax_role<D, kFP16>(p, warp >> 2, bars, tmem, abort_flag);
    } else if (warp == C::MMA_WARP) {
        if (lane == 0) mma_role<D, kFP16>(p, sQ, sKV, bars, tmem, abort_flag);
    } else {
        if (lane == 0) tma_role<D>(p, sQ, sKV, bars, abort_flag);
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
