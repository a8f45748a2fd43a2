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
//   * a work unit is one 128-row query tile of one (batch, head); the host
//     deals the units to the CTAs (least loaded first) in groups of heads
//     whose K and V fit in a third of the L2, so each K/V byte comes from
//     DRAM about once;
//   * warp 10 streams the Q tile and a ring of K tiles, warp 11 a ring of V
//     tiles, by TMA (128-byte swizzle, 64-column boxes; at d = 256 the rings
//     hold 128-column halves of the tiles);
//   * warp 8 issues S = Q K^T (tcgen05, both operands in shared memory) into
//     the S buffers in tensor memory (two; one at d = 256), each as soon as
//     the softmax has read that buffer's previous tile; warp 9 issues
//     O += P V with P read from tensor memory (two P areas; one at d = 128);
//   * warps 0-7 are the softmax: warp w owns 16 rows (TMEM lanes) and every
//     key column of a tile in the 16-lane tcgen05.ld layout, where a row's
//     columns sit in one quad of threads, so max and sum take two shuffles
//     and the warps never synchronise during a unit; they mask boundary
//     tiles, exponentiate, write P (16-bit), rescale O in tensor memory when
//     the reference max moves, and run the epilogue (O / l through a bulk
//     tensor store for d <= 128, and lse).
//
// Rescaling is deferred until the running max has grown by more than 2^8
// (log2 units).  Until then the accumulator and the sums both stay referenced
// to the same stale max, so the final O_acc / l is unchanged (the pages note
// that FlashAttention-2 postpones most of the rescaling); the stale reference
// only lets unnormalised weights reach 2^8, far from fp32/bf16/fp16 limits.
// The tile max itself is only computed when needed: a weight above 2^8
// pushes the tile's sum above 2^8, so a tile whose sum stays within the bound
// is valid as computed against the current reference.
#pragma once

#include <stdint.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBM = 128;  // query rows per tile = M of every MMA = TMEM lanes
constexpr int kMaskNone = 0;
constexpr int kMaskCausal = 1;
constexpr int kMaskWindow = 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // default limit of a pipeline wait: 2 s
constexpr float kRescaleLog2 = 8.0f;              // rescale O when the max grows > 2^8
constexpr float kRescaleBound = 256.0f;           // 2^kRescaleLog2
constexpr float kLn2 = 0.693147180559945309f;

// Per-CTA control block in shared memory.
struct Ctl {
    volatile int abort;  // a role gave up waiting: the others stop too
    int pad;
    uint64_t limit_ns;   // how long a pipeline wait may take
};

// Device status word: 0 = fine; else 0x100 + the wait site that timed out.
// (This header is compiled into exactly one translation unit.)
__device__ int g_fa_status = 0;

constexpr int kMaxSchedGrid = 256;     // CTAs a precomputed schedule can describe
// Units a precomputed schedule can hold.  The lists travel in the kernel
// parameters, which every launch copies: 4,096 entries keep them at 9 KB
// (a 25 KB block measured 2 us more per launch on an empty kernel).
constexpr int kMaxSchedUnits = 4096;

struct Params {
    CUtensorMap tm_q;  // [B, H, Sq, d] 16-bit, box {64, 128, 1, 1}, 128-B swizzle
    CUtensorMap tm_k;  // [B, Hkv, Sk, d], box {64, BN, 1, 1}
    CUtensorMap tm_v;  // [B, Hkv, Sk, d], box {64, BN, 1, 1}
    CUtensorMap tm_o;  // [B, H, Sq, d] 16-bit, box {64, 128, 1, 1}, 128-B swizzle (d <= 128)
    void *o;           // [B, H, Sq, d] 16-bit
    float *lse;        // [B, H, Sq] fp32
    int B, H, Sq, Sk;
    int mask_kind, window;
    float scale_log2;  // scale * log2(e), kept positive (see the API)
    int n_qtiles;      // ceil(Sq / 128): units per (batch, head)
    int n_units;       // B * H * n_qtiles
    int heads_per_group;  // (batch, head) pairs scheduled together (K/V kept in L2)
    int kv_group;      // query heads per K/V head (H / Hkv; 1 = multi-head)
    int o_vec8;        // O is 32-byte aligned: 32-byte stores
    uint64_t wait_limit_ns;  // limit of every pipeline wait
    int stall_test;          // test only: the softmax's first wait is on a barrier nothing completes
    // Schedule: with sched = 1, CTA c runs units sched_ids[sched_off[c] ..
    // sched_off[c+1]) in that order (built on the host); else the snake order.
    int sched;
    uint16_t sched_off[kMaxSchedGrid + 1];
    uint16_t sched_ids[kMaxSchedUnits];
};
static_assert(sizeof(Params) <= 32764, "kernel parameter space");

template <int D>
struct Cfg {
    // 128-key tiles.  K and V tiles stream through two rings of KST and VST
    // slots, filling the shared memory left after Q; a slot holds one piece
    // of a tile: the whole tile at d <= 128, a 128-column half at d = 256,
    // where 64 KB tiles would leave room for one K and one V tile only.
    // The S product of a tile runs piece by piece (N = 128 throughout, so
    // the tensor core, not the shared-memory reads, sets its pace), and so
    // does its P V product (one 128-column half of O per piece).
    static constexpr int BN = 128;                       // keys per K/V tile
    static constexpr int HALF = BN / 2;                  // key columns per softmax warpgroup
    static constexpr int NPC = (D == 256) ? 2 : 1;       // pieces per K or V tile
    static constexpr int KST = (D == 64) ? 4 : (D == 128) ? 2 : 3;  // K ring slots (pieces)
    static constexpr int VST = (D == 64) ? 4 : 2;                   // V ring slots (pieces)
    // Warps 0-7: two softmax warpgroups (warpgroup h owns key columns
    // [h*HALF, (h+1)*HALF) of every tile, all 128 rows); warp 8: S MMAs;
    // warp 9: P V MMAs; warp 10: TMA of Q and K; warp 11: TMA of V.
    static constexpr int NUM_SOFTMAX = 256;
    static constexpr int NUM_WARPS = 12;
    static constexpr int NUM_THREADS = 32 * NUM_WARPS;
    static constexpr int S_WARP = 8;
    static constexpr int PV_WARP = 9;
    static constexpr int TMA_WARP = 10;
    static constexpr int TMA_V_WARP = 11;
    static constexpr int CHUNKS = D / 64;              // 64-column (128-byte) boxes per row
    static constexpr int Q_CHUNK = kBM * 128;          // bytes of one Q box
    static constexpr int KV_CHUNK = BN * 128;          // bytes of one K or V box
    static constexpr int Q_BYTES = kBM * D * 2;
    static constexpr int TILE_BYTES = BN * D * 2;      // one K or one V tile
    static constexpr int PIECE_COLS = D / NPC;         // columns of one piece
    static constexpr int PIECE_CHUNKS = PIECE_COLS / 64;
    static constexpr int PIECE_BYTES = TILE_BYTES / NPC;
    // d <= 128: each V slot carries one more 64-column box after the tile's
    // boxes, whose first column is all ones (written once at the kernel's
    // start).  For bf16 the P V product then runs with N = D + 16 and also
    // accumulates, in O's column D, the sum of the rounded weights it used --
    // the divisor of O -- so the softmax spends no additions on it.
    static constexpr bool SUMCOL = (D <= 128);
    static constexpr int V_SLOT_BYTES = PIECE_BYTES + (SUMCOL ? KV_CHUNK : 0);
    // Tensor memory: NSB S buffers from column 0 (tile t in buffer t % NSB),
    // O from O_COL0, and two P areas (BN/2 columns each, two 16-bit values
    // per column) at P_COL0 and P_COL0 + P_STRIDE; P of key tile t goes to
    // area t & 1, so the softmax of tile t+1 never waits for P V of tile t.
    // d = 256: O takes 256 columns, leaving one S buffer; the tensor core's
    // 2,048 cycles per tile then exceed the softmax's, and S of tile t+1
    // (issued once the softmax has copied S of tile t out) is ready before
    // the softmax needs it.
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int NSB = (D == 256) ? 1 : 2;
    static constexpr uint32_t O_COL0 = (D == 256) ? 128 : 256;
    static constexpr uint32_t O_COLS = D + (SUMCOL ? 16 : 0);  // O, and for bf16 its sum column D
    // d = 128: one P area (its second area's columns hold O's sum column);
    // P of tile t+1 is written once P V of tile t has read the area
    // (measured +2 % on fp16 even without the sum column).
    static constexpr uint32_t P_COL0 = (D == 128) ? 448 : 384;
    static constexpr uint32_t P_STRIDE = (D == 128) ? 0 : 64;
    // Barrier indices.
    static constexpr int B_QFULL = 0;
    static constexpr int B_QEMPTY = 1;
    static constexpr int B_KFULL = 2;                   // [KST]: K slot loaded
    static constexpr int B_KEMPTY = B_KFULL + KST;      // [KST]: K slot read by its S MMAs
    static constexpr int B_VFULL = B_KEMPTY + KST;      // [VST]: V slot loaded
    static constexpr int B_VEMPTY = B_VFULL + VST;      // [VST]: V slot read by its P V MMAs
    static constexpr int B_SFULL = B_VEMPTY + VST;      // [2]: S buffer b computed
    static constexpr int B_SFREE = B_SFULL + 2;         // [2]: S buffer b read by the softmax
    static constexpr int B_PFULL = B_SFREE + 2;         // [2]: P area b written
    static constexpr int B_OFULL = B_PFULL + 2;         // [2]: P V from P area b done
    static constexpr int B_OFINAL = B_OFULL + 2;        // one phase per unit: last P V done
    static constexpr int B_OFREE = B_OFINAL + 1;        // epilogue has read O
    static constexpr int B_DRAIN = B_OFREE + 1;         // [2]: each issuer's MMAs finished
    static constexpr int B_NEVER = B_DRAIN + 2;         // no arrivals (the stall test's wait)
    static constexpr int NUM_BARS = B_NEVER + 1;
    // d <= 128: the epilogue stages the normalised O tile (the Q tile's shape)
    // in shared memory for one bulk tensor store; d = 256 has no room for it
    // and stores rows directly.
    static constexpr int O_STAGE_BYTES = (D <= 128) ? Q_BYTES : 0;
    static constexpr int SMEM_TILES = Q_BYTES + KST * PIECE_BYTES + VST * V_SLOT_BYTES + O_STAGE_BYTES;
    static constexpr int XCH_BYTES = 3 * kBM * 4;  // per row: two sums and the reference max
    static constexpr int SMEM_BYTES = 1024 + SMEM_TILES + NUM_BARS * 8 + 24 + XCH_BYTES;
    static_assert(O_COL0 + O_COLS <= P_COL0 && P_COL0 + P_STRIDE + BN / 2 <= TMEM_COLS,
                  "tensor memory overflow");
    static_assert(P_STRIDE == 0 || BN / 2 <= (int)P_STRIDE, "P areas overlap");
    static_assert(NSB * BN <= (int)O_COL0, "S buffers overlap O");
    static_assert(PIECE_COLS % 64 == 0 && D % NPC == 0, "pieces of whole 64-column boxes");
    static_assert(SMEM_BYTES <= 232448, "shared memory overflow");
};

// ---------------------------------------------------------------- helpers

// Shared-memory matrix descriptor, 128-byte swizzle, tcgen05 format.
// K-major operands: rows of 128 bytes, 8-row groups 1024 bytes apart (SBO);
// the leading offset is unused.  MN-major (V as the B operand of P V): 8-row
// groups along K 1024 bytes apart (SBO), 64-element column boxes `lbo` apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo = 1024) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
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
// word) after the control block's limit, or as soon as another role has
// aborted.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, Ctl *ctl,
                                           int site) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (ctl->abort) return false;
        if (ptx::globaltimer_ns() - t0 > ctl->limit_ns) {
            ctl->abort = 1;
            atomicCAS(&g_fa_status, 0, 0x100 + site);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Ctl *ctl,
                                         int site) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, ctl, site);
}

// Same bounded wait for the TMA producers, whose waits are off the critical
// path: a short sleep between polls leaves the issue slots of the
// sub-partition to the softmax warps that share it.
__device__ __noinline__ bool wait_bar_backoff(uint32_t bar, uint32_t parity, Ctl *ctl,
                                              int site) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (ctl->abort) return false;
        if (ptx::globaltimer_ns() - t0 > ctl->limit_ns) {
            ctl->abort = 1;
            atomicCAS(&g_fa_status, 0, 0x100 + site);
            return false;
        }
        __nanosleep(256);
    }
}

// Wait used only while shutting down after an abort: ignores the abort flag.
__device__ __noinline__ void wait_bar_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) return;
    }
}

// Unit k of this CTA (n_units once the CTA has no more): from the host's
// schedule, or else in a snake order (even rounds left to right, odd rounds
// right to left, so that with units sorted longest-first each CTA's sum of
// work stays close to the others').
__device__ __forceinline__ int unit_at(int k, const Params &p) {
    if (p.sched) {
        const int o = (int)p.sched_off[blockIdx.x] + k;
        return o < (int)p.sched_off[blockIdx.x + 1] ? (int)p.sched_ids[o] : p.n_units;
    }
    const int G = gridDim.x, c = blockIdx.x;
    return (k & 1) ? k * G + (G - 1 - c) : k * G + c;
}

// One work unit: query tile [i0, i0 + 128) of head (b, h) and the key tiles
// [lo, hi) it has to visit (tiles the mask hides entirely are skipped:
// causal keys past the tile's last row, window keys before its first row's
// window).  valid = the tile sees at least one key tile.
struct Unit {
    int b, h, kvh, i0, lo, hi;  // kvh: the K/V head query head h reads
    bool valid;
};

template <int D>
__device__ __forceinline__ Unit decode_unit(int u, const Params &p) {
    constexpr int BN = Cfg<D>::BN;
    Unit un;
    // Units come in groups of heads_per_group (batch, head) pairs whose K and
    // V fit in L2 together; inside a group, longest query tiles first
    // (causal / window work grows with the tile index), heads interleaved.
    const int BH = p.B * p.H;
    const int G = p.heads_per_group;
    const int grp = u / (G * p.n_qtiles);
    const int h0 = grp * G;
    const int Gg = min(G, BH - h0);  // heads in this (possibly last, smaller) group
    const int idx = u - h0 * p.n_qtiles;
    const int gi = idx / Gg;
    const int bh = h0 + (idx - gi * Gg);
    const int g = p.n_qtiles - 1 - gi;
    un.b = bh / p.H;
    un.h = bh - un.b * p.H;
    un.kvh = un.h / p.kv_group;
    un.i0 = g * kBM;
    const int row_end = min(un.i0 + kBM, p.Sq);
    int key_end = p.Sk;
    if (p.mask_kind != kMaskNone) key_end = min(p.Sk, row_end);
    int key_beg = 0;
    if (p.mask_kind == kMaskWindow) key_beg = max(0, un.i0 - p.window + 1);
    un.valid = key_beg < key_end;
    un.lo = un.valid ? key_beg / BN : 0;
    un.hi = un.valid ? (key_end + BN - 1) / BN : 0;
    return un;
}

// ---------------------------------------------------------------- TMA roles

// Loads tile `key0 / BN` of a K or V tensor, piece by piece, into the next
// slots of its ring (the whole warp waits for each slot, one lane issues).
// `it` counts pieces.
template <int D>
__device__ __forceinline__ bool load_kv_tile(const CUtensorMap *tm, uint8_t *ring, int slot_bytes, uint32_t bars,
                                             int full0, int empty0, int nslots, uint32_t &it,
                                             int key0, const Unit &un, bool leader, uint64_t pol,
                                             Ctl *ctl) {
    using C = Cfg<D>;
#pragma unroll
    for (int pc = 0; pc < C::NPC; ++pc) {
        const uint32_t slot = it % (uint32_t)nslots;
        if (!wait_bar_backoff(bar_addr(bars, empty0 + (int)slot), ((it / (uint32_t)nslots) & 1) ^ 1,
                              ctl, 2))
            return false;
        if (leader) {
            const uint32_t fb = bar_addr(bars, full0 + (int)slot);
            ptx::mbar_arrive_expect_tx(fb, C::PIECE_BYTES);
            const uint32_t dst = ptx::smem_addr(ring + slot * slot_bytes);
#pragma unroll
            for (int c = 0; c < C::PIECE_CHUNKS; ++c)
                ptx::tma_load_4d(dst + c * C::KV_CHUNK, tm, fb, pc * C::PIECE_COLS + c * 64, key0, un.kvh,
                                 un.b, pol);
        }
        ++it;
    }
    return true;
}

// Waits until every copy into a ring that was issued has landed (slot s of a
// ring with m slots has been filled ceil((it - s) / m) times).
__device__ __forceinline__ void drain_ring(uint32_t bars, int full0, int nslots, uint32_t it) {
    for (int sl = 0; sl < nslots; ++sl) {
        const uint32_t fills = it > (uint32_t)sl ? (it - (uint32_t)sl + nslots - 1) / (uint32_t)nslots : 0u;
        if (fills) wait_bar_drain(bar_addr(bars, full0 + sl), (fills - 1) & 1);
    }
}

// Q and K producer: per unit the Q tile, then the unit's key tiles in order.
// V has its own producer warp, so a key tile never waits behind a value slot.
template <int D>
__device__ void tma_qk_role(const Params &p, uint8_t *sQ, uint8_t *sK, uint32_t bars,
                            Ctl *ctl) {
    using C = Cfg<D>;
    const bool leader = ptx::lane_id() == 0;
    const uint64_t pol_kv = ptx::policy_evict_last();
    const uint64_t pol_q = ptx::policy_evict_first();
    uint32_t k_it = 0;   // K tiles loaded so far
    uint32_t q_cnt = 0;  // Q tiles loaded so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int u = unit_at(k, p);
        if (u >= p.n_units) break;
        const Unit un = decode_unit<D>(u, p);
        if (!un.valid) continue;
        if (!wait_bar_backoff(bar_addr(bars, C::B_QEMPTY), (q_cnt & 1) ^ 1, ctl, 1)) {
            ok = false;
            break;
        }
        if (leader) {
            const uint32_t fb = bar_addr(bars, C::B_QFULL);
            ptx::mbar_arrive_expect_tx(fb, C::Q_BYTES);
            const uint32_t dst = ptx::smem_addr(sQ);
#pragma unroll
            for (int c = 0; c < C::CHUNKS; ++c)
                ptx::tma_load_4d(dst + c * C::Q_CHUNK, &p.tm_q, fb, c * 64, un.i0, un.h, un.b, pol_q);
        }
        ++q_cnt;
        for (int j = un.lo; j < un.hi && ok; ++j)
            ok = load_kv_tile<D>(&p.tm_k, sK, C::PIECE_BYTES, bars, C::B_KFULL, C::B_KEMPTY, C::KST, k_it, j * C::BN, un,
                                 leader, pol_kv, ctl);
    }
    if (!ok) {  // let every copy already issued land before the CTA can exit
        drain_ring(bars, C::B_KFULL, C::KST, k_it);
        if (q_cnt) wait_bar_drain(bar_addr(bars, C::B_QFULL), (q_cnt - 1) & 1);
    }
}

// V producer: the units' value tiles in order.
template <int D>
__device__ void tma_v_role(const Params &p, uint8_t *sV, uint32_t bars, Ctl *ctl) {
    using C = Cfg<D>;
    const bool leader = ptx::lane_id() == 0;
    const uint64_t pol_kv = ptx::policy_evict_last();
    uint32_t v_it = 0;  // V tiles loaded so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int u = unit_at(k, p);
        if (u >= p.n_units) break;
        const Unit un = decode_unit<D>(u, p);
        if (!un.valid) continue;
        for (int j = un.lo; j < un.hi && ok; ++j)
            ok = load_kv_tile<D>(&p.tm_v, sV, C::V_SLOT_BYTES, bars, C::B_VFULL, C::B_VEMPTY, C::VST, v_it, j * C::BN, un,
                                 leader, pol_kv, ctl);
    }
    if (!ok) drain_ring(bars, C::B_VFULL, C::VST, v_it);
}

// ---------------------------------------------------------------- MMA roles

// S issuer: S_b = Q K^T for every key tile, into buffer b = t % NSB as soon
// as the softmax has read that buffer's previous tile, piece by piece of K.
template <int D, bool kFP16>
__device__ void mma_s_role(const Params &p, uint8_t *sQ, uint8_t *sK, uint32_t bars,
                           uint32_t tmem, Ctl *ctl) {
    using C = Cfg<D>;
    constexpr int BN = C::BN;
    constexpr uint32_t kIdescS = make_idesc(kBM, BN, kFP16, false);
    const bool leader = ptx::lane_id() == 0;  // the whole warp waits, one lane issues
    const uint64_t dq = smem_desc(ptx::smem_addr(sQ), 16);
    const uint32_t k_addr = ptx::smem_addr(sK);
    uint32_t k_it = 0;   // K pieces consumed
    uint32_t t_cnt = 0;  // key tiles issued (S buffer = t % NSB)
    uint32_t q_cnt = 0;  // Q tiles consumed
    bool ok = true;

    for (int k = 0; ok; ++k) {
        const int u = unit_at(k, p);
        if (u >= p.n_units) break;
        const Unit un = decode_unit<D>(u, p);
        if (!un.valid) continue;
        const int n = un.hi - un.lo;
        if (!wait_bar(bar_addr(bars, C::B_QFULL), q_cnt & 1, ctl, 6)) { ok = false; break; }
        for (int i = 0; i < n && ok; ++i) {
            const uint32_t t = t_cnt + (uint32_t)i;
            const uint32_t b = t % (uint32_t)C::NSB;
            const uint32_t d_tmem = tmem + b * BN;
#pragma unroll 1
            for (int pc = 0; pc < C::NPC; ++pc, ++k_it) {
                const uint32_t slot = k_it % C::KST;
                if (!wait_bar(bar_addr(bars, C::B_KFULL + (int)slot), (k_it / C::KST) & 1, ctl, 3)) {
                    ok = false;
                    break;
                }
                if (pc == 0 && t >= (uint32_t)C::NSB &&  // the softmax has read tile t-NSB out of this buffer
                    !wait_bar(bar_addr(bars, C::B_SFREE + (int)b), ((t / C::NSB) - 1u) & 1u, ctl, 12)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint64_t dk = smem_desc(k_addr + slot * C::PIECE_BYTES, 16);
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < C::PIECE_COLS / 16; ++kk) {
                        // 16-column steps: 32 bytes inside a 128-byte box, then the
                        // next box (Q: column step gk of the whole row, K: kk of the piece).
                        const int gk = pc * (C::PIECE_COLS / 16) + kk;
                        const uint32_t off_a = (uint32_t)(((gk >> 2) * C::Q_CHUNK + (gk & 3) * 32) >> 4);
                        const uint32_t off_b = (uint32_t)(((kk >> 2) * C::KV_CHUNK + (kk & 3) * 32) >> 4);
                        ptx::mma_ss(d_tmem, dq + off_a, dk + off_b, kIdescS, (pc > 0 || kk > 0) ? 1u : 0u);
                    }
                    if (pc + 1 == C::NPC) {
                        ptx::mma_commit(bar_addr(bars, C::B_SFULL + (int)b));
                        if (i + 1 == n) ptx::mma_commit(bar_addr(bars, C::B_QEMPTY));  // last read of Q
                    }
                    ptx::mma_commit(bar_addr(bars, C::B_KEMPTY + (int)slot));
                }
                __syncwarp();
            }
        }
        if (!ok) break;
        t_cnt += (uint32_t)n;
        ++q_cnt;
    }
    if (leader) ptx::mma_commit(bar_addr(bars, C::B_DRAIN));
    __syncwarp();
    wait_bar_drain(bar_addr(bars, C::B_DRAIN), 0);
}

// P V issuer: O (+)= P V for every key tile, as soon as the softmax has
// written P.
template <int D, bool kFP16>
__device__ void mma_pv_role(const Params &p, uint8_t *sV, uint32_t bars, uint32_t tmem,
                            Ctl *ctl) {
    using C = Cfg<D>;
    constexpr int BN = C::BN;
    // One product per piece: N = the piece's columns of O; bf16 with the sum
    // column: N = D + 16 (the ones box follows the tile's boxes).
    constexpr uint32_t kIdescO =
        make_idesc(kBM, (C::SUMCOL && !kFP16) ? (int)C::O_COLS : C::PIECE_COLS, kFP16, true);
    const bool leader = ptx::lane_id() == 0;  // the whole warp waits, one lane issues
    const uint32_t v_addr = ptx::smem_addr(sV);
    const uint32_t o_tmem = tmem + C::O_COL0;
    const uint32_t p_tmem = tmem + C::P_COL0;
    uint32_t v_it = 0;       // V pieces consumed
    uint32_t t_cnt = 0;      // key tiles processed (one P V each)
    uint32_t ofree_cnt = 0;  // epilogues waited for
    bool o_used = false;
    bool ok = true;

    for (int k = 0; ok; ++k) {
        const int u = unit_at(k, p);
        if (u >= p.n_units) break;
        const Unit un = decode_unit<D>(u, p);
        if (!un.valid) continue;
        const int n = un.hi - un.lo;
        for (int i = 0; i < n && ok; ++i) {
            const uint32_t t = t_cnt + (uint32_t)i;
            // P of tile t is in area t & 1; that area's barrier completes once per
            // two tiles, and the softmax cannot write P of tile t+2 before this
            // P V has run, so the parity wait is unambiguous.
            const uint32_t pb = t & 1u;
            if (!wait_bar(bar_addr(bars, C::B_VFULL + (int)(v_it % C::VST)), (v_it / C::VST) & 1, ctl, 3) ||
                !wait_bar(bar_addr(bars, C::B_PFULL + (int)pb), (t >> 1) & 1u, ctl, 4)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            if (i == 0 && o_used) {
                if (!wait_bar(bar_addr(bars, C::B_OFREE), ofree_cnt & 1, ctl, 5)) {
                    ok = false;
                    break;
                }
                ++ofree_cnt;
                ptx::tc_fence_after();
            }
#pragma unroll 1
            for (int pc = 0; pc < C::NPC; ++pc, ++v_it) {
                const uint32_t slot = v_it % C::VST;
                if (pc > 0) {  // the first piece was waited for above
                    if (!wait_bar(bar_addr(bars, C::B_VFULL + (int)slot), (v_it / C::VST) & 1, ctl, 3)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                }
                const uint64_t dv = smem_desc(v_addr + slot * C::V_SLOT_BYTES, C::KV_CHUNK);
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        // 16 keys = two 8-row groups (2048 bytes) of V; P: 8 columns.
                        ptx::mma_ts(o_tmem + (uint32_t)(pc * C::PIECE_COLS), p_tmem + pb * C::P_STRIDE + kk * 8,
                                    dv + (uint32_t)((kk * 2048) >> 4), kIdescO, (i > 0 || kk > 0) ? 1u : 0u);
                    }
                    if (pc + 1 == C::NPC) {
                        ptx::mma_commit(bar_addr(bars, C::B_OFULL + (int)pb));
                        if (i + 1 == n) ptx::mma_commit(bar_addr(bars, C::B_OFINAL));
                    }
                    ptx::mma_commit(bar_addr(bars, C::B_VEMPTY + (int)slot));
                }
                __syncwarp();
            }
        }
        if (!ok) break;
        t_cnt += (uint32_t)n;
        o_used = true;
    }
    if (leader) ptx::mma_commit(bar_addr(bars, C::B_DRAIN + 1));
    __syncwarp();
    wait_bar_drain(bar_addr(bars, C::B_DRAIN + 1), 0);
}

// ---------------------------------------------------------------- softmax role

// Softmax warp w (0..7) owns the 16 TMEM lanes [32 (w & 3) + 16 (w >> 2), +16)
// -- 16 query rows -- and every key column of each S tile.  In the 16-lane
// tcgen05 shapes, thread t holds rows t/4 and t/4 + 8 of that block; a row's
// columns are spread over the 4 threads of a quad, so its max and sum are
// combined with two shuffles and the softmax warps never wait for one another
// during a unit.  The epilogue uses the one-row-per-thread 32x32b shape (warp
// w: rows 32 (w & 3) + lane, O columns half w >> 2), so the two warps that own
// a 32-row block meet once per unit on named barrier 1 + (w & 3) to hand each
// other the row sums.
constexpr uint32_t kPairBar0 = 1;
constexpr uint32_t kPairThreads = 64;
// Barrier of all 256 softmax threads around the staged O tile.
constexpr uint32_t kEpilogueBar = 5;

template <bool kFP16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    return kFP16 ? ptx::pack_f16x2(lo, hi) : ptx::pack_bf16x2(lo, hi);
}

// True if some (row, key) pair of this query tile x N keys from kc is hidden.
template <int N>
__device__ __forceinline__ bool cols_need_mask(int i0, int kc, const Params &p) {
    if (kc + N > p.Sk) return true;
    if (p.mask_kind == kMaskNone) return false;
    if (kc + N - 1 > i0) return true;
    if (p.mask_kind == kMaskWindow && kc <= i0 + kBM - 1 - p.window) return true;
    return false;
}

// Register e of a thread's NR tile registers (16x256b layout) holds column
// 8 (e / 4) + 2 tq + (e & 1) of row a (e & 2 == 0) or row b.  Hidden keys --
// columns outside the row's [lo, hi] -- become -inf, whose weight
// 2^(-inf * c - m) is exactly 0 for the positive exponent scale c.
template <int NR>
__device__ __forceinline__ void quad_mask(uint32_t (&sr)[NR], int tq, int lo_a, int hi_a, int lo_b,
                                          int hi_b) {
#pragma unroll
    for (int e = 0; e < NR; ++e) {
        const int col = 8 * (e >> 2) + 2 * tq + (e & 1);
        const bool hid = (e & 2) ? (col < lo_b || col > hi_b) : (col < lo_a || col > hi_a);
        if (hid) sr[e] = __float_as_uint(-INFINITY);
    }
}

// Max over the thread's columns of row a (ma) and row b (mb), then over the
// quad: every thread of the quad ends with the two full-row maxima.
template <int NR>
__device__ __forceinline__ void quad_row_max(const uint32_t (&sr)[NR], float &ma, float &mb) {
    float a0 = __uint_as_float(sr[0]), a1 = __uint_as_float(sr[1]);
    float b0 = __uint_as_float(sr[2]), b1 = __uint_as_float(sr[3]);
#pragma unroll
    for (int e = 4; e < NR; e += 8) {
        a0 = ptx::max3(a0, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
        b0 = ptx::max3(b0, __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
        if (e + 4 < NR) {
            a1 = ptx::max3(a1, __uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5]));
            b1 = ptx::max3(b1, __uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7]));
        }
    }
    ma = fmaxf(a0, a1);
    mb = fmaxf(b0, b1);
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
}

// p = 2^(s*c - m) for the thread's NR scores (rows a and b, references ma and
// mb given as na = -ma, nb = -mb), packed to 16 bits into pk in the 16x128b
// register order (pk[2k] row a, pk[2k+1] row b of packed column 4k + tq).
// Adds the exact fp32 sums of p to le_a / le_b (for the logsumexp) and to
// lr_a / lr_b the divisor of O: for bf16 the sum of the rounded 16-bit p, so
// that the weights the P V product uses sum exactly to what O is divided by
// (bf16 keeps only 8 significant bits, enough for a dominant weight's
// rounding to show in O); fp16's 11 bits make that negligible, so fp16
// divides by the exact sum.
template <int NR, bool kFP16, bool kRoundedSum = !kFP16>
__device__ __forceinline__ void quad_exp(const uint32_t (&sr)[NR], float c, float na, float nb,
                                         uint32_t (&pk)[NR / 2], float &le_a, float &le_b,
                                         float &lr_a, float &lr_b) {
    const uint64_t c2 = ptx::f32x2(c, c);
    const uint64_t na2 = ptx::f32x2(na, na), nb2 = ptx::f32x2(nb, nb);
    uint64_t sa = ptx::f32x2(0.f, 0.f), sb = sa;
    float ra0 = 0.f, ra1 = 0.f, rb0 = 0.f, rb1 = 0.f;
#pragma unroll
    for (int e = 0; e < NR; e += 2) {
        const bool row_b = (e & 2) != 0;
        float y0, y1;
        ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                         c2, row_b ? nb2 : na2),
                          y0, y1);
        const float e0 = ptx::ex2_approx(y0);
        const float e1 = ptx::ex2_approx(y1);
        const uint32_t pw = pack2<kFP16>(e0, e1);
        pk[e / 2] = pw;
        if (row_b)
            sb = ptx::add_f32x2(sb, ptx::f32x2(e0, e1));
        else
            sa = ptx::add_f32x2(sa, ptx::f32x2(e0, e1));
        if constexpr (kRoundedSum) {
            const bool odd = (e >> 2) & 1;
            float &acc = row_b ? (odd ? rb1 : rb0) : (odd ? ra1 : ra0);
            acc = ptx::add_bf16x2_to_f32(pw, acc);
        }
    }
    float a0, a1, b0, b1;
    ptx::unpack_f32x2(sa, a0, a1);
    ptx::unpack_f32x2(sb, b0, b1);
    le_a += a0 + a1;
    le_b += b0 + b1;
    if constexpr (!kRoundedSum) {
        lr_a += a0 + a1;
        lr_b += b0 + b1;
    } else {
        lr_a += ra0 + ra1;
        lr_b += rb0 + rb1;
    }
}

// P of one tile (this thread's packed pairs) into its area of tensor memory.
template <int NR>
__device__ __forceinline__ void store_p(uint32_t col, const uint32_t (&pk)[NR / 2]) {
    if constexpr (NR == 64)
        ptx::tmem_st_16x128b_x16<0>(col, pk);
    else
        ptx::tmem_st_16x128b_x8<0>(col, pk);
}

// Sum over the quad (all 4 threads end with the total).
__device__ __forceinline__ float quad_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}

// A unit's epilogue: wait for its last P V; full-row sums over the quad,
// handed through shared memory to the one-row-per-thread layout; divide by l
// once; store this warp's half of the O row (and lse).
template <int D, bool kFP16>
__device__ __noinline__ void softmax_epilogue(const Params &p, uint32_t bars, Ctl *ctl, float *xch,
                                              uint8_t *sO, uint32_t o_tmem, uint32_t u_cnt, int i0,
                                              int hd, int bt, size_t row_flat, bool row_ok,
                                              uint8_t *ohalf, float m_a, float m_b, float l_a,
                                              float l_b, float le_a, float le_b) {
    using C = Cfg<D>;
    const int warp = (int)(threadIdx.x >> 5), t = (int)(threadIdx.x & 31);
    const int qw = warp & 3, hh = warp >> 2;
    const int tq = t & 3;
    const int ra = 32 * qw + 16 * hh + (t >> 2), rb = ra + 8;
    const int re = 32 * qw + t;
    const uint32_t pair_bar = kPairBar0 + (uint32_t)qw;
    float *xl = xch, *xle = xch + kBM, *xm = xch + 2 * kBM;
    wait_bar(bar_addr(bars, C::B_OFINAL), u_cnt & 1u, ctl, 9);  // u_cnt: units finished before
    ptx::tc_fence_after();
    {
        const float sa = quad_sum(l_a), sb = quad_sum(l_b);
        const float ea = kFP16 ? sa : quad_sum(le_a), eb = kFP16 ? sb : quad_sum(le_b);
        ptx::named_bar_sync(pair_bar, kPairThreads);  // the previous unit's values fully read
        if (tq == 0) {
            xl[ra] = sa;
            xl[rb] = sb;
            xle[ra] = ea;
            xle[rb] = eb;
            xm[ra] = m_a;
            xm[rb] = m_b;
        }
        ptx::named_bar_sync(pair_bar, kPairThreads);
    }
    float l_all = xl[re];
    const float le_all = xle[re], m_ref = xm[re];
    if constexpr (C::SUMCOL && !kFP16) {
        // the divisor the P V products accumulated in O's column D (o_tmem
        // addresses this warp's half of the row, at column hh * D/2)
        l_all = __uint_as_float(ptx::tmem_ld_x1(o_tmem - (uint32_t)(hh * (D / 2)) + D));
        ptx::tmem_wait_ld();
    }
    const float inv_l = (l_all > 0.f) ? 1.f / l_all : 0.f;
    if constexpr (C::O_STAGE_BYTES > 0) {
        // Normalise this thread's D/2 columns of O into registers, release
        // O to the next unit's P V, then stage the tile in shared memory in
        // the tensor map's layout (64-column boxes of 128-byte rows, 16-byte
        // chunks swizzled by row & 7) and write it with one bulk store.
        // Rows past Sq fall outside the tensor and are not written.
        uint32_t w[D / 4];
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
            uint32_t ov[32];
            ptx::tmem_ld_x32<0>(o_tmem + cc * 32, ov);
            ptx::tmem_wait_ld();
            ptx::reg_fence<32>(ov);
#pragma unroll
            for (int e = 0; e < 16; ++e)
                w[cc * 16 + e] = pack2<kFP16>(__uint_as_float(ov[2 * e]) * inv_l,
                                              __uint_as_float(ov[2 * e + 1]) * inv_l);
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_addr(bars, C::B_OFREE));
        const uint32_t so = ptx::smem_addr(sO);
        if (threadIdx.x == 0) ptx::bulk_wait_read_all();  // the previous tile has left sO
        ptx::named_bar_sync(kEpilogueBar, C::NUM_SOFTMAX);
#pragma unroll
        for (int cidx = 0; cidx < D / 16; ++cidx) {
            const int col = hh * (D / 2) + cidx * 8;  // first of the chunk's 8 columns
            const uint32_t addr = so + (uint32_t)((col >> 6) * (kBM * 128) + re * 128 +
                                                  ((((col & 63) >> 3) ^ (re & 7)) << 4));
            ptx::st_shared_v4(addr, w[4 * cidx], w[4 * cidx + 1], w[4 * cidx + 2], w[4 * cidx + 3]);
        }
        ptx::fence_proxy_async_smem();
        ptx::named_bar_sync(kEpilogueBar, C::NUM_SOFTMAX);
        if (threadIdx.x == 0) {
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx)
                ptx::tma_store_4d(&p.tm_o, so + bx * (kBM * 128), bx * 64, i0, hd, bt);
            ptx::bulk_commit_group();
        }
    } else {
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
            uint32_t ov[32];
            ptx::tmem_ld_x32<0>(o_tmem + cc * 32, ov);
            ptx::tmem_wait_ld();
            ptx::reg_fence<32>(ov);
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                w[e] = pack2<kFP16>(__uint_as_float(ov[2 * e]) * inv_l,
                                    __uint_as_float(ov[2 * e + 1]) * inv_l);
            if (row_ok) {
                uint8_t *dst = ohalf + cc * 64;
                if (p.o_vec8) {
                    ptx::st_global_v8(dst, *reinterpret_cast<const uint32_t(*)[8]>(&w[0]));
                    ptx::st_global_v8(dst + 32, *reinterpret_cast<const uint32_t(*)[8]>(&w[8]));
                } else {
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        ptx::st_global_v4(dst + v4 * 16, w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2],
                                          w[4 * v4 + 3]);
                }
            }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_addr(bars, C::B_OFREE));
    }
    if (row_ok && hh == 0)
        p.lse[row_flat] = (le_all > 0.f) ? (m_ref + log2f(le_all)) * kLn2 : -INFINITY;
}

template <int D, bool kFP16>
__device__ void softmax_role(const Params &p, uint32_t bars, uint32_t tmem, float *xch, uint8_t *sO,
                             Ctl *ctl) {
    using C = Cfg<D>;
    constexpr int BN = C::BN;
    constexpr int NR = BN / 2;  // registers of one S tile per thread: 2 rows x BN/4 columns
    const int warp = (int)(threadIdx.x >> 5), t = (int)(threadIdx.x & 31);
    const int qw = warp & 3, hh = warp >> 2;
    const int tq = t & 3;
    const int rblk = 32 * qw + 16 * hh;   // first tile row (TMEM lane) of this warp's 16
    const int ra = rblk + (t >> 2);       // this thread's two rows in the 16-lane shapes
    const int rb = ra + 8;
    const uint32_t blk = tmem + ((uint32_t)rblk << 16);
    const uint32_t o_blk = blk + C::O_COL0;   // all O columns of the 16 rows (rescales)
    const int re = 32 * qw + t;               // row of the one-row-per-thread epilogue
    const uint32_t o_tmem = tmem + ((uint32_t)(32 * qw) << 16) + C::O_COL0 + (uint32_t)(hh * (D / 2));
    const float c = p.scale_log2;
    uint32_t t_cnt = 0;  // key tiles processed (S buffer = t % NSB; one P V each)
    uint32_t u_cnt = 0;  // units completed (one O-final phase each)

    for (int k = 0;; ++k) {
        const int u = unit_at(k, p);
        if (u >= p.n_units) break;
        const Unit un = decode_unit<D>(u, p);
        const int row_e = un.i0 + re;
        const bool row_ok = row_e < p.Sq;
        const size_t head = (size_t)(un.b * p.H + un.h) * (size_t)p.Sq;
        const size_t row_flat = head + (size_t)row_e;
        uint8_t *ohalf = reinterpret_cast<uint8_t *>(p.o) + row_flat * D * 2 + (size_t)(hh * D);
        if (!un.valid) {
            // No key visible to any row of this tile: guarded output.
            if (row_ok) {
#pragma unroll
                for (int cc = 0; cc < D / 16; ++cc) ptx::st_global_v4(ohalf + cc * 16, 0, 0, 0, 0);
                if (hh == 0) p.lse[row_flat] = -INFINITY;
            }
            continue;
        }
        // Visible keys of rows a and b: absolute key indices [lo, hi].
        const int row_a = un.i0 + ra, row_b = un.i0 + rb;
        const int hi_a = (p.mask_kind == kMaskNone) ? p.Sk - 1 : min(row_a, p.Sk - 1);
        const int hi_b = (p.mask_kind == kMaskNone) ? p.Sk - 1 : min(row_b, p.Sk - 1);
        const int lo_a = (p.mask_kind == kMaskWindow) ? row_a - p.window + 1 : 0;
        const int lo_b = (p.mask_kind == kMaskWindow) ? row_b - p.window + 1 : 0;

        // Per row: the max the accumulator and sums are referenced to (log2
        // units), and this thread's share of the divisor of O and of the fp32
        // sum of P (for the logsumexp).
        float m_a = -INFINITY, m_b = -INFINITY;
        float l_a = 0.f, l_b = 0.f, le_a = 0.f, le_b = 0.f;

        for (int j = un.lo; j < un.hi; ++j) {
            const int i = j - un.lo;  // step within the unit
            const uint32_t tt = t_cnt++;
            const int b = (int)(tt % (uint32_t)C::NSB);
            // (Under the stall test the CTA's first wait is on a barrier no one
            // arrives at: it runs out, and the kernel winds down with the
            // device status word set.)
            wait_bar(bar_addr(bars, (p.stall_test && tt == 0) ? C::B_NEVER : C::B_SFULL + b),
                     (tt / C::NSB) & 1u, ctl, 7);
            ptx::tc_fence_after();
            uint32_t sr[NR];
            ptx::tmem_ld_16x256b_x8<0>(blk + (uint32_t)(b * BN), sr);
            if constexpr (NR == 64) ptx::tmem_ld_16x256b_x8<32>(blk + (uint32_t)(b * BN) + 64, sr);
            ptx::tmem_wait_ld();
            ptx::reg_fence<NR>(sr);
            // The S buffer may now be overwritten with tile t+NSB.
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_addr(bars, C::B_SFREE + b));

            const int kc = j * BN;  // first key of the tile
            if (cols_need_mask<BN>(un.i0, kc, p)) quad_mask<NR>(sr, tq, lo_a - kc, hi_a - kc, lo_b - kc, hi_b - kc);

            // A unit's first tile sets the references from the row maxima.
            // Later tiles exponentiate against the current references without
            // looking for the max: a weight above 2^8 (the max grew by more
            // than the deferral bound) pushes its thread's partial sum above
            // 2^8, so when no thread of the warp exceeds the bound every weight
            // is valid as computed.  Otherwise the warp takes the row maxima,
            // and each row whose max grew by more than the bound moves its
            // reference, rescales and is exponentiated (and stored) again.
            // d = 64 (two P areas, tensor work per tile half that of d = 128):
            // the area is nearly always free, and P goes to tensor memory
            // before that test, whose vote then overlaps the store (the P V
            // product sees P only after the arrival at the end of the tile;
            // measured +4 %).  d = 128 (one P area) runs the test while P V of
            // tile t-1 may still hold the area; d = 256 measured slower with
            // the store first.
            constexpr bool kStoreFirst = (D == 64);
            const bool first = (i == 0);
            if (first) {
                float ma, mb;
                quad_row_max<NR>(sr, ma, mb);
                m_a = (ma == -INFINITY) ? -INFINITY : ma * c;
                m_b = (mb == -INFINITY) ? -INFINITY : mb * c;
            }
            uint32_t pk[NR / 2];
            float le_at, le_bt, lr_at, lr_bt;  // this tile's sums (this thread's columns)
            float alpha_a = 1.f, alpha_b = 1.f;
            bool rescale = false;
            const uint32_t pb = tt & 1u;
            const uint32_t p_col = blk + C::P_COL0 + pb * C::P_STRIDE;
#pragma unroll 1
            for (int pass = 0;; ++pass) {
                if (kStoreFirst && pass > 0) ptx::tmem_wait_st();  // the first P has left the registers
                le_at = le_bt = lr_at = lr_bt = 0.f;
                quad_exp<NR, kFP16, !kFP16 && !C::SUMCOL>(sr, c, (m_a == -INFINITY) ? 0.f : -m_a,
                                    (m_b == -INFINITY) ? 0.f : -m_b, pk, le_at, le_bt, lr_at, lr_bt);
                if constexpr (kStoreFirst) {
                    if (pass == 0) {
                        if (i >= 2)  // P area t & 1 was last read by P V of tile t-2
                            wait_bar(bar_addr(bars, C::B_OFULL + (int)pb), ((tt >> 1) - 1u) & 1u, ctl, 10);
                        ptx::tc_fence_after();
                    }
                    store_p<NR>(p_col, pk);
                }
                if (first || pass > 0) break;
                // No reference yet (every earlier key of the row hidden) counts
                // as exceeding the bound as soon as a key is visible.
                const bool over = !(le_at <= kRescaleBound) || !(le_bt <= kRescaleBound) ||
                                  (m_a == -INFINITY && le_at != 0.f) ||
                                  (m_b == -INFINITY && le_bt != 0.f);
                if (!__any_sync(0xffffffffu, over)) break;
                float ma, mb;
                quad_row_max<NR>(sr, ma, mb);
                const float na = fmaxf(m_a, (ma == -INFINITY) ? -INFINITY : ma * c);
                const float nb = fmaxf(m_b, (mb == -INFINITY) ? -INFINITY : mb * c);
                const bool up_a = na > m_a + kRescaleLog2, up_b = nb > m_b + kRescaleLog2;
                if (!__any_sync(0xffffffffu, up_a || up_b)) break;  // weights within the bound
                if (up_a) {
                    alpha_a = ptx::ex2_approx(m_a - na);  // 0 while m_a is -inf
                    m_a = na;
                }
                if (up_b) {
                    alpha_b = ptx::ex2_approx(m_b - nb);
                    m_b = nb;
                }
                rescale = true;
            }
            // O barrier b completes once for each tile t with t & 1 == b:
            // completion k of barrier t & 1 is P V of tile t with k = t >> 1.
            // Rescaling O needs every earlier P V finished: wait for P V of tile
            // t-1 (a commit covers all earlier MMAs of its issuer).  Rewriting P
            // needs P V of tile t-2 (two areas) or t-1 (one area).  The P V of
            // the previous unit are covered by its final barrier.  Each
            // barrier's next completion needs a P this thread has not written
            // yet, and the one before was waited for two tiles ago, so the
            // parity waits are unambiguous.
            if (rescale) {  // warp-uniform
                if (i > 0)
                    wait_bar(bar_addr(bars, C::B_OFULL + (int)((tt - 1u) & 1u)), ((tt - 1u) >> 1) & 1u,
                             ctl, 8);
                ptx::tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < D / 64; ++cc) {
                    uint32_t ov[32];
                    ptx::tmem_ld_16x256b_x8<0>(o_blk + cc * 64, ov);
                    ptx::tmem_wait_ld();
                    ptx::reg_fence<32>(ov);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        ov[e] = __float_as_uint(__uint_as_float(ov[e]) * ((e & 2) ? alpha_b : alpha_a));
                    ptx::tmem_st_16x256b_x8<0>(o_blk + cc * 64, ov);
                }
                if constexpr (C::SUMCOL && !kFP16) {  // the divisor column rescales with O
                    uint32_t sv[8];
                    ptx::tmem_ld_16x256b_x2<0>(o_blk + D, sv);
                    ptx::tmem_wait_ld();
                    ptx::reg_fence<8>(sv);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        sv[e] = __float_as_uint(__uint_as_float(sv[e]) * ((e & 2) ? alpha_b : alpha_a));
                    ptx::tmem_st_16x256b_x2<0>(o_blk + D, sv);
                }
            }
            l_a = alpha_a * l_a + lr_at;
            l_b = alpha_b * l_b + lr_bt;
            le_a = alpha_a * le_a + le_at;
            le_b = alpha_b * le_b + le_bt;
            if constexpr (!kStoreFirst) {
                if (i >= 1)  // one P area: P V of tile t-1 has read it
                    wait_bar(bar_addr(bars, C::B_OFULL + (int)((tt - 1u) & 1u)), ((tt - 1u) >> 1) & 1u, ctl,
                             10);
                ptx::tc_fence_after();
                store_p<NR>(p_col, pk);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_addr(bars, C::B_PFULL + (int)pb));
        }

        // Epilogue, out of line: it runs once per unit, and keeping it out of
        // the tile loop keeps the loop's code compact.
        softmax_epilogue<D, kFP16>(p, bars, ctl, xch, sO, o_tmem, u_cnt, un.i0, un.h, un.b, row_flat,
                                   row_ok, ohalf, m_a, m_b, l_a, l_b, le_a, le_b);
        ++u_cnt;
    }
    if constexpr (C::O_STAGE_BYTES > 0) {
        if (threadIdx.x == 0) ptx::bulk_wait_all();  // sO must outlive the stores
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
    uint8_t *sK = smem + C::Q_BYTES;
    uint8_t *sV = sK + C::KST * C::PIECE_BYTES;
    uint8_t *sO = sV + C::VST * C::V_SLOT_BYTES;  // O staging (d <= 128)
    uint64_t *bar_mem = reinterpret_cast<uint64_t *>(smem + C::SMEM_TILES);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bar_mem + C::NUM_BARS);
    Ctl *ctl = reinterpret_cast<Ctl *>(tmem_holder + 2);    // 8-byte aligned
    float *xch = reinterpret_cast<float *>(tmem_holder + 6);
    const uint32_t bars = ptx::smem_addr(bar_mem);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const uint32_t lane = ptx::lane_id();

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_addr(bars, C::B_QFULL), 1);
        ptx::mbar_init(bar_addr(bars, C::B_QEMPTY), 1);
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
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_addr(bars, C::B_PFULL + b), C::NUM_SOFTMAX);
            ptx::mbar_init(bar_addr(bars, C::B_OFULL + b), 1);
        }
        ptx::mbar_init(bar_addr(bars, C::B_OFINAL), 1);
        ptx::mbar_init(bar_addr(bars, C::B_OFREE), C::NUM_SOFTMAX);
        ptx::mbar_init(bar_addr(bars, C::B_DRAIN), 1);
        ptx::mbar_init(bar_addr(bars, C::B_DRAIN + 1), 1);
        ptx::mbar_init(bar_addr(bars, C::B_NEVER), 1);
        ctl->abort = 0;
        ctl->limit_ns = p.wait_limit_ns;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == C::S_WARP) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == C::TMA_WARP && lane == 0) {
        ptx::prefetch_tensormap(&p.tm_q);
        ptx::prefetch_tensormap(&p.tm_k);
        ptx::prefetch_tensormap(&p.tm_v);
        if (C::O_STAGE_BYTES > 0) ptx::prefetch_tensormap(&p.tm_o);
    }
    if constexpr (C::SUMCOL && !kFP16) {
        // The ones box of every V slot, in the tile's 128-byte-swizzled layout
        // (key row r, 16-byte chunk c stored at chunk c ^ (r & 7)): column 0
        // (element 0 of logical chunk 0) is 1.0, the rest 0.
        constexpr int kChunks = C::KV_CHUNK / 16;  // 16-byte chunks of one box
        for (int idx = (int)threadIdx.x; idx < C::VST * kChunks; idx += C::NUM_THREADS) {
            const int slot = idx / kChunks, rem = idx - slot * kChunks;
            const int r = rem >> 3, phys = rem & 7;
            const uint32_t one = (phys == (r & 7)) ? 0x3F80u : 0u;  // bf16 1.0 in the low half
            ptx::st_shared_v4(ptx::smem_addr(sV + slot * C::V_SLOT_BYTES + C::CHUNKS * C::KV_CHUNK) + rem * 16, one,
                              0u, 0u, 0u);
        }
        ptx::fence_proxy_async_smem();  // the tensor core reads the boxes through the async proxy
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp < C::NUM_SOFTMAX / 32) {
        softmax_role<D, kFP16>(p, bars, tmem, xch, sO, ctl);
    } else if (warp == C::S_WARP) {
        mma_s_role<D, kFP16>(p, sQ, sK, bars, tmem, ctl);
    } else if (warp == C::PV_WARP) {
        mma_pv_role<D, kFP16>(p, sV, bars, tmem, ctl);
    } else if (warp == C::TMA_WARP) {
        tma_qk_role<D>(p, sQ, sK, bars, ctl);
    } else {
        tma_v_role<D>(p, sV, bars, ctl);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::S_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace fa
