// fa_bwd_kernel.cuh -- attention backward for sm_103a (GB300): dQ, dK, dV of
// O = softmax(scale * Q K^T) V from Q, K, V, O, the forward's per-row lse and
// dO, by recomputation ("FlashAttention: Why Tiling Attention Makes
// Transformers Fast Without Changing the Result", section "The backward pass:
// recompute instead of storing"): every score tile is rebuilt on chip from Q
// and K, its probabilities from the stored row statistic,
//   P_ij  = exp(scale q_i . k_j - lse_i)          (0 for hidden pairs)
//   dV_j  = sum_i P_ij dO_i
//   dP_ij = dO_i . v_j
//   dS_ij = P_ij (dP_ij - delta_i)                 (softmax Jacobian)
//   dQ_i  = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i,
// and no S x S matrix reaches device memory.  delta_i is the Jacobian's row
// term sum_j P_ij dP_ij, taken as dO_i . O_i: both equal sum_j P_ij dO_i . v_j
// because O_i = sum_j P_ij v_j, and the second needs one pass over a row of O
// instead of a row of P.
//
// Three launches on the caller's stream:
//   1. fa_bwd_prep_kernel: per query row, delta_i and lse_i * log2(e) (+inf
//      for a row that sees no key and for padding rows, so that their P is 0)
//      into a caller-provided workspace, rows padded per head to a multiple of
//      128;
//   2. fa_bwd_dkdv_kernel: one CTA per (batch, K/V head, 128-key tile).  K and
//      V stay in shared memory; 64-row tiles of Q and dO of every query head
//      that reads this K/V head stream through a ring.  Per step one MMA warp
//      computes S^T = K Q^T and dP^T = V dO^T into one of two score buffers
//      in tensor memory (lane = key), the compute warps turn them into P^T
//      and dS^T (16-bit, written over the step's own S^T and dP^T), and a
//      second MMA warp accumulates dV += P^T dO and dK += dS^T Q in tensor
//      memory (P^T and dS^T as the A operand from tensor memory), while the
//      next step's scores form in the other buffer;
//   3. fa_bwd_dq_kernel: one CTA per (batch, head, 128-row query tile).  Q and
//      dO stay in shared memory, K/V tiles stream through two rings; per step
//      one MMA warp computes S = Q K^T and dP = dO V^T (lane = query row), the
//      compute warps write dS to tensor memory, and a second MMA warp
//      accumulates dQ += dS K with K read as the MN-major B operand.
// Two kernels instead of one with atomic dQ updates keep the result
// deterministic and need no fp32 dQ buffer; the price is that S and dP are
// formed twice (7 tile products per (query, key) tile instead of 5).
#pragma once

#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "fa_fwd_kernel.cuh"

namespace fa {

struct BwdParams {
    CUtensorMap tm_q;   // [B, H, Sq, d] 16-bit, box {64, query rows per tile, 1, 1}
    CUtensorMap tm_do;  // like tm_q, over dO
    CUtensorMap tm_k;   // [B, Hkv, Sk, d], box {64, keys per tile, 1, 1}
    CUtensorMap tm_v;   // like tm_k, over V
    void *dq;           // [B, H, Sq, d] 16-bit
    void *dk;           // [B, Hkv, Sk, d] 16-bit
    void *dv;           // [B, Hkv, Sk, d] 16-bit
    const float *l2;    // [B*H, Sq_pad]: lse * log2(e); +inf for keyless and padding rows
    const float *delta; // [B*H, Sq_pad]: dO_i . O_i; 0 for padding rows
    int B, H, Hkv, kv_group, Sq, Sk, Sq_pad;
    int mask_kind, window;
    float scale_log2;  // scale * log2(e), kept positive (as in the forward)
    float scale;       // the multiplier of dQ and dK
    int n_units;       // CTAs of the launch
    int n_tiles;       // dK/dV: key tiles per K/V head; dQ: query tiles per head
    uint64_t wait_limit_ns;
    int stall_test;    // test only: the compute warps' first wait is on a barrier nothing completes
};

constexpr int kBwdPadRows = 128;  // workspace rows per head are padded to this multiple

// ---------------------------------------------------------------- prep

template <bool kFP16>
__device__ __forceinline__ float2 widen2(uint32_t w) {
    if constexpr (kFP16) {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    } else {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }
}

// One row per D/8 threads (16 bytes of O and dO each).
template <int D, bool kFP16>
__global__ void __launch_bounds__(256)
    fa_bwd_prep_kernel(const uint16_t *__restrict__ o, const uint16_t *__restrict__ dout,
                       const float *__restrict__ lse, float *__restrict__ l2,
                       float *__restrict__ delta, long long BH, int Sq, int Sq_pad) {
    constexpr int TPR = D / 8;
    constexpr int RPB = 256 / TPR;
    const int sub = (int)threadIdx.x % TPR;
    const long long r = (long long)blockIdx.x * RPB + (long long)(threadIdx.x / TPR);
    const long long rows = BH * (long long)Sq_pad;
    const long long bh = r / Sq_pad;
    const int i = (int)(r - bh * Sq_pad);
    const bool real = r < rows && i < Sq;
    float acc = 0.f;
    if (real) {
        const size_t off = ((size_t)bh * (size_t)Sq + (size_t)i) * D + (size_t)sub * 8;
        const uint4 a = *reinterpret_cast<const uint4 *>(o + off);
        const uint4 g = *reinterpret_cast<const uint4 *>(dout + off);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = widen2<kFP16>(aw[e]), y = widen2<kFP16>(gw[e]);
            acc = fmaf(x.x, y.x, acc);
            acc = fmaf(x.y, y.y, acc);
        }
    }
#pragma unroll
    for (int m = TPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (sub == 0 && r < rows) {
        float L = INFINITY;
        if (real) {
            const float ls = lse[(size_t)bh * (size_t)Sq + (size_t)i];
            L = (ls == -INFINITY) ? INFINITY : ls * 1.4426950408889634f;
        }
        l2[r] = L;
        delta[r] = real ? acc : 0.f;
    }
}

// ---------------------------------------------------------------- shared helpers

template <bool kFP16>
__device__ __forceinline__ uint32_t pack2b(float lo, float hi) {
    return kFP16 ? ptx::pack_f16x2(lo, hi) : ptx::pack_bf16x2(lo, hi);
}

// Stores 32 fp32 values (times `mul`) of one row as 16-bit to dst (16-byte aligned).
template <bool kFP16>
__device__ __forceinline__ void store_row32(void *dst, const uint32_t (&r)[32], float mul) {
    uint32_t w[16];
#pragma unroll
    for (int c = 0; c < 16; ++c)
        w[c] = pack2b<kFP16>(__uint_as_float(r[2 * c]) * mul, __uint_as_float(r[2 * c + 1]) * mul);
    uint8_t *d8 = static_cast<uint8_t *>(dst);
#pragma unroll
    for (int c = 0; c < 4; ++c)
        ptx::st_global_v4(d8 + 16 * c, w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

__device__ __forceinline__ void store_zero_row(void *dst, int bytes) {
    uint8_t *d8 = static_cast<uint8_t *>(dst);
    for (int c = 0; c < bytes; c += 16) ptx::st_global_v4(d8 + c, 0u, 0u, 0u, 0u);
}

// Warp-uniform bounded waits: every lane gets the answer of the whole warp,
// so a timeout seen by one lane never splits the warp in front of a
// warp-collective tcgen05 load or store, or of a __syncwarp.  (Callers keep
// their `ok` flags warp-uniform too.)
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, Ctl *ctl, int site) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, ctl, site));
}

__device__ __forceinline__ bool wait_warp_backoff(uint32_t bar, uint32_t parity, Ctl *ctl, int site) {
    return __all_sync(0xffffffffu, wait_bar_backoff(bar, parity, ctl, site));
}

// 16-column steps of a 128-byte-swizzled K-major operand made of 64-column
// boxes `box` bytes apart: 32 bytes inside a box, then the next box.
__device__ __forceinline__ uint32_t kmajor_step(int kk, int box) {
    return (uint32_t)(((kk >> 2) * box + (kk & 3) * 32) >> 4);
}

// ---------------------------------------------------------------- dK / dV

template <int D>
struct BwdKVCfg {
    static constexpr int BM = 64;    // query rows per step (N of S^T, K of dV / dK)
    static constexpr int BN = 128;   // keys per CTA (M of every MMA = TMEM lanes)
    // d = 256: the dK and dV accumulators of a 128-key tile would need all 512
    // tensor-memory columns, so two CTAs share the tile by role: role 0
    // accumulates dV (it forms S^T and P^T only), role 1 dK (S^T, dP^T and
    // dS^T), each over the whole d.  dP^T is thus formed once per tile, and
    // the role-0 CTAs, which carry about 60 % of the role-1 work, let the
    // block scheduler balance the rest.  K, V, Q and dO leave room for one
    // Q/dO stage plus 32 KB: the dK role, whose dO is done once dP^T is
    // formed, keeps dO on a ring of its own (one buffer) and Q with the
    // statistics on a ring of two (the second in those 32 KB); the dV role
    // loads no V and takes a second Q/dO stage in its place.  A stage is free
    // only after dV and dK of its step, a step after the compute warps have
    // seen it, so the ring runs about two stages ahead of the score products;
    // d = 128 fits four stages, d = 64 six.
    static constexpr int DA = D;                    // accumulator columns per CTA
    static constexpr bool ROLES = (D > 128);        // one of dV, dK per CTA
    static constexpr int NH = ROLES ? 2 : 1;        // CTAs per key tile
    static constexpr int ST = (D > 128) ? 1 : (D == 128) ? 4 : 6;  // stages of the (Q, dO, statistics) ring
    static constexpr int ST_DV = ROLES ? 2 : ST;  // stages of the dV role; the dK role's Q ring
    static constexpr int STM = ST_DV > ST ? ST_DV : ST;  // barriers and statistics slots
    static constexpr int KV_BOX = BN * 128;
    static constexpr int Q_BOX = BM * 128;
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int STAT_BYTES = 2 * BM * 4;  // l2 of the step's rows, then delta
    // Compute warps: one warpgroup at d >= 128, two at d = 64, where they
    // take alternate steps (warpgroup g works on the steps t with
    // t & 1 == g).  Warp w owns key rows 32 (w & 3) .. + 31 (its TMEM
    // lanes), one per thread, and all 64 query columns of its steps (two
    // warpgroups: in two halves of 32, for registers).  At d = 64 the tensor
    // core's work per step halves and one warp per sub-partition leaves the
    // latency-bound exponent and packing chain exposed; at d = 128 a second
    // warpgroup measured slower (the MMA issuers then share their
    // sub-partitions with two compute warps).  The next warps issue S^T and
    // dP^T, dV and dK, and the copies.
    static constexpr int NUM_COMPUTE = (D == 64) ? 256 : 128;
    static constexpr int WG = NUM_COMPUTE / 128;   // warpgroups alternating steps
    static constexpr int COLS = BM;                // query columns per compute thread and step
    static constexpr int MMA_WARP = NUM_COMPUTE / 32;  // issues S^T and dP^T
    static constexpr int MMA_G_WARP = MMA_WARP + 1;    // issues dV and dK
    static constexpr int TMA_WARP = MMA_WARP + 2;
    static constexpr int NUM_THREADS = NUM_COMPUTE + 96;
    // Tensor memory: dV and dK accumulators, then two score buffers; step t
    // uses buffer t & 1: S^T and dP^T (fp32, 64 columns each) at S_COL and
    // DP_COL + BUF * (t & 1).  P^T and dS^T of the step (16-bit pairs, 32
    // columns each) are written over the first halves of its own S^T and
    // dP^T, which the compute warps have read by then, so the score products
    // of step t+1 run on the tensor core while the compute warps work on
    // step t, and a buffer is free again once dV and dK of its step are done.
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t DV_COL = 0;
    static constexpr uint32_t DK_COL = ROLES ? 0 : 128;  // roles: the one accumulator at 0
    static constexpr uint32_t S_COL = 256;
    static constexpr uint32_t DP_COL = 320;
    static constexpr uint32_t BUF = 128;
    static constexpr int B_KVFULL = 0;
    static constexpr int B_QFULL = 1;               // [STM]
    static constexpr int B_QEMPTY = B_QFULL + STM;  // [STM]
    // One compute warpgroup: S^T of a buffer is announced on its own, so the
    // exponentials start while dP^T is still being formed.
    static constexpr bool SPLIT = (WG == 1);
    static constexpr int B_SFULL = B_QEMPTY + STM;  // [2]: S^T (and dP^T, unless SPLIT) of buffer b formed
    static constexpr int B_DPFULL = B_SFULL + 2;   // [2]: SPLIT: dP^T of buffer b formed
    static constexpr int B_PFULL = B_DPFULL + 2;   // [2]: P^T, dS^T of buffer b written
    static constexpr int B_PFREE = B_PFULL + 2;    // [2]: dV, dK of buffer b done
    static constexpr int B_DOFULL = B_PFREE + 2;   // ROLES, dK role: the dO buffer loaded
    static constexpr int B_DOEMPTY = B_DOFULL + 1; // ROLES, dK role: dP^T done with it
    static constexpr int B_DONE = B_DOEMPTY + 1;
    static constexpr int B_DRAIN = B_DONE + 1;  // [2]: each issuer's MMAs finished
    static constexpr int B_NEVER = B_DRAIN + 2;  // no arrivals (the stall test's wait)
    static constexpr int NUM_BARS = B_NEVER + 1;
    static constexpr int X_BYTES = ROLES ? Q_BYTES : 0;  // the dK role's second Q buffer
    static constexpr int SMEM_TILES = 2 * KV_BYTES + ST * 2 * Q_BYTES + X_BYTES + STM * STAT_BYTES;
    static_assert(ST_DV == ST || (ST_DV == ST + 1 && 2 * Q_BYTES <= KV_BYTES), "the dV role's extra stage fits in V's place");
    static_assert(!ROLES || ST == 1, "the dK role's dO ring holds one buffer, at stage 0's dO area");
    static constexpr int SMEM_BYTES = 1024 + SMEM_TILES + NUM_BARS * 8 + 32;
    static_assert(DK_COL + DA <= S_COL && DV_COL + DA <= S_COL && (ROLES || DV_COL + DA <= DK_COL) &&
                      DP_COL + BUF + BM <= TMEM_COLS && S_COL + BM <= DP_COL,
                  "tensor memory overflow");
    static_assert(SMEM_BYTES <= 232448, "shared memory overflow");
};

// The rows of the K/V tile of one CTA and the query tiles that see them.
struct KVUnit {
    int role;              // d = 256: 0 = this CTA accumulates dV, 1 = dK (else 0: both)
    int b, kvh, j0, jend;  // keys [j0, jend)
    int it_lo, n_i;        // query tiles it_lo .. it_lo + n_i of every query head of the group
    int steps;             // kv_group * n_i
};

template <int D>
__device__ __forceinline__ KVUnit decode_kv_unit(const BwdParams &p) {
    KVUnit u;
    constexpr int NH = BwdKVCfg<D>::NH;
    const int n_bk = p.B * p.Hkv;
    u.role = (int)blockIdx.x % NH;
    const int id = (int)blockIdx.x / NH;
    const int jt = id / n_bk;  // key tile: all heads' first tiles first (longest)
    const int bk = id - jt * n_bk;
    u.b = bk / p.Hkv;
    u.kvh = bk - u.b * p.Hkv;
    u.j0 = jt * 128;
    u.jend = min(u.j0 + 128, p.Sk);
    // query rows that see one of these keys
    const int row_lo = (p.mask_kind == kMaskNone) ? 0 : u.j0;
    long long row_hi = p.Sq;
    if (p.mask_kind == kMaskWindow) row_hi = min(row_hi, (long long)u.jend - 1 + (long long)p.window);
    if (row_lo >= row_hi) {
        u.it_lo = 0;
        u.n_i = 0;
    } else {
        u.it_lo = row_lo / 64;
        u.n_i = (int)((row_hi + 63) / 64) - u.it_lo;
    }
    u.steps = p.kv_group * u.n_i;
    return u;
}

// Q (and statistics) stages of this CTA, whether its dO has a ring of its
// own (the dK role: one buffer), and the Q and dO buffers of stage `slot`:
// stages below ST have their own area; the dV role's extra stage uses V's,
// the dK role's extra Q buffer the area after the dO stages (sX).
template <int D>
__device__ __forceinline__ int kv_stages(const KVUnit &un) {
    using C = BwdKVCfg<D>;
    return C::ROLES ? C::ST_DV : C::ST;
}
template <int D>
__device__ __forceinline__ bool own_do_ring(const KVUnit &un) {
    return BwdKVCfg<D>::ROLES && un.role == 1;
}
template <int D>
__device__ __forceinline__ uint8_t *q_stage(uint8_t *sQ, uint8_t *sV, uint8_t *sX, const KVUnit &un, int slot) {
    using C = BwdKVCfg<D>;
    return slot < C::ST ? sQ + slot * C::Q_BYTES : (own_do_ring<D>(un) ? sX : sV);
}
template <int D>
__device__ __forceinline__ uint8_t *do_stage(uint8_t *sDO, uint8_t *sV, const KVUnit &un, int slot) {
    using C = BwdKVCfg<D>;
    return (slot < C::ST || own_do_ring<D>(un)) ? sDO + (own_do_ring<D>(un) ? 0 : slot * C::Q_BYTES)
                                                 : sV + C::Q_BYTES;
}

template <int D>
__device__ void bwd_kv_tma_role(const BwdParams &p, const KVUnit &un, uint8_t *sK, uint8_t *sV,
                                uint8_t *sQ, uint8_t *sDO, uint8_t *sX, uint8_t *sStat, uint32_t bars,
                                Ctl *ctl) {
    using C = BwdKVCfg<D>;
    const bool leader = ptx::lane_id() == 0;
    const uint64_t pol_last = ptx::policy_evict_last();
    if (un.steps == 0) return;  // no query row sees these keys: nothing to load
    const bool need_v = !(C::ROLES && un.role == 0);  // the dV role forms no dP^T
    if (leader) {
        const uint32_t fb = bar_addr(bars, C::B_KVFULL);
        ptx::mbar_arrive_expect_tx(fb, (need_v ? 2 : 1) * C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            ptx::tma_load_4d(ptx::smem_addr(sK) + c * C::KV_BOX, &p.tm_k, fb, c * 64, un.j0, un.kvh, un.b,
                             pol_last);
            if (need_v)
                ptx::tma_load_4d(ptx::smem_addr(sV) + c * C::KV_BOX, &p.tm_v, fb, c * 64, un.j0, un.kvh, un.b,
                                 pol_last);
        }
    }
    int issued = 0, do_issued = 0;
    bool ok = true;
    const int nst = kv_stages<D>(un);
    const bool sep = own_do_ring<D>(un);  // dO on a ring of its own (one buffer)
    for (int s = 0; s < un.steps; ++s) {
        const int slot = s % nst;
        if (!wait_warp_backoff(bar_addr(bars, C::B_QEMPTY + slot), ((s / nst) & 1) ^ 1, ctl, 21)) {
            ok = false;
            break;
        }
        const int hq = un.kvh * p.kv_group + s / un.n_i;
        const int i0 = (un.it_lo + s % un.n_i) * C::BM;
        if (leader) {
            const uint32_t fb = bar_addr(bars, C::B_QFULL + slot);
            ptx::mbar_arrive_expect_tx(fb, (sep ? 1 : 2) * C::Q_BYTES + C::STAT_BYTES);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                ptx::tma_load_4d(ptx::smem_addr(q_stage<D>(sQ, sV, sX, un, slot)) + c * C::Q_BOX, &p.tm_q, fb,
                                 c * 64, i0, hq, un.b, pol_last);
                if (!sep)
                    ptx::tma_load_4d(ptx::smem_addr(do_stage<D>(sDO, sV, un, slot)) + c * C::Q_BOX, &p.tm_do,
                                     fb, c * 64, i0, hq, un.b, pol_last);
            }
            const size_t row0 = ((size_t)un.b * p.H + hq) * (size_t)p.Sq_pad + (size_t)i0;
            const uint32_t st = ptx::smem_addr(sStat + slot * C::STAT_BYTES);
            ptx::bulk_load(st, p.l2 + row0, C::BM * 4, fb);
            ptx::bulk_load(st + C::BM * 4, p.delta + row0, C::BM * 4, fb);
        }
        __syncwarp();
        ++issued;
        if (sep) {
            if (!wait_warp_backoff(bar_addr(bars, C::B_DOEMPTY), (s & 1) ^ 1, ctl, 74)) {
                ok = false;
                break;
            }
            if (leader) {
                const uint32_t fd = bar_addr(bars, C::B_DOFULL);
                ptx::mbar_arrive_expect_tx(fd, C::Q_BYTES);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_4d(ptx::smem_addr(sDO) + c * C::Q_BOX, &p.tm_do, fd, c * 64, i0, hq, un.b,
                                     pol_last);
            }
            __syncwarp();
            ++do_issued;
        }
    }
    // Let every copy already issued land before the CTA can exit.
    wait_bar_drain(bar_addr(bars, C::B_KVFULL), 0);
    if (!ok) {
        for (int s = issued - nst > 0 ? issued - nst : 0; s < issued; ++s)
            wait_bar_drain(bar_addr(bars, C::B_QFULL + s % nst), (s / nst) & 1);
        if (do_issued) wait_bar_drain(bar_addr(bars, C::B_DOFULL), (do_issued - 1) & 1);
    }
}

// The two MMA issuers of the dK/dV kernel.  A tcgen05.mma blocks its issuing
// thread while the tensor pipe's queue is full (an N = 64 score product with
// both operands in shared memory takes about 48 cycles, bound by the
// shared-memory reads), so the score products (S^T, dP^T) and the gradient
// products (dV, dK) go out from two warps and neither waits behind the
// other's queue.  A Q/dO stage is free once both have read it (QEMPTY takes
// one commit from each).
template <int D, bool kFP16>
__device__ void bwd_kv_mma_s_role(const BwdParams &p, const KVUnit &un, uint8_t *sK, uint8_t *sV,
                                  uint8_t *sQ, uint8_t *sDO, uint8_t *sX, uint32_t bars, uint32_t tmem,
                                  Ctl *ctl) {
    using C = BwdKVCfg<D>;
    constexpr uint32_t kIdescS = make_idesc(C::BN, C::BM, kFP16, false);  // M = keys, N = query rows
    const bool leader = ptx::lane_id() == 0;
    const uint64_t dk_desc = smem_desc(ptx::smem_addr(sK), 16);
    const uint64_t dv_desc = smem_desc(ptx::smem_addr(sV), 16);
    bool ok = un.steps == 0 || wait_warp(bar_addr(bars, C::B_KVFULL), 0, ctl, 22);
    const int nst = kv_stages<D>(un);
    for (int t = 0; ok && t < un.steps; ++t) {
        const int slot = t % nst;
        if (!wait_warp(bar_addr(bars, C::B_QFULL + slot), (t / nst) & 1, ctl, 23)) {
            ok = false;
            break;
        }
        // buffer t & 1 is free once dV and dK of step t-2 are done
        const int b = t & 1;
        if (t >= 2 && !wait_warp(bar_addr(bars, C::B_PFREE + b), ((t - 2) >> 1) & 1, ctl, 24)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        const bool sep = own_do_ring<D>(un);
        const uint64_t qd = smem_desc(ptx::smem_addr(q_stage<D>(sQ, sV, sX, un, slot)), 16);
        const uint64_t od = smem_desc(ptx::smem_addr(do_stage<D>(sDO, sV, un, slot)), 16);
        const uint32_t boff = (uint32_t)b * C::BUF;
        if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::mma_ss(tmem + C::S_COL + boff, dk_desc + kmajor_step(kk, C::KV_BOX),
                            qd + kmajor_step(kk, C::Q_BOX), kIdescS, kk > 0 ? 1u : 0u);
            if constexpr (C::SPLIT) ptx::mma_commit(bar_addr(bars, C::B_SFULL + b));
            if (sep) ptx::mma_commit(bar_addr(bars, C::B_QEMPTY + slot));  // Q's last read here
        }
        if (!(C::ROLES && un.role == 0)) {
            if (sep) {  // dO on its own ring (one buffer)
                __syncwarp();
                if (!wait_warp(bar_addr(bars, C::B_DOFULL), t & 1, ctl, 73)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
            }
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + C::DP_COL + boff, dv_desc + kmajor_step(kk, C::KV_BOX),
                                od + kmajor_step(kk, C::Q_BOX), kIdescS, kk > 0 ? 1u : 0u);
                ptx::mma_commit(bar_addr(bars, C::SPLIT ? C::B_DPFULL + b : C::B_SFULL + b));
                if (sep) ptx::mma_commit(bar_addr(bars, C::B_DOEMPTY));
            }
        }
        if (leader && !sep) ptx::mma_commit(bar_addr(bars, C::B_QEMPTY + slot));
        __syncwarp();
    }
    if (leader) ptx::mma_commit(bar_addr(bars, C::B_DRAIN));
    __syncwarp();
    wait_bar_drain(bar_addr(bars, C::B_DRAIN), 0);
}

template <int D, bool kFP16>
__device__ void bwd_kv_mma_g_role(const BwdParams &p, const KVUnit &un, uint8_t *sQ, uint8_t *sDO,
                                  uint8_t *sV, uint8_t *sX, uint32_t bars, uint32_t tmem, Ctl *ctl) {
    using C = BwdKVCfg<D>;
    constexpr uint32_t kIdescG = make_idesc(C::BN, C::DA, kFP16, true);  // dV, dK: N = DA, B MN-major
    const bool leader = ptx::lane_id() == 0;
    bool ok = true;
    const int nst = kv_stages<D>(un);
    for (int t = 0; ok && t < un.steps; ++t) {
        const int slot = t % nst;
        const int b = t & 1;
        if (!wait_warp(bar_addr(bars, C::B_QFULL + slot), (t / nst) & 1, ctl, 30) ||
            !wait_warp(bar_addr(bars, C::B_PFULL + b), (t >> 1) & 1, ctl, 25)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        if (leader) {
            // dO and Q as MN-major B operands: K = query rows (16 = two 8-row
            // groups, 2048 bytes), N = d in 64-column boxes Q_BOX apart.
            const uint64_t om = smem_desc(ptx::smem_addr(do_stage<D>(sDO, sV, un, slot)), C::Q_BOX);
            const uint64_t qm = smem_desc(ptx::smem_addr(q_stage<D>(sQ, sV, sX, un, slot)), C::Q_BOX);
            const uint32_t boff = (uint32_t)b * C::BUF;
            if (!(C::ROLES && un.role == 1)) {
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    ptx::mma_ts(tmem + C::DV_COL, tmem + C::S_COL + boff + kk * 8,
                                om + (uint32_t)((kk * 2048) >> 4), kIdescG, (t > 0 || kk > 0) ? 1u : 0u);
            }
            if (!(C::ROLES && un.role == 0)) {
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    ptx::mma_ts(tmem + C::DK_COL, tmem + C::DP_COL + boff + kk * 8,
                                qm + (uint32_t)((kk * 2048) >> 4), kIdescG, (t > 0 || kk > 0) ? 1u : 0u);
            }
            ptx::mma_commit(bar_addr(bars, C::B_PFREE + b));
            ptx::mma_commit(bar_addr(bars, C::B_QEMPTY + slot));
            if (t + 1 == un.steps) ptx::mma_commit(bar_addr(bars, C::B_DONE));
        }
        __syncwarp();
    }
    if (leader) ptx::mma_commit(bar_addr(bars, C::B_DRAIN + 1));
    __syncwarp();
    wait_bar_drain(bar_addr(bars, C::B_DRAIN + 1), 0);
}

// P^T = exp2(S^T c - lse2) (masked) and dS^T = P^T (dP^T - delta) of the
// query columns col0 .. col0 + NC of one step, for this thread's key row j:
// s and dp hold the row's S^T and dP^T there, L4 and D4 the step's row
// statistics; pw and dsw get the 16-bit pairs.
template <int NC, bool kFP16>
__device__ __forceinline__ void bwd_kv_p_ds(const uint32_t (&s)[NC], const uint32_t (&dp)[NC],
                                            const float4 *L4, const float4 *D4, int col0, int lo, int hi,
                                            bool masked, float c, uint32_t (&pw)[NC / 2],
                                            uint32_t (&dsw)[NC / 2]) {
    const uint64_t c2 = ptx::f32x2(c, c);
    const uint64_t z2 = ptx::f32x2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < NC / 4; ++q) {
        const int cq = col0 + 4 * q;  // query column of element 0
        const float4 l = L4[cq / 4], dl = D4[cq / 4];
        float x0, x1, x2, x3, g0, g1, g2, g3;
        ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(s[4 * q]), __uint_as_float(s[4 * q + 1])),
                                         c2, ptx::f32x2(-l.x, -l.y)), x0, x1);
        ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(s[4 * q + 2]), __uint_as_float(s[4 * q + 3])),
                                         c2, ptx::f32x2(-l.z, -l.w)), x2, x3);
        float pv[4] = {ptx::ex2_approx(x0), ptx::ex2_approx(x1), ptx::ex2_approx(x2), ptx::ex2_approx(x3)};
        if (masked) {
#pragma unroll
            for (int e = 0; e < 4; ++e) pv[e] = (cq + e >= lo && cq + e < hi) ? pv[e] : 0.f;
        }
        ptx::unpack_f32x2(ptx::add_f32x2(ptx::f32x2(__uint_as_float(dp[4 * q]), __uint_as_float(dp[4 * q + 1])),
                                         ptx::f32x2(-dl.x, -dl.y)), g0, g1);
        ptx::unpack_f32x2(ptx::add_f32x2(ptx::f32x2(__uint_as_float(dp[4 * q + 2]), __uint_as_float(dp[4 * q + 3])),
                                         ptx::f32x2(-dl.z, -dl.w)), g2, g3);
        float d0, d1, d2, d3;
        ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(pv[0], pv[1]), ptx::f32x2(g0, g1), z2), d0, d1);
        ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(pv[2], pv[3]), ptx::f32x2(g2, g3), z2), d2, d3);
        pw[2 * q] = pack2b<kFP16>(pv[0], pv[1]);
        pw[2 * q + 1] = pack2b<kFP16>(pv[2], pv[3]);
        dsw[2 * q] = pack2b<kFP16>(d0, d1);
        dsw[2 * q + 1] = pack2b<kFP16>(d2, d3);
    }
}

// The two halves of bwd_kv_p_ds for a split step: P^T (fp32 into s, and
// packed into pw) from S^T alone, then dS^T from the fp32 P^T and dP^T.
template <int NC, bool kFP16>
__device__ __forceinline__ void bwd_kv_p(uint32_t (&s)[NC], const float4 *L4, int lo, int hi, bool masked,
                                         float c, uint32_t (&pw)[NC / 2]) {
    const uint64_t c2 = ptx::f32x2(c, c);
#pragma unroll
    for (int q = 0; q < NC / 4; ++q) {
        const float4 l = L4[q];
        float x0, x1, x2, x3;
        ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(s[4 * q]), __uint_as_float(s[4 * q + 1])),
                                         c2, ptx::f32x2(-l.x, -l.y)), x0, x1);
        ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(s[4 * q + 2]), __uint_as_float(s[4 * q + 3])),
                                         c2, ptx::f32x2(-l.z, -l.w)), x2, x3);
        float pv[4] = {ptx::ex2_approx(x0), ptx::ex2_approx(x1), ptx::ex2_approx(x2), ptx::ex2_approx(x3)};
        if (masked) {
#pragma unroll
            for (int e = 0; e < 4; ++e) pv[e] = (4 * q + e >= lo && 4 * q + e < hi) ? pv[e] : 0.f;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) s[4 * q + e] = __float_as_uint(pv[e]);
        pw[2 * q] = pack2b<kFP16>(pv[0], pv[1]);
        pw[2 * q + 1] = pack2b<kFP16>(pv[2], pv[3]);
    }
}

template <int NC, bool kFP16>
__device__ __forceinline__ void bwd_kv_ds(const uint32_t (&pf)[NC], const uint32_t (&dp)[NC], const float4 *D4,
                                          uint32_t (&dsw)[NC / 2]) {
    const uint64_t z2 = ptx::f32x2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < NC / 4; ++q) {
        const float4 dl = D4[q];
        float g0, g1, g2, g3, d0, d1, d2, d3;
        ptx::unpack_f32x2(ptx::add_f32x2(ptx::f32x2(__uint_as_float(dp[4 * q]), __uint_as_float(dp[4 * q + 1])),
                                         ptx::f32x2(-dl.x, -dl.y)), g0, g1);
        ptx::unpack_f32x2(ptx::add_f32x2(ptx::f32x2(__uint_as_float(dp[4 * q + 2]), __uint_as_float(dp[4 * q + 3])),
                                         ptx::f32x2(-dl.z, -dl.w)), g2, g3);
        ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(pf[4 * q]), __uint_as_float(pf[4 * q + 1])),
                                         ptx::f32x2(g0, g1), z2), d0, d1);
        ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(pf[4 * q + 2]), __uint_as_float(pf[4 * q + 3])),
                                         ptx::f32x2(g2, g3), z2), d2, d3);
        dsw[2 * q] = pack2b<kFP16>(d0, d1);
        dsw[2 * q + 1] = pack2b<kFP16>(d2, d3);
    }
}

template <int D, bool kFP16>
__device__ void bwd_kv_compute_role(const BwdParams &p, const KVUnit &un, const uint8_t *sStat,
                                    uint32_t bars, uint32_t tmem, Ctl *ctl) {
    using C = BwdKVCfg<D>;
    constexpr int NC = C::COLS;
    constexpr int HC = NC / C::WG;  // columns per pass: P^T and dS^T of a pass overwrite only
                                    // columns of S^T and dP^T that this thread has read
    const int warp = (int)threadIdx.x >> 5;
    const int r = 32 * (warp & 3) + ((int)threadIdx.x & 31);  // key row of the tile = TMEM lane
    const int h = C::WG == 1 ? 0 : warp >> 2;                 // warpgroup: steps t = h mod WG
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const int j = un.j0 + r;
    const bool row_ok = j < p.Sk;
    const float c = p.scale_log2;
    bool ok = true;
    const int nst = kv_stages<D>(un);
    for (int t = h; t < un.steps; t += C::WG) {
        const int slot = t % nst;
        const int b = t & 1;  // score buffer
        const uint32_t s_col = C::S_COL + (uint32_t)b * C::BUF, dp_col = C::DP_COL + (uint32_t)b * C::BUF;
        const int i0 = (un.it_lo + t % un.n_i) * C::BM;  // first query row of the step
        // The statistics arrived with the step's Q tile; S^T and dP^T are ready.
        ok = ok && wait_warp(bar_addr(bars, C::B_QFULL + slot), (t / nst) & 1, ctl, 26);
        ok = ok && wait_warp(bar_addr(bars, (p.stall_test && t == 0) ? C::B_NEVER : C::B_SFULL + b),
                             (t >> 1) & 1, ctl, 27);
        if (!ok) break;
        ptx::tc_fence_after();
        // Query row i0 + col is visible to key j iff lo <= col < hi.
        int lo = 0, hi = NC;
        if (p.mask_kind != kMaskNone) lo = j - i0;
        if (p.mask_kind == kMaskWindow) hi = (int)min((long long)NC, (long long)j + p.window - i0);
        if (!row_ok) lo = NC;
        const bool masked = lo > 0 || hi < NC;
        const float4 *L4 = reinterpret_cast<const float4 *>(sStat + slot * C::STAT_BYTES);
        const float4 *D4 = reinterpret_cast<const float4 *>(sStat + slot * C::STAT_BYTES + C::BM * 4);
        if constexpr (C::SPLIT) {
            uint32_t s[NC], dp[NC], pw[NC / 2], dsw[NC / 2];
            ptx::tmem_ld_x32<0>(lane_base + s_col, s);
            ptx::tmem_ld_x32<32>(lane_base + s_col + 32, s);
            ptx::tmem_wait_ld();
            ptx::reg_fence<NC>(s);
            bwd_kv_p<NC, kFP16>(s, L4, lo, hi, masked, c, pw);
            if (C::ROLES && un.role == 0) {
                // dV role: P^T over the first half of this step's S^T
                ptx::tmem_st_x32<0>(lane_base + s_col, pw);
            } else {
                if (!wait_warp(bar_addr(bars, C::B_DPFULL + b), (t >> 1) & 1, ctl, 57)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                ptx::tmem_ld_x32<0>(lane_base + dp_col, dp);
                ptx::tmem_ld_x32<32>(lane_base + dp_col + 32, dp);
                ptx::tmem_wait_ld();
                ptx::reg_fence<NC>(dp);
                bwd_kv_ds<NC, kFP16>(s, dp, D4, dsw);
                // P^T (unless the dK role) and dS^T over the first halves of
                // this step's S^T and dP^T (read into registers above)
                if (!C::ROLES) ptx::tmem_st_x32<0>(lane_base + s_col, pw);
                ptx::tmem_st_x32<0>(lane_base + dp_col, dsw);
            }
        } else {
#pragma unroll
        for (int pass = 0; pass < C::WG; ++pass) {
            uint32_t s[HC], dp[HC], pw[HC / 2], dsw[HC / 2];
            ptx::tmem_ld_x32<0>(lane_base + s_col + pass * HC, s);
            ptx::tmem_ld_x32<0>(lane_base + dp_col + pass * HC, dp);
            if constexpr (HC == 64) {
                ptx::tmem_ld_x32<32>(lane_base + s_col + 32, s);
                ptx::tmem_ld_x32<32>(lane_base + dp_col + 32, dp);
            }
            ptx::tmem_wait_ld();
            ptx::reg_fence<HC>(s);
            ptx::reg_fence<HC>(dp);
            bwd_kv_p_ds<HC, kFP16>(s, dp, L4, D4, pass * HC, lo, hi, masked, c, pw, dsw);
            // P^T and dS^T of the pass over the step's S^T and dP^T columns
            // pass * HC / 2 .. + HC / 2 (one pass: 0..31 after reading 0..63;
            // two: 0..15 after 0..31, then 16..31 after 32..63)
            if constexpr (HC == 64) {
                ptx::tmem_st_x32<0>(lane_base + s_col, pw);
                ptx::tmem_st_x32<0>(lane_base + dp_col, dsw);
            } else {
                ptx::tmem_st_x16<0>(lane_base + s_col + pass * (HC / 2), pw);
                ptx::tmem_st_x16<0>(lane_base + dp_col + pass * (HC / 2), dsw);
            }
        }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_addr(bars, C::B_PFULL + b));
    }

    // Epilogue: dV and scale * dK of this thread's key row, columns h*D/WG ..
    if (un.steps > 0) {
        if (!ok || !wait_warp(bar_addr(bars, C::B_DONE), 0, ctl, 29)) return;
        ptx::tc_fence_after();
    }
    constexpr int HALF = C::DA / C::WG;  // accumulator columns this warp stores
    const bool st_dv = !(C::ROLES && un.role == 1), st_dk = !(C::ROLES && un.role == 0);
    const size_t row = ((size_t)un.b * p.Hkv + un.kvh) * (size_t)p.Sk + (size_t)j;
    const size_t col = (size_t)h * HALF;
    uint8_t *dv_row = static_cast<uint8_t *>(p.dv) + (row * D + col) * 2;
    uint8_t *dk_row = static_cast<uint8_t *>(p.dk) + (row * D + col) * 2;
    if (un.steps == 0) {
        if (row_ok) {
            if (st_dv) store_zero_row(dv_row, HALF * 2);
            if (st_dk) store_zero_row(dk_row, HALF * 2);
        }
        return;
    }
#pragma unroll
    for (int cc = 0; cc < HALF / 32; ++cc) {
        uint32_t rr[32];
        if (st_dv) {
            ptx::tmem_ld_x32<0>(lane_base + C::DV_COL + h * HALF + cc * 32, rr);
            ptx::tmem_wait_ld();
            ptx::reg_fence<32>(rr);
            if (row_ok) store_row32<kFP16>(dv_row + cc * 64, rr, 1.f);
        }
        if (st_dk) {
            ptx::tmem_ld_x32<0>(lane_base + C::DK_COL + h * HALF + cc * 32, rr);
            ptx::tmem_wait_ld();
            ptx::reg_fence<32>(rr);
            if (row_ok) store_row32<kFP16>(dk_row + cc * 64, rr, p.scale);
        }
    }
}

template <int D, bool kFP16>
__global__ void __launch_bounds__(BwdKVCfg<D>::NUM_THREADS, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdKVCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sK = smem;
    uint8_t *sV = sK + C::KV_BYTES;
    uint8_t *sQ = sV + C::KV_BYTES;
    uint8_t *sDO = sQ + C::ST * C::Q_BYTES;
    uint8_t *sX = sDO + C::ST * C::Q_BYTES;     // X_BYTES
    uint8_t *sStat = sX + C::X_BYTES;           // STM slots
    uint64_t *bar_mem = reinterpret_cast<uint64_t *>(smem + C::SMEM_TILES);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bar_mem + C::NUM_BARS);
    Ctl *ctl = reinterpret_cast<Ctl *>(tmem_holder + 2);  // 8-byte aligned
    const uint32_t bars = ptx::smem_addr(bar_mem);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_addr(bars, C::B_KVFULL), 1);
        for (int s = 0; s < C::STM; ++s) {
            ptx::mbar_init(bar_addr(bars, C::B_QFULL + s), 1);
            ptx::mbar_init(bar_addr(bars, C::B_QEMPTY + s), 2);  // one commit from each issuer
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_addr(bars, C::B_SFULL + b), 1);
            ptx::mbar_init(bar_addr(bars, C::B_DPFULL + b), 1);
            ptx::mbar_init(bar_addr(bars, C::B_PFULL + b), C::NUM_COMPUTE / C::WG);
            ptx::mbar_init(bar_addr(bars, C::B_PFREE + b), 1);
        }
        ptx::mbar_init(bar_addr(bars, C::B_DOFULL), 1);
        ptx::mbar_init(bar_addr(bars, C::B_DOEMPTY), 1);
        ptx::mbar_init(bar_addr(bars, C::B_DONE), 1);
        ptx::mbar_init(bar_addr(bars, C::B_DRAIN), 1);
        ptx::mbar_init(bar_addr(bars, C::B_DRAIN + 1), 1);
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
        ptx::prefetch_tensormap(&p.tm_do);
        ptx::prefetch_tensormap(&p.tm_k);
        ptx::prefetch_tensormap(&p.tm_v);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const KVUnit un = decode_kv_unit<D>(p);

    if (warp < C::NUM_COMPUTE / 32) {
        bwd_kv_compute_role<D, kFP16>(p, un, sStat, bars, tmem, ctl);
    } else if (warp == C::MMA_WARP) {
        bwd_kv_mma_s_role<D, kFP16>(p, un, sK, sV, sQ, sDO, sX, bars, tmem, ctl);
    } else if (warp == C::MMA_G_WARP) {
        bwd_kv_mma_g_role<D, kFP16>(p, un, sQ, sDO, sV, sX, bars, tmem, ctl);
    } else {
        bwd_kv_tma_role<D>(p, un, sK, sV, sQ, sDO, sX, sStat, bars, ctl);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------- dQ

template <int D>
struct BwdQCfg {
    static constexpr int BM = 128;                // query rows per CTA = TMEM lanes
    // d = 256 takes 64-key steps: its 256-column dQ accumulator then fits in
    // tensor memory next to S, dP and dS, and its tiles in shared memory.
    static constexpr int BN = (D == 256) ? 64 : 128;               // keys per step
    static constexpr int KST = (D == 64) ? 4 : (D == 128) ? 3 : 2;  // K stages (free after dQ)
    static constexpr int VST = (D == 64) ? 3 : (D == 128) ? 2 : 1;  // V stages (free after dP)
    static constexpr int Q_BOX = BM * 128;
    static constexpr int KV_BOX = BN * 128;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;
    // Warps 0-7 compute: warp w owns query rows 32 (w & 3) .. + 31 (its TMEM
    // lanes), one per thread, and key columns 64 (w >> 2) .. + 63 of every
    // step; warp 8 issues S and dP, warp 9 dQ, warp 10 the copies.  A
    // tcgen05.mma blocks its issuing thread while the tensor pipe's queue is
    // full, so with one issuer dQ of step t waited behind the score products
    // of step t+1 and the next score products behind dQ.
    static constexpr int NUM_COMPUTE = 256;
    static constexpr int COLS = BN / 2;
    static constexpr int MMA_WARP = 8;
    static constexpr int MMA_G_WARP = 9;
    static constexpr int TMA_WARP = 10;
    static constexpr int NUM_THREADS = 352;
    // Tensor memory: S and dP (fp32, BN columns each), the dQ accumulator,
    // dS (16-bit pairs, BN/2 columns).
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0;
    static constexpr uint32_t DP_COL = BN;
    static constexpr uint32_t DQ_COL = 2 * BN;
    static constexpr uint32_t DS_COL = 384;
    static constexpr int B_QFULL = 0;
    static constexpr int B_KFULL = 1;                 // [KST]
    static constexpr int B_KEMPTY = B_KFULL + KST;    // [KST]
    static constexpr int B_VFULL = B_KEMPTY + KST;    // [VST]
    static constexpr int B_VEMPTY = B_VFULL + VST;    // [VST]
    // d = 128: S and dP have their own ready and free barriers, so the
    // compute warps exponentiate S while dP is still being formed and the
    // next S starts as soon as this one is read.  At d = 64 and 256 the extra
    // round trip cost more than it hid: there dP goes first (its V slot frees
    // earlier) and S's barriers cover both.
    static constexpr bool SPLIT = (D == 128);
    static constexpr int B_SFULL = B_VEMPTY + VST;  // S formed (and dP, unless SPLIT)
    static constexpr int B_SFREE = B_SFULL + 1;     // S (and dP) read by the compute warps
    static constexpr int B_DPFULL = B_SFREE + 1;    // SPLIT: dP formed
    static constexpr int B_DPFREE = B_DPFULL + 1;   // SPLIT: dP read by the compute warps
    static constexpr int B_PFULL = B_DPFREE + 1;
    static constexpr int B_PFREE = B_PFULL + 1;
    static constexpr int B_DONE = B_PFREE + 1;
    static constexpr int B_DRAIN = B_DONE + 1;    // [2]: each issuer's MMAs finished
    static constexpr int B_NEVER = B_DRAIN + 2;  // no arrivals (the stall test's wait)
    static constexpr int NUM_BARS = B_NEVER + 1;
    static constexpr int SMEM_TILES = 2 * Q_BYTES + (KST + VST) * KV_BYTES;
    static constexpr int SMEM_BYTES = 1024 + SMEM_TILES + NUM_BARS * 8 + 32;
    static_assert(DQ_COL + D <= DS_COL && DS_COL + BN / 2 <= TMEM_COLS, "tensor memory overflow");
    static_assert(SMEM_BYTES <= 232448, "shared memory overflow");
};

struct QUnit {
    int b, h, kvh, i0;
    int lo, n;  // key tiles lo .. lo + n
};

template <int D>
__device__ __forceinline__ QUnit decode_q_unit(const BwdParams &p) {
    constexpr int BN = BwdQCfg<D>::BN;
    QUnit u;
    const int BH = p.B * p.H;
    const int g = p.n_tiles - 1 - (int)blockIdx.x / BH;  // longest query tiles first
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

template <int D>
__device__ void bwd_q_tma_role(const BwdParams &p, const QUnit &un, uint8_t *sQ, uint8_t *sDO,
                               uint8_t *sK, uint8_t *sV, uint32_t bars, Ctl *ctl) {
    using C = BwdQCfg<D>;
    const bool leader = ptx::lane_id() == 0;
    const uint64_t pol_last = ptx::policy_evict_last();
    const uint64_t pol_first = ptx::policy_evict_first();
    if (un.n == 0) return;
    if (leader) {
        const uint32_t fb = bar_addr(bars, C::B_QFULL);
        ptx::mbar_arrive_expect_tx(fb, 2 * C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            ptx::tma_load_4d(ptx::smem_addr(sQ) + c * C::Q_BOX, &p.tm_q, fb, c * 64, un.i0, un.h, un.b,
                             pol_first);
            ptx::tma_load_4d(ptx::smem_addr(sDO) + c * C::Q_BOX, &p.tm_do, fb, c * 64, un.i0, un.h, un.b,
                             pol_first);
        }
    }
    // V of a step frees earlier (after dP) than K (after dQ), so the copies
    // go out in the order K_t, V_t and a V copy rarely waits behind a K slot.
    int k_issued = 0, v_issued = 0;
    bool ok = true;
    for (int t = 0; t < un.n && ok; ++t) {
        const int k0 = (un.lo + t) * C::BN;
        const int ks = t % C::KST, vs = t % C::VST;
        if (!wait_warp_backoff(bar_addr(bars, C::B_KEMPTY + ks), ((t / C::KST) & 1) ^ 1, ctl, 31)) {
            ok = false;
            break;
        }
        if (leader) {
            const uint32_t fb = bar_addr(bars, C::B_KFULL + ks);
            ptx::mbar_arrive_expect_tx(fb, C::KV_BYTES);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                ptx::tma_load_4d(ptx::smem_addr(sK + ks * C::KV_BYTES) + c * C::KV_BOX, &p.tm_k, fb, c * 64,
                                 k0, un.kvh, un.b, pol_last);
        }
        __syncwarp();
        ++k_issued;
        if (!wait_warp_backoff(bar_addr(bars, C::B_VEMPTY + vs), ((t / C::VST) & 1) ^ 1, ctl, 39)) {
            ok = false;
            break;
        }
        if (leader) {
            const uint32_t fb = bar_addr(bars, C::B_VFULL + vs);
            ptx::mbar_arrive_expect_tx(fb, C::KV_BYTES);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                ptx::tma_load_4d(ptx::smem_addr(sV + vs * C::KV_BYTES) + c * C::KV_BOX, &p.tm_v, fb, c * 64,
                                 k0, un.kvh, un.b, pol_last);
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

// The two MMA issuers of the dQ kernel: S of step t goes out as soon as the
// compute warps have read S of step t-1, then dP as soon as they have read
// dP of step t-1 (without SPLIT: dP, then S, once both of step t-1 are
// read); dQ += dS K of step t as soon as its dS is written.  A K slot is free
// after dQ, a V slot after dP.
template <int D, bool kFP16>
__device__ void bwd_q_mma_s_role(const BwdParams &p, const QUnit &un, uint8_t *sQ, uint8_t *sDO,
                                 uint8_t *sK, uint8_t *sV, uint32_t bars, uint32_t tmem, Ctl *ctl) {
    using C = BwdQCfg<D>;
    constexpr uint32_t kIdescS = make_idesc(C::BM, C::BN, kFP16, false);
    const bool leader = ptx::lane_id() == 0;
    const uint64_t qd = smem_desc(ptx::smem_addr(sQ), 16);
    const uint64_t od = smem_desc(ptx::smem_addr(sDO), 16);
    bool ok = un.n == 0 || wait_warp(bar_addr(bars, C::B_QFULL), 0, ctl, 32);
    for (int t = 0; ok && t < un.n; ++t) {
        const int ks = t % C::KST, vs = t % C::VST;
        if (!wait_warp(bar_addr(bars, C::B_KFULL + ks), (t / C::KST) & 1, ctl, 33) ||
            !wait_warp(bar_addr(bars, C::B_VFULL + vs), (t / C::VST) & 1, ctl, 40)) {
            ok = false;
            break;
        }
        if (t >= 1 && !wait_warp(bar_addr(bars, C::B_SFREE), (t - 1) & 1, ctl, 34)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        if constexpr (C::SPLIT) {
            const uint64_t kd = smem_desc(ptx::smem_addr(sK + ks * C::KV_BYTES), 16);
            const uint64_t vd = smem_desc(ptx::smem_addr(sV + vs * C::KV_BYTES), 16);
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + C::S_COL, qd + kmajor_step(kk, C::Q_BOX), kd + kmajor_step(kk, C::KV_BOX),
                                kIdescS, kk > 0 ? 1u : 0u);
                ptx::mma_commit(bar_addr(bars, C::B_SFULL));
            }
            __syncwarp();
            if (t >= 1 && !wait_warp(bar_addr(bars, C::B_DPFREE), (t - 1) & 1, ctl, 55)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + C::DP_COL, od + kmajor_step(kk, C::Q_BOX), vd + kmajor_step(kk, C::KV_BOX),
                                kIdescS, kk > 0 ? 1u : 0u);
                ptx::mma_commit(bar_addr(bars, C::B_DPFULL));
                ptx::mma_commit(bar_addr(bars, C::B_VEMPTY + vs));
            }
        } else if (leader) {
            const uint64_t kd = smem_desc(ptx::smem_addr(sK + ks * C::KV_BYTES), 16);
            const uint64_t vd = smem_desc(ptx::smem_addr(sV + vs * C::KV_BYTES), 16);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::mma_ss(tmem + C::DP_COL, od + kmajor_step(kk, C::Q_BOX), vd + kmajor_step(kk, C::KV_BOX),
                            kIdescS, kk > 0 ? 1u : 0u);
            ptx::mma_commit(bar_addr(bars, C::B_VEMPTY + vs));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::mma_ss(tmem + C::S_COL, qd + kmajor_step(kk, C::Q_BOX), kd + kmajor_step(kk, C::KV_BOX),
                            kIdescS, kk > 0 ? 1u : 0u);
            ptx::mma_commit(bar_addr(bars, C::B_SFULL));
        }
        __syncwarp();
    }
    if (leader) ptx::mma_commit(bar_addr(bars, C::B_DRAIN));
    __syncwarp();
    wait_bar_drain(bar_addr(bars, C::B_DRAIN), 0);
}

template <int D, bool kFP16>
__device__ void bwd_q_mma_g_role(const BwdParams &p, const QUnit &un, uint8_t *sK, uint32_t bars,
                                 uint32_t tmem, Ctl *ctl) {
    using C = BwdQCfg<D>;
    constexpr uint32_t kIdescG = make_idesc(C::BM, D, kFP16, true);  // dQ: N = d, K MN-major
    const bool leader = ptx::lane_id() == 0;
    bool ok = true;
    for (int t = 0; ok && t < un.n; ++t) {
        const int slot = t % C::KST;
        // K of step t has landed (this warp reads it too); dS of step t is written
        if (!wait_warp(bar_addr(bars, C::B_KFULL + slot), (t / C::KST) & 1, ctl, 52) ||
            !wait_warp(bar_addr(bars, C::B_PFULL), t & 1, ctl, 35)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        if (leader) {
            // K as the MN-major B operand: K = keys (16 = 2048 bytes), N = d.
            const uint64_t km = smem_desc(ptx::smem_addr(sK + slot * C::KV_BYTES), C::KV_BOX);
#pragma unroll
            for (int kk = 0; kk < C::BN / 16; ++kk)
                ptx::mma_ts(tmem + C::DQ_COL, tmem + C::DS_COL + kk * 8, km + (uint32_t)((kk * 2048) >> 4),
                            kIdescG, (t > 0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(bar_addr(bars, C::B_PFREE));
            ptx::mma_commit(bar_addr(bars, C::B_KEMPTY + slot));
            if (t + 1 == un.n) ptx::mma_commit(bar_addr(bars, C::B_DONE));
        }
        __syncwarp();
    }
    if (leader) ptx::mma_commit(bar_addr(bars, C::B_DRAIN + 1));
    __syncwarp();
    wait_bar_drain(bar_addr(bars, C::B_DRAIN + 1), 0);
}

template <int D, bool kFP16>
__device__ void bwd_q_compute_role(const BwdParams &p, const QUnit &un, uint32_t bars, uint32_t tmem,
                                   Ctl *ctl) {
    using C = BwdQCfg<D>;
    constexpr int NC = C::COLS;
    const int warp = (int)threadIdx.x >> 5;
    const int r = 32 * (warp & 3) + ((int)threadIdx.x & 31);  // query row of the tile = TMEM lane
    const int h = warp >> 2;                                  // key columns h*NC .. + NC
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const int i = un.i0 + r;
    const bool row_ok = i < p.Sq;
    const size_t srow = ((size_t)un.b * p.H + un.h) * (size_t)p.Sq_pad + (size_t)i;
    const float L = p.l2[srow];      // +inf on padding rows: P = 0
    const float Dl = p.delta[srow];
    const float c = p.scale_log2;
    const uint64_t c2 = ptx::f32x2(c, c), nl2 = ptx::f32x2(-L, -L), nd2 = ptx::f32x2(-Dl, -Dl);
    const uint64_t mz2 = ptx::f32x2(-0.f, -0.f);
    bool ok = true;
    for (int t = 0; t < un.n; ++t) {
        const int k0 = (un.lo + t) * C::BN + h * NC;  // first key of this warp's columns
        // Key column k0 + col is visible to row i iff lo <= col < hi.
        int lo = 0, hi = min(NC, p.Sk - k0);
        if (p.mask_kind != kMaskNone) hi = min(hi, i - k0 + 1);
        if (p.mask_kind == kMaskWindow) lo = max(0, i - p.window + 1 - k0);
        const bool masked = lo > 0 || hi < NC;
        if (!wait_warp(bar_addr(bars, (p.stall_test && t == 0) ? C::B_NEVER : C::B_SFULL), t & 1, ctl, 36)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        uint32_t s[NC], dp[NC], w[NC / 2];
        ptx::tmem_ld_x32<0>(lane_base + C::S_COL + h * NC, s);
        if constexpr (!C::SPLIT) ptx::tmem_ld_x32<0>(lane_base + C::DP_COL + h * NC, dp);
        if constexpr (NC == 64) {
            ptx::tmem_ld_x32<32>(lane_base + C::S_COL + h * NC + 32, s);
            if constexpr (!C::SPLIT) ptx::tmem_ld_x32<32>(lane_base + C::DP_COL + h * NC + 32, dp);
        }
        ptx::tmem_wait_ld();
        ptx::reg_fence<NC>(s);
        if constexpr (!C::SPLIT) ptx::reg_fence<NC>(dp);
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_addr(bars, C::B_SFREE));
        // Packed fp32 pairs: s c - L and dP - delta as one instruction per
        // pair each, and P (dP - delta) as an fma with -0 (the exact product,
        // sign of zero included).
        if constexpr (C::SPLIT) {
            // P = exp2(s c - L) (masked) while dP is still being formed
#pragma unroll
            for (int e = 0; e < NC; e += 2) {
                float x0, x1;
                ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(s[e]), __uint_as_float(s[e + 1])),
                                                 c2, nl2), x0, x1);
                float p0 = ptx::ex2_approx(x0);
                float p1 = ptx::ex2_approx(x1);
                if (masked) {
                    p0 = (e >= lo && e < hi) ? p0 : 0.f;
                    p1 = (e + 1 >= lo && e + 1 < hi) ? p1 : 0.f;
                }
                s[e] = __float_as_uint(p0);
                s[e + 1] = __float_as_uint(p1);
            }
            if (!wait_warp(bar_addr(bars, C::B_DPFULL), t & 1, ctl, 56)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            ptx::tmem_ld_x32<0>(lane_base + C::DP_COL + h * NC, dp);
            if constexpr (NC == 64) ptx::tmem_ld_x32<32>(lane_base + C::DP_COL + h * NC + 32, dp);
            ptx::tmem_wait_ld();
            ptx::reg_fence<NC>(dp);
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_addr(bars, C::B_DPFREE));
#pragma unroll
            for (int e = 0; e < NC; e += 2) {
                float g0, g1, d0, d1;
                ptx::unpack_f32x2(ptx::add_f32x2(ptx::f32x2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                                 nd2), g0, g1);
                ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(s[e]), __uint_as_float(s[e + 1])),
                                                 ptx::f32x2(g0, g1), mz2), d0, d1);
                w[e / 2] = pack2b<kFP16>(d0, d1);
            }
        } else {
#pragma unroll
            for (int e = 0; e < NC; e += 2) {
                float x0, x1, g0, g1, d0, d1;
                ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(s[e]), __uint_as_float(s[e + 1])),
                                                 c2, nl2), x0, x1);
                float p0 = ptx::ex2_approx(x0);
                float p1 = ptx::ex2_approx(x1);
                if (masked) {
                    p0 = (e >= lo && e < hi) ? p0 : 0.f;
                    p1 = (e + 1 >= lo && e + 1 < hi) ? p1 : 0.f;
                }
                ptx::unpack_f32x2(ptx::add_f32x2(ptx::f32x2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                                 nd2), g0, g1);
                ptx::unpack_f32x2(ptx::fma_f32x2(ptx::f32x2(p0, p1), ptx::f32x2(g0, g1), mz2), d0, d1);
                w[e / 2] = pack2b<kFP16>(d0, d1);
            }
        }
        // dQ of step t-1 has read the dS area
        if (t >= 1 && !wait_warp(bar_addr(bars, C::B_PFREE), (t - 1) & 1, ctl, 37)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        if constexpr (NC == 64) {
            ptx::tmem_st_x32<0>(lane_base + C::DS_COL + h * (NC / 2), w);
        } else {
            ptx::tmem_st_x16<0>(lane_base + C::DS_COL + h * (NC / 2), w);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_addr(bars, C::B_PFULL));
    }

    constexpr int HALF = D / 2;
    uint8_t *dq_row = static_cast<uint8_t *>(p.dq) +
                      (((size_t)un.b * p.H + un.h) * (size_t)p.Sq + (size_t)i) * D * 2 + h * HALF * 2;
    if (un.n == 0) {
        if (row_ok) store_zero_row(dq_row, HALF * 2);
        return;
    }
    if (!ok || !wait_warp(bar_addr(bars, C::B_DONE), 0, ctl, 38)) return;
    ptx::tc_fence_after();
#pragma unroll
    for (int cc = 0; cc < HALF / 32; ++cc) {
        uint32_t rr[32];
        ptx::tmem_ld_x32<0>(lane_base + C::DQ_COL + h * HALF + cc * 32, rr);
        ptx::tmem_wait_ld();
        ptx::reg_fence<32>(rr);
        if (row_ok) store_row32<kFP16>(dq_row + cc * 64, rr, p.scale);
    }
}

template <int D, bool kFP16>
__global__ void __launch_bounds__(BwdQCfg<D>::NUM_THREADS, 1)
    fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdQCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem;
    uint8_t *sDO = sQ + C::Q_BYTES;
    uint8_t *sK = sDO + C::Q_BYTES;
    uint8_t *sV = sK + C::KST * C::KV_BYTES;
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
        ptx::mbar_init(bar_addr(bars, C::B_SFULL), 1);
        ptx::mbar_init(bar_addr(bars, C::B_SFREE), C::NUM_COMPUTE);
        ptx::mbar_init(bar_addr(bars, C::B_DPFULL), 1);
        ptx::mbar_init(bar_addr(bars, C::B_DPFREE), C::NUM_COMPUTE);
        ptx::mbar_init(bar_addr(bars, C::B_PFULL), C::NUM_COMPUTE);
        ptx::mbar_init(bar_addr(bars, C::B_PFREE), 1);
        ptx::mbar_init(bar_addr(bars, C::B_DONE), 1);
        ptx::mbar_init(bar_addr(bars, C::B_DRAIN), 1);
        ptx::mbar_init(bar_addr(bars, C::B_DRAIN + 1), 1);
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
        ptx::prefetch_tensormap(&p.tm_do);
        ptx::prefetch_tensormap(&p.tm_k);
        ptx::prefetch_tensormap(&p.tm_v);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const QUnit un = decode_q_unit<D>(p);

    if (warp < C::NUM_COMPUTE / 32) {
        bwd_q_compute_role<D, kFP16>(p, un, bars, tmem, ctl);
    } else if (warp == C::MMA_WARP) {
        bwd_q_mma_s_role<D, kFP16>(p, un, sQ, sDO, sK, sV, bars, tmem, ctl);
    } else if (warp == C::MMA_G_WARP) {
        bwd_q_mma_g_role<D, kFP16>(p, un, sK, bars, tmem, ctl);
    } else {
        bwd_q_tma_role<D>(p, un, sQ, sDO, sK, sV, bars, ctl);
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
