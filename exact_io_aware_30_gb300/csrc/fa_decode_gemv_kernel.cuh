// fa_decode_gemv_kernel.cuh -- decoding over a paged K/V cache when at most
// two query rows share a K/V head (one new row per request and head, or a
// pair), for sm_103a (GB300).
//
// The arithmetic is that of the tiled forward pass ("FlashAttention: Why
// Tiling Attention Makes Transformers Fast Without Changing the Result",
// sections "Online softmax: correct as you go" and "The tiled forward pass"):
// a running max and sum per row, O rescaled when the max grows, one division
// at the end.  The cache walk, the key ranges and their merge are those of
// fa_decode_kernel ("Flash attention and memory-efficient attention
// variants", sections "A different bottleneck: the KV cache during inference"
// and "PagedAttention: memory management borrowed from an operating system").
//
// With R <= 2 rows, S = q K^T and O += P V are matrix-vector products: a
// 128-row tensor-core tile would be 98 % padding, and the kernel is bound by
// reading the cache.  So the products run on the CUDA cores in fp32, and the
// design is about keeping HBM busy:
//   - a producer warp gathers each stage's blocks with plain bulk copies
//     (cp.async.bulk: one copy per block slab of K and of V, each block of one
//     head being contiguous in the cache) into a ring of three 32 KB stages;
//   - about 105 KB of shared memory per CTA, so two CTAs share an SM and one
//     CTA's start (barrier set-up, first copies) hides behind the other's
//     stream;
//   - four compute warps split each stage's keys.  Scores: d/16 lanes per key,
//     16 elements each, reduced by shuffles.  P V: each lane owns d/32 output
//     columns and reads one stage row per key (conflict-free), the key's
//     weights arriving by one broadcast shared-memory load.  Each warp keeps
//     its own running max, sum and O; the four are merged at the end with the
//     same rescaling.  Products use packed fp32 pairs (fma.rn.f32x2).
// Weights stay fp32 (not rounded to 16 bits before P V).  At four rows the
// score phase (4 x d FMAs and the lane reductions per key) no longer hides
// under the cache stream, and the tensor-core kernel serves those.
#pragma once

#include <math.h>
#include <stdint.h>

#include "fa_decode_kernel.cuh"

namespace fa {

struct GemvParams {
    const void *q;           // [B*H*Sq, d] 16-bit
    const void *k_cache;     // [num_blocks, Hkv, bs, d] 16-bit
    const void *v_cache;     // same layout
    const int *block_table;  // [B, max_blocks]
    const int *seq_lens;     // [B]
    float *part_o;           // [n_splits, B*H*Sq, d] fp32, normalised per split
    float *part_lse;         // [n_splits, B*H*Sq] fp32, natural log; -inf: split saw no key
    int B, H, Hkv, kv_group, Sq, R;  // R = kv_group * Sq rows per CTA (<= 2)
    int bs, max_blocks, num_blocks, max_seq_len;
    int mask_kind;
    int n_splits, keys_per_split;  // keys_per_split: a multiple of the stage's keys
    float scale_log2;
    uint64_t wait_limit_ns;
    int stall_test;          // test only: the compute warps' first wait is on a barrier nothing completes
};

template <int D>
struct GemvCfg {
    static constexpr int LPK = D / 16;       // lanes per key in the score phase (16 elements each)
    static constexpr int KPI = 32 / LPK;     // keys per warp per step
    static constexpr int CK = 8192 / D;      // keys per stage: 16 KB of K and 16 KB of V
    static constexpr int NW = 4;             // compute warps
    static constexpr int KPW = CK / NW;      // keys per compute warp per stage
    static constexpr int STEPS = KPW / KPI;  // score steps per warp per stage
    static constexpr int CPL = D / 32;       // output columns per lane
    static constexpr int RMAX = 2;
    static constexpr int NST = 3;            // stages in the ring
    static constexpr int HALF = CK * D * 2;  // bytes of K (or of V) in a stage
    static constexpr int STAGE = 2 * HALF;
    static constexpr int PRODUCER = NW;      // warp index of the producer
    static constexpr int NUM_THREADS = 32 * (NW + 1);
    static constexpr int B_FULL = 0;          // [NST]: stage loaded
    static constexpr int B_EMPTY = NST;       // [NST]: stage read by the four compute warps
    static constexpr int B_NEVER = 2 * NST;   // no arrivals (the stall test's wait)
    static constexpr int NUM_BARS = B_NEVER + 1;
    static constexpr int MERGE_BYTES = NW * RMAX * (D + 2) * 4;
    static constexpr int PBUF_BYTES = NW * KPW * RMAX * 4;  // per warp: the weights of its keys, rows inner
    static constexpr int SMEM_BYTES = 128 + NST * STAGE + MERGE_BYTES + PBUF_BYTES + NUM_BARS * 8 + 16;
    static_assert(STEPS * KPI == KPW && KPW * NW == CK, "stage split");
    static_assert(2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs per SM");
};

struct GemvUnit {
    int b, kvh, split, L, k_beg, k_end, n;  // keys [k_beg, k_end) in n stages
};

template <int D>
__device__ __forceinline__ GemvUnit decode_gemv_unit(const GemvParams &p) {
    GemvUnit u;
    u.split = (int)blockIdx.x % p.n_splits;
    const int bk = (int)blockIdx.x / p.n_splits;
    u.b = bk / p.Hkv;
    u.kvh = bk - u.b * p.Hkv;
    // the caller guarantees Sq <= seq_lens[b] <= max_seq_len; clamp anyway so
    // that no index leaves the block table
    u.L = min(max(p.seq_lens[u.b], p.Sq), p.max_seq_len);
    u.k_beg = u.split * p.keys_per_split;
    u.k_end = min(u.k_beg + p.keys_per_split, u.L);
    constexpr int CK = GemvCfg<D>::CK;
    u.n = u.k_end > u.k_beg ? (u.k_end - u.k_beg + CK - 1) / CK : 0;
    return u;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t ld_shared_b32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// Two 16-bit values (low half first) as fp32.
template <bool kFP16>
__device__ __forceinline__ void unpack2(uint32_t w, float &lo, float &hi) {
    if constexpr (kFP16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
        lo = f.x;
        hi = f.y;
    } else {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xffff0000u);
    }
}

// Two 16-bit values as one packed fp32 pair (for the f32x2 instructions).
template <bool kFP16>
__device__ __forceinline__ uint64_t pair2(uint32_t w) {
    float lo, hi;
    unpack2<kFP16>(w, lo, hi);
    return ptx::f32x2(lo, hi);
}

template <bool kFP16>
__device__ __forceinline__ void unpack8(uint4 v, float *f) {
    unpack2<kFP16>(v.x, f[0], f[1]);
    unpack2<kFP16>(v.y, f[2], f[3]);
    unpack2<kFP16>(v.z, f[4], f[5]);
    unpack2<kFP16>(v.w, f[6], f[7]);
}

// Producer warp: per stage, the blocks holding keys [key0, key0 + CK) of this
// unit (whole blocks when block_size <= CK, else the CK-key part of one
// block), one bulk copy of K and one of V per block, by one lane each.  A
// table entry outside [0, num_blocks) reads as zeros: the warp clears that
// part of the stage instead.
template <int D>
__device__ void gemv_producer(const GemvParams &p, const GemvUnit &u, uint8_t *stages, uint32_t bars,
                              Ctl *ctl) {
    using C = GemvCfg<D>;
    const int lane = ptx::lane_id();
    const int *row = p.block_table + (size_t)u.b * p.max_blocks;
    const size_t slab = (size_t)p.bs * D * 2;  // one block of one head
    const size_t blk_stride = (size_t)p.Hkv * slab;
    const uint8_t *kc = static_cast<const uint8_t *>(p.k_cache) + (size_t)u.kvh * slab;
    const uint8_t *vc = static_cast<const uint8_t *>(p.v_cache) + (size_t)u.kvh * slab;
    const int piece_keys = p.bs <= C::CK ? p.bs : C::CK;
    const uint32_t piece_bytes = (uint32_t)piece_keys * D * 2;
    int issued = 0;
    bool ok = true;
    for (int s = 0; s < u.n; ++s) {
        const int slot = s % C::NST;
        if (!wait_warp_backoff(bar_addr(bars, C::B_EMPTY + slot), ((s / C::NST) & 1) ^ 1, ctl, 81)) {
            ok = false;
            break;
        }
        const int key0 = u.k_beg + s * C::CK;  // a multiple of CK, so of piece_keys
        const int key_hi = min(key0 + C::CK, u.k_end);
        const int pieces = (key_hi - key0 + piece_keys - 1) / piece_keys;  // <= CK / 16 <= 8
        uint8_t *dK = stages + slot * C::STAGE;
        uint8_t *dV = dK + C::HALF;
        bool valid = false;
        size_t src = 0;
        if (lane < pieces) {
            const int first = key0 + lane * piece_keys;
            const int nb = first / p.bs;  // < max_blocks: first < L <= max_seq_len <= max_blocks * bs
            const int phys = row[nb];
            valid = phys >= 0 && phys < p.num_blocks;
            src = (size_t)(valid ? phys : 0) * blk_stride + (size_t)(first - nb * p.bs) * D * 2;
        }
        const unsigned vmask = __ballot_sync(0xffffffffu, lane < pieces && valid);
        unsigned zmask = __ballot_sync(0xffffffffu, lane < pieces && !valid);
        if (zmask) {
            while (zmask) {
                const int j = __ffs(zmask) - 1;
                zmask &= zmask - 1;
                for (uint32_t off = (uint32_t)lane * 16u; off < piece_bytes; off += 512u) {
                    ptx::st_shared_v4(ptx::smem_addr(dK + j * piece_bytes + off), 0u, 0u, 0u, 0u);
                    ptx::st_shared_v4(ptx::smem_addr(dV + j * piece_bytes + off), 0u, 0u, 0u, 0u);
                }
            }
            ptx::fence_proxy_async_smem();
        }
        __syncwarp();
        const uint32_t fb = bar_addr(bars, C::B_FULL + slot);
        if (lane == 0) ptx::mbar_arrive_expect_tx(fb, 2u * piece_bytes * (uint32_t)__popc(vmask));
        __syncwarp();
        if (lane < pieces && valid) {
            ptx::bulk_load(ptx::smem_addr(dK + lane * piece_bytes), kc + src, piece_bytes, fb);
            ptx::bulk_load(ptx::smem_addr(dV + lane * piece_bytes), vc + src, piece_bytes, fb);
        }
        __syncwarp();
        ++issued;
    }
    if (!ok) {
        for (int t = issued - C::NST > 0 ? issued - C::NST : 0; t < issued; ++t)
            wait_bar_drain(bar_addr(bars, C::B_FULL + t % C::NST), (t / C::NST) & 1);
    }
}

// Compute warps.  RT = rows handled (R: 1 or 2).
template <int D, bool kFP16, int RT>
__device__ void gemv_compute(const GemvParams &p, const GemvUnit &u, const uint8_t *stages, float *mrg,
                             float *pbuf, uint32_t bars, Ctl *ctl, int warp) {
    using C = GemvCfg<D>;
    const int lane = ptx::lane_id();
    const int g = lane / C::LPK;  // key of the step within the warp's KPI
    const int e = lane % C::LPK;  // 16-byte chunks e and e + LPK of the key's row
    const size_t row0 = (size_t)(u.b * p.H + u.kvh * p.kv_group) * p.Sq;

    // q rows (zeros past R), the lane's 16 elements each as 8 fp32 pairs
    uint64_t q2[RT][8];
    int last[RT];  // last key each row sees
#pragma unroll
    for (int r = 0; r < RT; ++r) {
        const bool have = r < p.R;
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(p.q) +
                                                           (row0 + (have ? r : 0)) * D * 2);
        const uint4 a = have ? src[e] : make_uint4(0u, 0u, 0u, 0u);
        const uint4 b = have ? src[e + C::LPK] : make_uint4(0u, 0u, 0u, 0u);
        q2[r][0] = pair2<kFP16>(a.x);
        q2[r][1] = pair2<kFP16>(a.y);
        q2[r][2] = pair2<kFP16>(a.z);
        q2[r][3] = pair2<kFP16>(a.w);
        q2[r][4] = pair2<kFP16>(b.x);
        q2[r][5] = pair2<kFP16>(b.y);
        q2[r][6] = pair2<kFP16>(b.z);
        q2[r][7] = pair2<kFP16>(b.w);
        last[r] = (p.mask_kind == kMaskCausal) ? u.L - p.Sq + (r % p.Sq) : u.L - 1;
    }
    const float c = p.scale_log2;
    const uint64_t zero2 = ptx::f32x2(0.f, 0.f);
    float m[RT], l[RT];
    uint64_t o2[RT][C::CPL / 2];  // the lane's output columns, in pairs
#pragma unroll
    for (int r = 0; r < RT; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int cc = 0; cc < C::CPL / 2; ++cc) o2[r][cc] = zero2;
    }

    bool ok = true;
    for (int s = 0; s < u.n; ++s) {
        const int slot = s % C::NST;
        if (!wait_warp(bar_addr(bars, (p.stall_test && s == 0) ? C::B_NEVER : C::B_FULL + slot), (s / C::NST) & 1,
                       ctl, 82)) {
            ok = false;
            break;
        }
        const uint32_t sK = ptx::smem_addr(stages + slot * C::STAGE);
        const uint32_t sV = sK + C::HALF;
        const int kw0 = warp * C::KPW;                    // warp's first key in the stage
        const int key_base = u.k_beg + s * C::CK + kw0;   // its absolute index

        // scores (log2 units), hidden keys -inf: past the range or the row's
        // last key, or a stage row that holds no key of this request (a
        // select, so whatever such a row holds never enters)
        float sc[C::STEPS][RT];
#pragma unroll
        for (int it = 0; it < C::STEPS; ++it) {
            const uint32_t kr = sK + (uint32_t)((kw0 + it * C::KPI + g) * D * 2);
            const uint4 a = ld_shared_v4(kr + e * 16);
            const uint4 b = ld_shared_v4(kr + (e + C::LPK) * 16);
            const uint64_t k2[8] = {pair2<kFP16>(a.x), pair2<kFP16>(a.y), pair2<kFP16>(a.z), pair2<kFP16>(a.w),
                                    pair2<kFP16>(b.x), pair2<kFP16>(b.y), pair2<kFP16>(b.z), pair2<kFP16>(b.w)};
            const int key = key_base + it * C::KPI + g;
#pragma unroll
            for (int r = 0; r < RT; ++r) {
                uint64_t acc0 = ptx::fma_f32x2(q2[r][0], k2[0], zero2);
                uint64_t acc1 = ptx::fma_f32x2(q2[r][1], k2[1], zero2);
#pragma unroll
                for (int t = 2; t < 8; t += 2) {
                    acc0 = ptx::fma_f32x2(q2[r][t], k2[t], acc0);
                    acc1 = ptx::fma_f32x2(q2[r][t + 1], k2[t + 1], acc1);
                }
                float x0, x1, x2, x3;
                ptx::unpack_f32x2(acc0, x0, x1);
                ptx::unpack_f32x2(acc1, x2, x3);
                float acc = (x0 + x1) + (x2 + x3);
#pragma unroll
                for (int off = C::LPK / 2; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                sc[it][r] = (key < u.k_end && key <= last[r]) ? acc * c : -INFINITY;
            }
        }
        // running max, weights, sum, rescale
#pragma unroll
        for (int r = 0; r < RT; ++r) {
            float mt = sc[0][r];
#pragma unroll
            for (int it = 1; it < C::STEPS; ++it) mt = fmaxf(mt, sc[it][r]);
#pragma unroll
            for (int off = C::LPK; off < 32; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            const float m_new = fmaxf(m[r], mt);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // no visible key yet: weights 0
            const float alpha = ptx::ex2_approx(m[r] - m_use);        // 0 while m is -inf
            float ps = 0.f;
#pragma unroll
            for (int it = 0; it < C::STEPS; ++it) {
                sc[it][r] = ptx::ex2_approx(sc[it][r] - m_use);
                ps += sc[it][r];
            }
            l[r] = l[r] * alpha + ps;  // this lane's key group only; summed over groups at the end
            if (alpha != 1.f) {
                const uint64_t a2 = ptx::f32x2(alpha, alpha);
#pragma unroll
                for (int cc = 0; cc < C::CPL / 2; ++cc) o2[r][cc] = ptx::fma_f32x2(o2[r][cc], a2, zero2);
            }
            m[r] = m_new;
        }
        // this warp's weights to shared memory, [key][row]: one broadcast load
        // per key then gives P V every row's weight
        const uint32_t pw = ptx::smem_addr(pbuf + warp * C::KPW * C::RMAX);
        if (e == 0) {
#pragma unroll
            for (int it = 0; it < C::STEPS; ++it) {
                const uint32_t a = pw + (uint32_t)((it * C::KPI + g) * C::RMAX * 4);
                if constexpr (RT == 2)
                    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(a), "r"(__float_as_uint(sc[it][0])),
                                 "r"(__float_as_uint(sc[it][1])) : "memory");
                else
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(__float_as_uint(sc[it][0])) : "memory");
            }
        }
        __syncwarp();
        // O += P V over the stage's keys of this request (a key past the
        // range is never read: its row may hold anything)
#pragma unroll
        for (int it = 0; it < C::STEPS; ++it) {
#pragma unroll
            for (int gg = 0; gg < C::KPI; ++gg) {
                if (key_base + it * C::KPI + gg >= u.k_end) continue;  // warp-uniform
                const uint32_t vr = sV + (uint32_t)((kw0 + it * C::KPI + gg) * D * 2 + lane * C::CPL * 2);
                uint64_t v2[C::CPL / 2];
                if constexpr (C::CPL == 8) {
                    const uint4 w = ld_shared_v4(vr);
                    v2[0] = pair2<kFP16>(w.x);
                    v2[1] = pair2<kFP16>(w.y);
                    v2[2] = pair2<kFP16>(w.z);
                    v2[3] = pair2<kFP16>(w.w);
                } else if constexpr (C::CPL == 4) {
                    const uint2 w = ld_shared_v2(vr);
                    v2[0] = pair2<kFP16>(w.x);
                    v2[1] = pair2<kFP16>(w.y);
                } else {
                    v2[0] = pair2<kFP16>(ld_shared_b32(vr));
                }
                float pr[RT];
                const uint32_t pa = pw + (uint32_t)((it * C::KPI + gg) * C::RMAX * 4);
                if constexpr (RT == 2) {
                    const uint2 w = ld_shared_v2(pa);
                    pr[0] = __uint_as_float(w.x);
                    pr[1] = __uint_as_float(w.y);
                } else {
                    pr[0] = __uint_as_float(ld_shared_b32(pa));
                }
#pragma unroll
                for (int r = 0; r < RT; ++r) {
                    const uint64_t p2 = ptx::f32x2(pr[r], pr[r]);
#pragma unroll
                    for (int cc = 0; cc < C::CPL / 2; ++cc) o2[r][cc] = ptx::fma_f32x2(p2, v2[cc], o2[r][cc]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_addr(bars, C::B_EMPTY + slot));
    }

    // Merge the four warps' (m, l, O) per row.  Every compute thread reaches
    // the barrier, failed or not; the merge is skipped after a failure.
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int off = C::LPK; off < 32; off <<= 1) l[r] += __shfl_xor_sync(0xffffffffu, l[r], off);
    float *mo = mrg;                                   // [NW][RMAX][D]
    float *mm = mrg + C::NW * C::RMAX * D;             // [NW][RMAX]
    float *ml = mm + C::NW * C::RMAX;                  // [NW][RMAX]
#pragma unroll
    for (int r = 0; r < RT; ++r) {
#pragma unroll
        for (int cc = 0; cc < C::CPL / 2; ++cc) {
            float lo, hi;
            ptx::unpack_f32x2(o2[r][cc], lo, hi);
            mo[(warp * C::RMAX + r) * D + lane * C::CPL + 2 * cc] = lo;
            mo[(warp * C::RMAX + r) * D + lane * C::CPL + 2 * cc + 1] = hi;
        }
        if (lane == 0) {
            mm[warp * C::RMAX + r] = m[r];
            ml[warp * C::RMAX + r] = l[r];
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(C::NW * 32) : "memory");
    if (!ok || ctl->abort) return;
    const size_t n_rows = (size_t)p.B * p.H * p.Sq;
    const int tid = (int)threadIdx.x;
    for (int idx = tid; idx < RT * D; idx += C::NW * 32) {
        const int r = idx / D, col = idx - r * D;
        if (r >= p.R) break;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NW; ++w) M = fmaxf(M, mm[w * C::RMAX + r]);
        float acc = 0.f, wsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < C::NW; ++w) {
                const float f = ptx::ex2_approx(mm[w * C::RMAX + r] - M);  // 0 for a warp that saw no key
                wsum = fmaf(f, ml[w * C::RMAX + r], wsum);
                acc = fmaf(f, mo[(w * C::RMAX + r) * D + col], acc);
            }
        }
        const bool seen = wsum > 0.f;
        p.part_o[((size_t)u.split * n_rows + row0 + r) * D + col] = seen ? acc / wsum : 0.f;
        if (col == 0)
            p.part_lse[(size_t)u.split * n_rows + row0 + r] = seen ? (M + __log2f(wsum)) * kLn2 : -INFINITY;
    }
}

template <int D, bool kFP16, int RT>
__global__ void __launch_bounds__(GemvCfg<D>::NUM_THREADS, 2)
    fa_decode_gemv_kernel(const __grid_constant__ GemvParams p) {
    using C = GemvCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    uint8_t *stages = smem;
    float *mrg = reinterpret_cast<float *>(smem + C::NST * C::STAGE);
    float *pbuf = reinterpret_cast<float *>(smem + C::NST * C::STAGE + C::MERGE_BYTES);
    uint64_t *bar_mem = reinterpret_cast<uint64_t *>(smem + C::NST * C::STAGE + C::MERGE_BYTES + C::PBUF_BYTES);
    Ctl *ctl = reinterpret_cast<Ctl *>(bar_mem + C::NUM_BARS);
    const uint32_t bars = ptx::smem_addr(bar_mem);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NST; ++s) {
            ptx::mbar_init(bar_addr(bars, C::B_FULL + s), 1);
            ptx::mbar_init(bar_addr(bars, C::B_EMPTY + s), C::NW);
        }
        ptx::mbar_init(bar_addr(bars, C::B_NEVER), 1);
        ctl->abort = 0;
        ctl->limit_ns = p.wait_limit_ns;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    __syncthreads();
    const GemvUnit u = decode_gemv_unit<D>(p);
    if (warp == C::PRODUCER) {
        gemv_producer<D>(p, u, stages, bars, ctl);
    } else {
        gemv_compute<D, kFP16, RT>(p, u, stages, mrg, pbuf, bars, ctl, warp);
    }
}

}  // namespace fa
