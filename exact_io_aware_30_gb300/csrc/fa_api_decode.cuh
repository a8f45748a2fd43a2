// fa_api_decode.cuh -- host side of decoding over a paged cache
// (fa_decode_paged, fa_decode_workspace_query).
// Included once, by fa_api.cu, after its shared helpers (device probe, tensor
// maps, argument checks); holds the argument checks, tensor maps and launches
// of these entry points.
#pragma once

#include "fa_decode_gemv_kernel.cuh"

namespace fa {

namespace {

// ---------------------------------------------------------------- paged decode

struct DecPlan {
    int n_splits = 1, tiles_per_split = 1, keys_per_split = 0;
    size_t part_o_bytes = 0, bytes = 0;
    size_t order_off = 0;  // tensor-core kernel: the longest-first CTA order (0: none)
};

// Units up to which the tensor-core kernel's CTAs are put in longest-first
// order by fa_decode_order_kernel (one CTA, about 2 us at this size).
constexpr long long kDecOrderMax = 1 << 18;

// The kernel that serves R rows per K/V head.  FA_DECODE_AUTO: the CUDA-core
// one (fa_decode_gemv_kernel) up to 2 rows, where the products are
// matrix-vector ones and it streams the cache faster, else the tensor-core
// one (fa_decode_kernel).  FA_DECODE_TENSOR_CORES / FA_DECODE_CUDA_CORES
// force one; the CUDA-core kernel takes at most 2 rows.
constexpr int kDecMma = 0;
constexpr int kDecGemv = 1;
constexpr int kGemvMaxRows = 2;

fa_status decode_path(int R, int choice, int *path) {
    if (choice == FA_DECODE_TENSOR_CORES) {
        *path = kDecMma;
    } else if (choice == FA_DECODE_CUDA_CORES) {
        if (R > kGemvMaxRows) return FA_ERR_UNSUPPORTED;
        *path = kDecGemv;
    } else if (choice == FA_DECODE_AUTO) {
        *path = R <= kGemvMaxRows ? kDecGemv : kDecMma;
    } else {
        return FA_ERR_UNSUPPORTED;
    }
    return FA_OK;
}

fa_status check_dec_sizes(int B, int H, int Hkv, int Sq, int d, int block_size, int max_blocks,
                          int num_blocks, int max_seq_len, int mask_kind, int dtype) {
    if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_UNSUPPORTED;
    if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    if (mask_kind != FA_MASK_NONE && mask_kind != FA_MASK_CAUSAL) return FA_ERR_UNSUPPORTED;
    if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128)
        return FA_ERR_UNSUPPORTED;
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || Sq < 1) return FA_ERR_INVALID_ARG;
    if ((long long)(H / Hkv) * Sq > 128) return FA_ERR_UNSUPPORTED;  // packed rows of one K/V head
    if (max_blocks < 1 || num_blocks < 1 || max_seq_len < Sq ||
        (long long)max_seq_len > (long long)max_blocks * block_size)
        return FA_ERR_INVALID_ARG;
    if ((long long)B * H * Sq > 0x7fffffffLL / 2 || (long long)B * max_blocks > 0x7fffffffLL)
        return FA_ERR_INVALID_ARG;
    return FA_OK;
}

// Key ranges per (request, K/V head).  Tensor-core kernel (one CTA per SM):
// enough splits that about two CTAs per SM are in flight, never more than the
// longest request has 128-key tiles.  CUDA-core kernel (two CTAs per SM):
// about eight CTAs per SM over the grid, in whole stages of 8192 / d keys.
DecPlan plan_decode(int B, int H, int Hkv, int Sq, int d, int max_seq_len, int num_sms, int path) {
    DecPlan pl;
    const int bn = path == kDecGemv ? 8192 / d : d == 256 ? DecCfg<256>::BN : DecCfg<128>::BN;
    const long long tiles = (max_seq_len + bn - 1) / bn;
    const long long base = (long long)B * Hkv;
    const long long want = (path == kDecGemv ? 8LL : 2LL) * num_sms;
    long long n = (want + base - 1) / base;
    n = std::max(1LL, std::min(n, tiles));
    const long long per = (tiles + n - 1) / n;
    pl.tiles_per_split = (int)per;
    pl.keys_per_split = (int)(per * bn);
    pl.n_splits = (int)((tiles + per - 1) / per);
    const size_t rows = (size_t)B * H * Sq;
    pl.part_o_bytes = ((size_t)pl.n_splits * rows * d * 4 + 255) / 256 * 256;
    pl.bytes = pl.part_o_bytes + (size_t)pl.n_splits * rows * 4;
    const long long units = base * pl.n_splits;
    if (path == kDecMma && units <= kDecOrderMax) {
        pl.order_off = (pl.bytes + 255) / 256 * 256;
        pl.bytes = pl.order_off + (size_t)units * 4;
    }
    return pl;
}

template <int D, bool kFP16>
fa_status launch_decode(const DecParams &p, void *o, float *lse, DeviceInfo &info, cudaStream_t stream) {
    using C = DecCfg<D>;
    auto kern = fa_decode_kernel<D, kFP16>;
    const int slot = (D == 256 ? 4 : D == 128 ? 2 : 0) + (kFP16 ? 1 : 0);
    const int smem = std::max(C::SMEM_BYTES, kBwdMinSmem);  // one CTA (and its 512 TMEM columns) per SM
    if (set_smem(kern, smem, info.attr_dec[slot]) != FA_OK) return FA_ERR_CUDA;
    const long long grid = (long long)p.B * p.Hkv * p.n_splits;
    if (p.order) {
        fa_decode_order_kernel<C::BN><<<1, 1024, 0, stream>>>(p.seq_lens, p.B, p.Hkv, p.Sq, p.max_seq_len,
                                                              p.n_splits, p.tiles_per_split,
                                                              const_cast<int *>(p.order));
        if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    }
    kern<<<(unsigned)grid, C::NUM_THREADS, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    const int rows = p.B * p.H * p.Sq;
    fa_decode_combine_kernel<D, kFP16><<<(rows + 7) / 8, 256, 0, stream>>>(p.part_o, p.part_lse, o, lse,
                                                                          rows, p.n_splits);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

template <int D, bool kFP16, int RT>
fa_status launch_gemv_rt(const GemvParams &p, void *o, float *lse, DeviceInfo &info, cudaStream_t stream) {
    using C = GemvCfg<D>;
    auto kern = fa_decode_gemv_kernel<D, kFP16, RT>;
    const int slot = ((D == 256 ? 2 : D == 128 ? 1 : 0) * 2 + (kFP16 ? 1 : 0)) * 2 + (RT - 1);
    if (set_smem(kern, C::SMEM_BYTES, info.attr_gemv[slot]) != FA_OK) return FA_ERR_CUDA;
    const long long grid = (long long)p.B * p.Hkv * p.n_splits;
    kern<<<(unsigned)grid, C::NUM_THREADS, C::SMEM_BYTES, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    const int rows = p.B * p.H * p.Sq;
    fa_decode_combine_kernel<D, kFP16><<<(rows + 7) / 8, 256, 0, stream>>>(p.part_o, p.part_lse, o, lse,
                                                                          rows, p.n_splits);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

template <int D, bool kFP16>
fa_status launch_gemv(const GemvParams &p, void *o, float *lse, DeviceInfo &info, cudaStream_t stream) {
    if (p.R == 1) return launch_gemv_rt<D, kFP16, 1>(p, o, lse, info, stream);
    return launch_gemv_rt<D, kFP16, 2>(p, o, lse, info, stream);
}

fa_status decode_impl(const void *q, const void *k_cache, const void *v_cache, const int *block_table,
                      const int *seq_lens, void *o, float *lse, void *workspace, size_t workspace_bytes,
                      int B, int H, int Hkv, int Sq, int d, int block_size, int max_blocks,
                      int num_blocks, int max_seq_len, float scale, int mask_kind, int dtype,
                      int kernel, cudaStream_t stream) {
    fa_status st = check_dec_sizes(B, H, Hkv, Sq, d, block_size, max_blocks, num_blocks, max_seq_len,
                                   mask_kind, dtype);
    if (st != FA_OK) return st;
    if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !lse || !workspace)
        return FA_ERR_INVALID_ARG;
    const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
                          reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(o);
    const uintptr_t a4 = reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(block_table) |
                         reinterpret_cast<uintptr_t>(seq_lens);
    if ((a16 & 15u) || (a4 & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FA_ERR_MISALIGNED;
    int path = kDecMma;
    st = decode_path((H / Hkv) * Sq, kernel, &path);
    if (st != FA_OK) return st;
    int dev = 0;
    DeviceInfo *info = nullptr;
    st = device_info(&dev, &info);
    if (st != FA_OK) return st;
    const DecPlan pl = plan_decode(B, H, Hkv, Sq, d, max_seq_len, info->num_sms, path);
    if (workspace_bytes < pl.bytes) return FA_ERR_INVALID_ARG;
    const size_t rows = (size_t)B * H * Sq;
    const size_t qo = rows * d * 2, cache = (size_t)num_blocks * Hkv * block_size * d * 2;
    const void *ins[5] = {q, k_cache, v_cache, block_table, seq_lens};
    const size_t in_bytes[5] = {qo, cache, cache, (size_t)B * max_blocks * 4, (size_t)B * 4};
    void *outs[3] = {o, lse, workspace};
    const size_t out_bytes[3] = {qo, rows * 4, pl.bytes};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 5; ++b)
            if (overlaps(outs[a], out_bytes[a], ins[b], in_bytes[b])) return FA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 3; ++b)
            if (overlaps(outs[a], out_bytes[a], outs[b], out_bytes[b])) return FA_ERR_INVALID_ARG;
    }

    const bool fp16 = dtype == FA_DTYPE_FP16;
    if (log_enabled())
        std::fprintf(stderr, "[fa] fa_decode_paged %s d=%d B=%d H=%d Hkv=%d Sq=%d bs=%d max_len=%d splits=%d x %d keys\n",
                     path == kDecGemv ? "gemv" : "mma", d, B, H, Hkv, Sq, block_size, max_seq_len, pl.n_splits,
                     pl.keys_per_split);
    if (path == kDecGemv) {
        GemvParams g;
        std::memset(&g, 0, sizeof(g));
        g.q = q;
        g.k_cache = k_cache;
        g.v_cache = v_cache;
        g.block_table = block_table;
        g.seq_lens = seq_lens;
        g.part_o = static_cast<float *>(workspace);
        g.part_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + pl.part_o_bytes);
        g.B = B;
        g.H = H;
        g.Hkv = Hkv;
        g.kv_group = H / Hkv;
        g.Sq = Sq;
        g.R = g.kv_group * Sq;
        g.bs = block_size;
        g.max_blocks = max_blocks;
        g.num_blocks = num_blocks;
        g.max_seq_len = max_seq_len;
        g.mask_kind = mask_kind;
        g.n_splits = pl.n_splits;
        g.keys_per_split = pl.keys_per_split;
        g.scale_log2 = std::fmax((float)((double)scale * 1.4426950408889634), FLT_MIN);
        g.wait_limit_ns = fa::kWaitLimitNs;
        if (const uint64_t ns = debug_stall_ns()) {
            g.stall_test = 1;
            g.wait_limit_ns = ns;
        }
        if (d == 64)
            return fp16 ? launch_gemv<64, true>(g, o, lse, *info, stream)
                        : launch_gemv<64, false>(g, o, lse, *info, stream);
        if (d == 256)
            return fp16 ? launch_gemv<256, true>(g, o, lse, *info, stream)
                        : launch_gemv<256, false>(g, o, lse, *info, stream);
        return fp16 ? launch_gemv<128, true>(g, o, lse, *info, stream)
                    : launch_gemv<128, false>(g, o, lse, *info, stream);
    }
    const int bn_tile = d == 256 ? DecCfg<256>::BN : DecCfg<128>::BN;
    DecParams p;
    std::memset(&p, 0, sizeof(p));
    if (!make_map(&p.tm_q, q, d, (int)rows, 1, 1, 128, fp16) ||
        !make_map(&p.tm_k, k_cache, d, block_size, Hkv, num_blocks, std::min(block_size, bn_tile), fp16) ||
        !make_map(&p.tm_v, v_cache, d, block_size, Hkv, num_blocks, std::min(block_size, bn_tile), fp16))
        return FA_ERR_CUDA;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.part_o = static_cast<float *>(workspace);
    p.part_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + pl.part_o_bytes);
    p.order = pl.order_off ? reinterpret_cast<const int *>(static_cast<uint8_t *>(workspace) + pl.order_off)
                           : nullptr;
    p.B = B;
    p.H = H;
    p.Hkv = Hkv;
    p.kv_group = H / Hkv;
    p.Sq = Sq;
    p.R = p.kv_group * Sq;
    p.bs = block_size;
    p.max_blocks = max_blocks;
    p.max_seq_len = max_seq_len;
    p.mask_kind = mask_kind;
    p.n_splits = pl.n_splits;
    p.tiles_per_split = pl.tiles_per_split;
    p.scale_log2 = std::fmax((float)((double)scale * 1.4426950408889634), FLT_MIN);
    p.wait_limit_ns = fa::kWaitLimitNs;
    if (const uint64_t ns = debug_stall_ns()) {
        p.stall_test = 1;
        p.wait_limit_ns = ns;
    }
    if (d == 64)
        return fp16 ? launch_decode<64, true>(p, o, lse, *info, stream)
                    : launch_decode<64, false>(p, o, lse, *info, stream);
    if (d == 256)
        return fp16 ? launch_decode<256, true>(p, o, lse, *info, stream)
                    : launch_decode<256, false>(p, o, lse, *info, stream);
    return fp16 ? launch_decode<128, true>(p, o, lse, *info, stream)
                : launch_decode<128, false>(p, o, lse, *info, stream);
}


}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_decode_paged(const void *q, const void *k_cache, const void *v_cache,
                          const int *block_table, const int *seq_lens, void *o, float *lse,
                          void *workspace, size_t workspace_bytes, int B, int H, int H_kv, int Sq,
                          int d, int block_size, int max_blocks, int num_blocks, int max_seq_len,
                          float scale, int mask_kind, int dtype, int kernel, fa_stream_t stream) {
    return fa::decode_impl(q, k_cache, v_cache, block_table, seq_lens, o, lse, workspace,
                           workspace_bytes, B, H, H_kv, Sq, d, block_size, max_blocks, num_blocks,
                           max_seq_len, scale, mask_kind, dtype, kernel,
                           reinterpret_cast<cudaStream_t>(stream));
}

fa_status fa_decode_workspace_query(int B, int H, int H_kv, int Sq, int d, int block_size,
                                    int max_blocks, int num_blocks, int max_seq_len, int mask_kind,
                                    int dtype, int kernel, size_t *bytes) {
    if (!bytes) return FA_ERR_INVALID_ARG;
    *bytes = 0;
    fa_status st = fa::check_dec_sizes(B, H, H_kv, Sq, d, block_size, max_blocks, num_blocks,
                                       max_seq_len, mask_kind, dtype);
    if (st != FA_OK) return st;
    int path = fa::kDecMma;
    st = fa::decode_path((H / H_kv) * Sq, kernel, &path);
    if (st != FA_OK) return st;
    int dev = 0;
    fa::DeviceInfo *info = nullptr;
    st = fa::device_info(&dev, &info);
    if (st != FA_OK) return st;
    *bytes = fa::plan_decode(B, H, H_kv, Sq, d, max_seq_len, info->num_sms, path).bytes;
    return FA_OK;
}

}  // extern "C"
