// fa_api_fp8.cuh -- host side of the 8-bit forward (fa_fwd_fp8).
// Included once, by fa_api.cu, after its shared helpers (device probe, tensor
// maps, argument checks); holds the argument checks, tensor maps and launches
// of these entry points.
#pragma once

#include "fa_fp8_kernel.cuh"

namespace fa {

namespace {

// 4-D map over a contiguous 8-bit tensor with dims {x, y, z, w} (x
// contiguous), box {bx, by, 1, 1}; rows of bx bytes with the swizzle of that
// width (128 or 64 bytes).
bool make_map8(CUtensorMap *m, const void *base, int x, int y, int z, int w, int bx, int by) {
    if (bx != 128 && bx != 64) return false;
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)x, (cuuint64_t)y, (cuuint64_t)z, (cuuint64_t)w};
    cuuint64_t strides[3] = {(cuuint64_t)x, (cuuint64_t)x * y, (cuuint64_t)x * y * z};
    cuuint32_t box[4] = {(cuuint32_t)bx, (cuuint32_t)by, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     bx == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- 8-bit forward

template <int D>
fa_status launch_fp8(Fp8Params &p, const void *q, const void *k, const void *vt, long long units,
                     DeviceInfo *info, cudaStream_t stream) {
    using C = typename Fp8Pick<D>::C;
    // Q and K in row chunks of at most 128 bytes; V^T in boxes of BN keys x d rows
    if (!make_map8(&p.tm_q, q, D, p.Sq, p.H, p.B, C::CHUNK, 128) ||
        !make_map8(&p.tm_k, k, D, p.Sk, p.Hkv, p.B, C::CHUNK, C::BN) ||
        !make_map8(&p.tm_vt, vt, p.Sk, D, p.Hkv, p.B, C::BN, D))
        return FA_ERR_CUDA;
    const int slot = D == 64 ? 0 : D == 128 ? 1 : 2;
    // Request enough shared memory that no more CTAs share an SM than their
    // tensor-memory allocations fit (two of 256 columns, or one of 512).
    const int smem = C::SMEM_BYTES > 80 * 1024 ? C::SMEM_BYTES : 80 * 1024;
    if (set_smem(fa_fwd_fp8_kernel<C>, smem, info->attr_fp8[slot]) != FA_OK) return FA_ERR_CUDA;
    fa_fwd_fp8_kernel<C><<<(unsigned)units, C::NUM_THREADS, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

fa_status fp8_impl(const void *q, const void *k, const void *vt, void *o, float *lse, int B, int H,
                   int Hkv, int Sq, int Sk, int d, float scale, float q_descale, float k_descale,
                   float v_descale, int mask_kind, int window, cudaStream_t stream) {
    if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    if (mask_kind != FA_MASK_NONE && mask_kind != FA_MASK_CAUSAL && mask_kind != FA_MASK_SLIDING_WINDOW)
        return FA_ERR_UNSUPPORTED;
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || Sk < 1 || Sq < 0) return FA_ERR_INVALID_ARG;
    if (Sk % 16 != 0) return FA_ERR_INVALID_ARG;  // rows of V^T must be 16-byte multiples
    if (mask_kind == FA_MASK_SLIDING_WINDOW && window < 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
    for (float f : {q_descale, k_descale, v_descale})
        if (!std::isfinite(f) || f <= 0.f) return FA_ERR_INVALID_ARG;
    const long long units = (long long)B * H * (((long long)Sq + 127) / 128);
    if (units > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    if (Sq == 0) return FA_OK;
    if (!q || !k || !vt || !o || !lse) return FA_ERR_INVALID_ARG;
    const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(vt) | reinterpret_cast<uintptr_t>(o);
    if ((a16 & 15u) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_MISALIGNED;
    const size_t qb = (size_t)B * H * Sq * d, kvb = (size_t)B * Hkv * Sk * d;
    const size_t ob = qb * 2, lb = (size_t)B * H * Sq * 4;
    if (overlaps(o, ob, q, qb) || overlaps(o, ob, k, kvb) || overlaps(o, ob, vt, kvb) ||
        overlaps(lse, lb, o, ob) || overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kvb) ||
        overlaps(lse, lb, vt, kvb))
        return FA_ERR_INVALID_ARG;
    int dev = 0;
    DeviceInfo *info = nullptr;
    fa_status st = device_info(&dev, &info);
    if (st != FA_OK) return st;
    Fp8Params p;
    std::memset(&p, 0, sizeof(p));
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.Hkv = Hkv;
    p.kv_group = H / Hkv;
    p.Sq = Sq;
    p.Sk = Sk;
    p.mask_kind = mask_kind;
    p.window = (mask_kind == FA_MASK_SLIDING_WINDOW) ? window : 0;
    p.c = std::fmax((float)((double)scale * q_descale * k_descale * 1.4426950408889634), FLT_MIN);
    p.o_mul = v_descale;  // the weights' factor 2^P_LOG2 cancels in O / l
    p.n_qtiles = (Sq + 127) / 128;
    p.wait_limit_ns = fa::kWaitLimitNs;
    if (const uint64_t ns = debug_stall_ns()) {
        p.stall_test = 1;
        p.wait_limit_ns = ns;
    }
    if (d == 64) return launch_fp8<64>(p, q, k, vt, units, info, stream);
    if (d == 128) return launch_fp8<128>(p, q, k, vt, units, info, stream);
    return launch_fp8<256>(p, q, k, vt, units, info, stream);
}


}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_fwd_fp8(const void *q, const void *k, const void *vt, void *o, float *lse, int B, int H,
                     int H_kv, int Sq, int Sk, int d, float scale, float q_descale,
                     float k_descale, float v_descale, int mask_kind, int window,
                     fa_stream_t stream) {
    return fa::fp8_impl(q, k, vt, o, lse, B, H, H_kv, Sq, Sk, d, scale, q_descale, k_descale,
                        v_descale, mask_kind, window, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
