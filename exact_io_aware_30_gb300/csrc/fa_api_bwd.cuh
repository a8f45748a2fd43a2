// fa_api_bwd.cuh -- host side of the backward (fa_bwd, fa_bwd_noalloc,
// fa_bwd_workspace_query).
// Included once, by fa_api.cu, after its shared helpers (device probe, tensor
// maps, argument checks); holds the argument checks, tensor maps and launches
// of these entry points.
#pragma once

#include "fa_bwd_kernel.cuh"

namespace fa {

// Fixed device workspace of fa_bwd_noalloc (32 MiB: 4,194,304 padded query
// rows of two fp32 statistics each).  Shared by every call on a device, so
// calls that overlap in time on that device race on it.
constexpr size_t kNoAllocWsBytes = (size_t)32 << 20;
static __device__ __align__(256) unsigned char g_noalloc_ws[kNoAllocWsBytes];


namespace {

// ---------------------------------------------------------------- backward

// The dQ kernel needs only the row statistics, not dK or dV, so it runs on a
// second stream beside the dK/dV kernel: launched after it, its CTAs take
// the SMs that the dK/dV kernel's last wave leaves idle.  The caller's
// stream waits for it before its next work (a fork and join of events,
// which stream capture records as graph edges).  Created by a device's
// first backward call; a lock serialises the enqueue, so the shared events
// are never interleaved.
struct BwdStreams {
    bool ready = false;
    cudaStream_t side = nullptr;
    cudaEvent_t stats = nullptr, dq_done = nullptr;
};
BwdStreams g_bwd[kMaxDevices];  // guarded by g_bwd_mutex
std::mutex g_bwd_mutex;

fa_status bwd_streams(int dev, BwdStreams **bs) {
    BwdStreams &b = g_bwd[dev];
    if (!b.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if (!b.side && cudaStreamCreateWithFlags(&b.side, cudaStreamNonBlocking) != cudaSuccess)
            return FA_ERR_CUDA;
        if (!b.stats && cudaEventCreateWithFlags(&b.stats, ef) != cudaSuccess) return FA_ERR_CUDA;
        if (!b.dq_done && cudaEventCreateWithFlags(&b.dq_done, ef) != cudaSuccess) return FA_ERR_CUDA;
        b.ready = true;
    }
    *bs = &b;
    return FA_OK;
}

size_t bwd_pad_rows(int Sq) {
    return ((size_t)Sq + kBwdPadRows - 1) / kBwdPadRows * kBwdPadRows;
}

// Workspace of the backward: lse * log2(e) and delta = dO . O per query row,
// rows padded per head to a multiple of 128 (so every 64-row slice is
// 256-byte aligned for the bulk copies).
size_t bwd_workspace_bytes(int B, int H, int Sq) {
    return 2 * (size_t)B * (size_t)H * bwd_pad_rows(Sq) * sizeof(float);
}

fa_status check_bwd_sizes(int B, int H, int Hkv, int Sq, int Sk, int d, int mask_kind, int window,
                          int dtype) {
    fa_status st = check_sizes(B, H, Sq, Sk, d, mask_kind, window, dtype);
    if (st != FA_OK) return st;
    if (Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
    const long long kv_units = (long long)B * Hkv * (((long long)Sk + 127) / 128) * (d > 128 ? 2 : 1);
    if (kv_units > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

template <int D, bool kFP16>
fa_status launch_bwd(const BwdParams &pkv, const BwdParams &pq, const void *o, const void *dout,
                     const float *lse, DeviceInfo &info, int dev, cudaStream_t stream) {
    const int slot = (D == 256 ? 4 : D == 128 ? 2 : 0) + (kFP16 ? 1 : 0);
    const long long rows = (long long)pq.B * pq.H * pq.Sq_pad;
    constexpr int RPB = 256 / (D / 8);
    fa_bwd_prep_kernel<D, kFP16><<<(unsigned)((rows + RPB - 1) / RPB), 256, 0, stream>>>(
        static_cast<const uint16_t *>(o), static_cast<const uint16_t *>(dout), lse,
        const_cast<float *>(pq.l2), const_cast<float *>(pq.delta), (long long)pq.B * pq.H, pq.Sq,
        pq.Sq_pad);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;

    auto kv = fa_bwd_dkdv_kernel<D, kFP16>;
    const int kv_smem = std::max(BwdKVCfg<D>::SMEM_BYTES, kBwdMinSmem);
    if (set_smem(kv, kv_smem, info.attr_bwd[slot]) != FA_OK) return FA_ERR_CUDA;
    auto kq = fa_bwd_dq_kernel<D, kFP16>;
    const int q_smem = std::max(BwdQCfg<D>::SMEM_BYTES, kBwdMinSmem);
    if (set_smem(kq, q_smem, info.attr_bwd[6 + slot]) != FA_OK) return FA_ERR_CUDA;

    std::lock_guard<std::mutex> lock(g_bwd_mutex);
    BwdStreams *bs = nullptr;
    if (bwd_streams(dev, &bs) != FA_OK) return FA_ERR_CUDA;
    // the statistics are ready: fork
    if (cudaEventRecord(bs->stats, stream) != cudaSuccess ||
        cudaStreamWaitEvent(bs->side, bs->stats, 0) != cudaSuccess)
        return FA_ERR_CUDA;
    kv<<<pkv.n_units, BwdKVCfg<D>::NUM_THREADS, kv_smem, stream>>>(pkv);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    kq<<<pq.n_units, BwdQCfg<D>::NUM_THREADS, q_smem, bs->side>>>(pq);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    // join: the caller's stream continues once dQ is done as well
    if (cudaEventRecord(bs->dq_done, bs->side) != cudaSuccess ||
        cudaStreamWaitEvent(stream, bs->dq_done, 0) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

fa_status bwd_impl(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dout, void *dq, void *dk, void *dv, void *workspace,
                   size_t workspace_bytes, int B, int H, int Hkv, int Sq, int Sk, int d,
                   float scale, int mask_kind, int window, int dtype, cudaStream_t stream) {
    fa_status st = check_bwd_sizes(B, H, Hkv, Sq, Sk, d, mask_kind, window, dtype);
    if (st != FA_OK) return st;
    if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) {
        // Sq == 0 still defines dK = dV = 0, so only dq, q, o, lse, dout may be absent then.
        if (Sq != 0 || !k || !v || !dk || !dv) return FA_ERR_INVALID_ARG;
    }
    const size_t need = bwd_workspace_bytes(B, H, Sq);
    if (need > 0 && (!workspace || workspace_bytes < need)) return FA_ERR_INVALID_ARG;
    const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                          reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                          reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv);
    if ((a16 & 15u) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FA_ERR_MISALIGNED;
    const size_t qo = (size_t)B * H * Sq * d * 2, kvb = (size_t)B * Hkv * Sk * d * 2;
    const size_t lb = (size_t)B * H * Sq * 4;
    // outputs may not overlap one another, the inputs or the workspace
    const void *ins[6] = {q, k, v, o, lse, dout};
    const size_t in_bytes[6] = {qo, kvb, kvb, qo, lb, qo};
    void *outs[4] = {dq, dk, dv, workspace};
    const size_t out_bytes[4] = {qo, kvb, kvb, need};
    for (int a = 0; a < 4; ++a) {
        if (!outs[a] || out_bytes[a] == 0) continue;
        for (int b = 0; b < 6; ++b)
            if (ins[b] && in_bytes[b] && overlaps(outs[a], out_bytes[a], ins[b], in_bytes[b]))
                return FA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 4; ++b)
            if (outs[b] && out_bytes[b] && overlaps(outs[a], out_bytes[a], outs[b], out_bytes[b]))
                return FA_ERR_INVALID_ARG;
    }

    int dev = 0;
    DeviceInfo *info = nullptr;
    st = device_info(&dev, &info);
    if (st != FA_OK) return st;
    if (Sq == 0) {  // no query row: every dK and dV is zero
        if (cudaMemsetAsync(dk, 0, kvb, stream) != cudaSuccess ||
            cudaMemsetAsync(dv, 0, kvb, stream) != cudaSuccess)
            return FA_ERR_CUDA;
        return FA_OK;
    }

    const bool fp16 = dtype == FA_DTYPE_FP16;
    BwdParams pkv, pq;
    std::memset(&pkv, 0, sizeof(pkv));
    if (!make_map(&pkv.tm_q, q, d, Sq, H, B, BwdKVCfg<128>::BM, fp16) ||
        !make_map(&pkv.tm_do, dout, d, Sq, H, B, BwdKVCfg<128>::BM, fp16) ||
        !make_map(&pkv.tm_k, k, d, Sk, Hkv, B, BwdKVCfg<128>::BN, fp16) ||
        !make_map(&pkv.tm_v, v, d, Sk, Hkv, B, BwdKVCfg<128>::BN, fp16))
        return FA_ERR_CUDA;
    pkv.dq = dq;
    pkv.dk = dk;
    pkv.dv = dv;
    pkv.l2 = static_cast<const float *>(workspace);
    pkv.delta = static_cast<const float *>(workspace) + (size_t)B * H * bwd_pad_rows(Sq);
    pkv.B = B;
    pkv.H = H;
    pkv.Hkv = Hkv;
    pkv.kv_group = H / Hkv;
    pkv.Sq = Sq;
    pkv.Sk = Sk;
    pkv.Sq_pad = (int)bwd_pad_rows(Sq);
    pkv.mask_kind = mask_kind;
    pkv.window = (mask_kind == FA_MASK_SLIDING_WINDOW) ? window : 0;
    // positive exponent scale, as in the forward
    pkv.scale_log2 = std::fmax((float)((double)scale * 1.4426950408889634), FLT_MIN);
    pkv.scale = scale;
    pkv.wait_limit_ns = fa::kWaitLimitNs;
    if (const uint64_t ns = debug_stall_ns()) {
        pkv.stall_test = 1;
        pkv.wait_limit_ns = ns;
    }
    pq = pkv;
    pkv.n_tiles = (Sk + 127) / 128;
    pkv.n_units = B * Hkv * pkv.n_tiles * (d > 128 ? 2 : 1);  // d = 256: two CTAs (dV, dK) per key tile
    const int q_bn = d == 256 ? BwdQCfg<256>::BN : BwdQCfg<128>::BN;
    if (!make_map(&pq.tm_q, q, d, Sq, H, B, BwdQCfg<128>::BM, fp16) ||
        !make_map(&pq.tm_do, dout, d, Sq, H, B, BwdQCfg<128>::BM, fp16) ||
        !make_map(&pq.tm_k, k, d, Sk, Hkv, B, q_bn, fp16) ||
        !make_map(&pq.tm_v, v, d, Sk, Hkv, B, q_bn, fp16))
        return FA_ERR_CUDA;
    pq.n_tiles = (Sq + 127) / 128;
    pq.n_units = B * H * pq.n_tiles;

    if (log_enabled())
        std::fprintf(stderr, "[fa] fa_bwd d=%d %s B=%d H=%d Hkv=%d Sq=%d Sk=%d dkdv_ctas=%d dq_ctas=%d\n", d,
                     fp16 ? "fp16" : "bf16", B, H, Hkv, Sq, Sk, pkv.n_units, pq.n_units);
    switch (d) {
        case 64:
            return fp16 ? launch_bwd<64, true>(pkv, pq, o, dout, lse, *info, dev, stream)
                        : launch_bwd<64, false>(pkv, pq, o, dout, lse, *info, dev, stream);
        case 128:
            return fp16 ? launch_bwd<128, true>(pkv, pq, o, dout, lse, *info, dev, stream)
                        : launch_bwd<128, false>(pkv, pq, o, dout, lse, *info, dev, stream);
        case 256:
            return fp16 ? launch_bwd<256, true>(pkv, pq, o, dout, lse, *info, dev, stream)
                        : launch_bwd<256, false>(pkv, pq, o, dout, lse, *info, dev, stream);
        default:
            return FA_ERR_UNSUPPORTED;
    }
}


}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                 const void *dout, void *dq, void *dk, void *dv, void *workspace,
                 size_t workspace_bytes, int B, int H, int H_kv, int Sq, int Sk, int d, float scale,
                 int mask_kind, int window, int dtype, fa_stream_t stream) {
    return fa::bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H, H_kv,
                        Sq, Sk, d, scale, mask_kind, window, dtype,
                        reinterpret_cast<cudaStream_t>(stream));
}

fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                         int H, int H_kv, int Sq, int Sk, int d, float scale, int mask_kind,
                         int window, int dtype, fa_stream_t stream) {
    fa_status st = fa::check_bwd_sizes(B, H, H_kv, Sq, Sk, d, mask_kind, window, dtype);
    if (st != FA_OK) return st;
    if (fa::bwd_workspace_bytes(B, H, Sq) > fa::kNoAllocWsBytes) return FA_ERR_INVALID_ARG;
    int dev = 0;
    fa::DeviceInfo *info = nullptr;
    st = fa::device_info(&dev, &info);
    if (st != FA_OK) return st;
    void *ws = nullptr;
    const unsigned long long ctx = fa::current_ctx_id();
    {
        std::lock_guard<std::mutex> lock(fa::g_mutex);
        // The first call on this device (current here) looks the array up;
        // so does the first call in a new context of the device (after a
        // cudaDeviceReset the old address is stale).  A failed lookup is not
        // cached: the next call tries again.
        if (!info->noalloc_ws || (ctx != 0 && ctx != info->noalloc_ctx)) {
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, fa::g_noalloc_ws) != cudaSuccess || !addr)
                return FA_ERR_CUDA;
            info->noalloc_ws = addr;
            info->noalloc_ctx = ctx;
        }
        ws = info->noalloc_ws;
    }
    // Nothing in the workspace has to start at zero: the row-statistics kernel
    // writes every entry the other two kernels read.
    return fa::bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, ws, fa::kNoAllocWsBytes, B, H, H_kv,
                        Sq, Sk, d, scale, mask_kind, window, dtype,
                        reinterpret_cast<cudaStream_t>(stream));
}

fa_status fa_bwd_workspace_query(int B, int H, int H_kv, int Sq, int Sk, int d, int mask_kind,
                                 int window, int dtype, size_t *bytes) {
    if (!bytes) return FA_ERR_INVALID_ARG;
    *bytes = 0;
    fa_status st = fa::check_bwd_sizes(B, H, H_kv, Sq, Sk, d, mask_kind, window, dtype);
    if (st != FA_OK) return st;
    int dev = 0;
    fa::DeviceInfo *info = nullptr;
    st = fa::device_info(&dev, &info);
    if (st == FA_OK) *bytes = fa::bwd_workspace_bytes(B, H, Sq);
    return st;
}

}  // extern "C"
