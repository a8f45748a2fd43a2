// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument
// validation, TMA tensor-map encoding, kernel selection and launch.
//
// Validation happens before anything is enqueued and never falls back to a
// different kernel: an unsupported head dim, dtype or mask is an error
// ("FlashAttention: IO-aware attention kernels", section "Failure modes" --
// a silent fallback is the failure to avoid).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <algorithm>
#include <queue>
#include <utility>
#include <vector>

#include "fa.h"
#include "fa_fwd_kernel.cuh"
#include "fa_bwd_kernel.cuh"
#include "fa_decode_kernel.cuh"
#include "fa_fp8_kernel.cuh"

namespace fa {

// Fixed device workspace of fa_bwd_noalloc (32 MiB: 4,194,304 padded query
// rows of two fp32 statistics each).  Shared by every call on a device, so
// calls that overlap in time on that device race on it.
constexpr size_t kNoAllocWsBytes = (size_t)32 << 20;
static __device__ __align__(256) unsigned char g_noalloc_ws[kNoAllocWsBytes];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int num_sms = 0;
    int l2_bytes = 0;
    bool attr_set[6] = {false, false, false, false, false, false};
    bool attr_bwd[8] = {false, false, false, false, false, false, false, false};
    void *noalloc_ws = nullptr;  // device address of g_noalloc_ws in this device's context
    bool attr_dec[4] = {false, false, false, false};
    bool attr_fp8 = false;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_probed = false;

bool log_enabled() {
    const char *e = std::getenv("FA_LOG");
    return e && e[0] && e[0] != '0';
}

// Probe the current device once: compute capability 10.3 and SM count.
fa_status device_info(int *dev_out, DeviceInfo **info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        d.supported = (major == 10 && minor == 3);
        d.num_sms = sms;
        int l2 = 0;
        if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) == cudaSuccess) d.l2_bytes = l2;
        d.probed = true;
    }
    *dev_out = dev;
    *info = &d;
    return d.supported ? FA_OK : FA_ERR_UNSUPPORTED;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode_probed) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &qres) == cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        g_encode_probed = true;
    }
    return g_encode;
}

// 4-D map over a contiguous [B, H, S, d] 16-bit tensor: dims {d, S, H, B},
// box {64, rows, 1, 1}, 128-byte swizzle.  Rows past S read as zero, per
// head, because S is its own dimension.
bool make_map(CUtensorMap *m, const void *base, int d, int S, int H, int B, int rows, bool fp16) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t e = 2;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)d * e, (cuuint64_t)S * d * e, (cuuint64_t)H * S * d * e};
    cuuint32_t box[4] = {64, (cuuint32_t)rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                     const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D map over a contiguous 8-bit tensor with dims {x, y, z, w} (x
// contiguous), box {bx, by, 1, 1}, 128-byte swizzle.
bool make_map8(CUtensorMap *m, const void *base, int x, int y, int z, int w, int bx, int by) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)x, (cuuint64_t)y, (cuuint64_t)z, (cuuint64_t)w};
    cuuint64_t strides[3] = {(cuuint64_t)x, (cuuint64_t)x * y, (cuuint64_t)x * y * z};
    cuuint32_t box[4] = {(cuuint32_t)bx, (cuuint32_t)by, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int head_dim_index(int d) { return d == 64 ? 0 : d == 128 ? 1 : d == 256 ? 2 : -1; }

int bn_for(int d) { return d == 256 ? Cfg<256>::BN : d == 128 ? Cfg<128>::BN : Cfg<64>::BN; }
int k_slots_for(int d) { return d == 256 ? Cfg<256>::KST : d == 128 ? Cfg<128>::KST : Cfg<64>::KST; }
int v_slots_for(int d) { return d == 256 ? Cfg<256>::VST : d == 128 ? Cfg<128>::VST : Cfg<64>::VST; }

// Key tiles a query tile visits (the kernel's decode, on the host).
int unit_tiles(const Params &p, int gq, int bn) {
    const int i0 = gq * 128;
    const int row_end = i0 + 128 < p.Sq ? i0 + 128 : p.Sq;
    int key_end = p.Sk;
    if (p.mask_kind != FA_MASK_NONE) key_end = p.Sk < row_end ? p.Sk : row_end;
    int key_beg = 0;
    if (p.mask_kind == FA_MASK_SLIDING_WINDOW) key_beg = i0 - p.window + 1 > 0 ? i0 - p.window + 1 : 0;
    if (key_beg >= key_end) return 0;
    return (key_end + bn - 1) / bn - key_beg / bn;
}

// (Batch, head) pairs are scheduled in groups whose K and V -- what every
// query tile of a head re-reads -- fit in a third of the L2, so that the CTAs
// working on a group find them there: K/V then come from DRAM about once and
// DRAM traffic grows with S rather than S^2.  With grouped-query attention a
// group holds whole runs of the kv_group query heads that share a K/V head.
int heads_per_group(const Params &p, int d, int l2_bytes) {
    const int BH = p.B * p.H;
    const double kv_head = 2.0 * (double)p.Sk * d * 2.0;
    const double budget = (l2_bytes > 0 ? (double)l2_bytes : 96.0e6) / 3.0;
    const long long n_kv = (long long)(budget / kv_head);
    const long long g = (n_kv < 1 ? 1 : n_kv) * p.kv_group;
    return g > BH ? BH : (int)g;
}

// The kernel's unit numbering (decode_unit): groups of heads_per_group
// heads, longest query tiles first inside a group.  Returns the query tile.
int unit_qtile(const Params &p, int u) {
    const int BH = p.B * p.H, G = p.heads_per_group, nq = p.n_qtiles;
    const int h0 = (u / (G * nq)) * G;
    const int Gg = G < BH - h0 ? G : BH - h0;
    return nq - 1 - (u - h0 * nq) / Gg;
}

// Per-CTA unit lists: units in the numbering above are dealt in turn to the
// CTA with the least work so far (cost: key tiles plus three tiles of
// per-unit overhead), and each CTA runs its units in the order received, so
// that all CTAs work on the same group of heads at about the same time.
// Schedules are cached per shape.  Returns false (snake order) when the
// shape is too large to describe in the kernel parameters.
struct SchedKey {
    int B, H, Sq, Sk, d, mask, window, grid, G;
    bool operator==(const SchedKey &o) const {
        return B == o.B && H == o.H && Sq == o.Sq && Sk == o.Sk && d == o.d && mask == o.mask &&
               window == o.window && grid == o.grid && G == o.G;
    }
};
struct SchedEntry {
    SchedKey key;
    std::vector<uint16_t> off, ids;
};
std::vector<SchedEntry> g_sched_cache;  // guarded by g_mutex; a few recent shapes

bool build_schedule(Params &p, int d, int bn, int grid) {
    if (grid > kMaxSchedGrid || p.n_units > kMaxSchedUnits) return false;
    const SchedKey key{p.B, p.H, p.Sq, p.Sk, d, p.mask_kind, p.window, grid, p.heads_per_group};
    std::lock_guard<std::mutex> lock(g_mutex);
    const SchedEntry *hit = nullptr;
    for (const auto &e : g_sched_cache)
        if (e.key == key) hit = &e;
    if (!hit) {
        const int nq = p.n_qtiles;
        std::vector<double> cost(nq);
        for (int g = 0; g < nq; ++g) {
            const int t = unit_tiles(p, g, bn);
            cost[g] = t > 0 ? t + 3.0 : 0.5;
        }
        std::vector<std::vector<uint16_t>> lists(grid);
        using Slot = std::pair<double, int>;
        std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
        for (int c = 0; c < grid; ++c) free_at.push({0.0, c});
        for (int u = 0; u < p.n_units; ++u) {
            const Slot s = free_at.top();
            free_at.pop();
            lists[s.second].push_back((uint16_t)u);
            free_at.push({s.first + cost[unit_qtile(p, u)], s.second});
        }
        SchedEntry e;
        e.key = key;
        e.off.assign(grid + 1, 0);
        for (int c = 0; c < grid; ++c) {
            e.off[c + 1] = (uint16_t)(e.off[c] + lists[c].size());
            e.ids.insert(e.ids.end(), lists[c].begin(), lists[c].end());
        }
        if (g_sched_cache.size() >= 8) g_sched_cache.erase(g_sched_cache.begin());
        g_sched_cache.push_back(std::move(e));
        hit = &g_sched_cache.back();
    }
    std::memcpy(p.sched_off, hit->off.data(), hit->off.size() * sizeof(uint16_t));
    std::memcpy(p.sched_ids, hit->ids.data(), hit->ids.size() * sizeof(uint16_t));
    return true;
}

// Size / kind checks shared by fa_fwd and fa_workspace_query.
fa_status check_sizes(int B, int H, int Sq, int Sk, int d, int mask_kind, int window, int dtype) {
    if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_UNSUPPORTED;
    if (head_dim_index(d) < 0) return FA_ERR_UNSUPPORTED;
    if (mask_kind != FA_MASK_NONE && mask_kind != FA_MASK_CAUSAL &&
        mask_kind != FA_MASK_SLIDING_WINDOW)
        return FA_ERR_UNSUPPORTED;
    if (B < 1 || H < 1 || Sk < 1 || Sq < 0) return FA_ERR_INVALID_ARG;
    if (mask_kind == FA_MASK_SLIDING_WINDOW && window < 1) return FA_ERR_INVALID_ARG;
    const long long groups = ((long long)Sq + 127) / 128;
    if ((long long)B * H * groups > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    if ((long long)B * H > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + nb && pb < pa + na;
}

template <int D, bool kFP16>
fa_status launch(const Params &p, int num_sms, DeviceInfo &info, cudaStream_t stream) {
    using C = Cfg<D>;
    auto kern = fa_fwd_kernel<D, kFP16>;
    const int slot = head_dim_index(D) * 2 + (kFP16 ? 1 : 0);
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!info.attr_set[slot]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::SMEM_BYTES) != cudaSuccess)
                return FA_ERR_CUDA;
            info.attr_set[slot] = true;
        }
    }
    const int grid = p.n_units < num_sms ? p.n_units : num_sms;
    kern<<<grid, C::NUM_THREADS, C::SMEM_BYTES, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

fa_status fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                   int Hkv, int Sq, int Sk, int d, float scale, int mask_kind, int window,
                   int dtype, cudaStream_t stream) {
    fa_status st = check_sizes(B, H, Sq, Sk, d, mask_kind, window, dtype);
    if (st != FA_OK) return st;
    if (Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
    if (Sq == 0) return FA_OK;  // nothing to compute; empty tensors may have null pointers
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
    if ((a16 & 15u) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_MISALIGNED;
    const size_t qo_bytes = (size_t)B * H * Sq * d * 2, kv_bytes = (size_t)B * Hkv * Sk * d * 2;
    const size_t lse_bytes = (size_t)B * H * Sq * 4;
    if (overlaps(o, qo_bytes, q, qo_bytes) || overlaps(o, qo_bytes, k, kv_bytes) ||
        overlaps(o, qo_bytes, v, kv_bytes) || overlaps(lse, lse_bytes, o, qo_bytes) ||
        overlaps(lse, lse_bytes, q, qo_bytes) || overlaps(lse, lse_bytes, k, kv_bytes) ||
        overlaps(lse, lse_bytes, v, kv_bytes))
        return FA_ERR_INVALID_ARG;

    int dev = 0;
    DeviceInfo *info = nullptr;
    st = device_info(&dev, &info);
    if (st != FA_OK) return st;

    const bool fp16 = dtype == FA_DTYPE_FP16;
    const int bn = bn_for(d);
    Params p;
    std::memset(&p, 0, sizeof(p));
    if (!make_map(&p.tm_q, q, d, Sq, H, B, 128, fp16) ||
        !make_map(&p.tm_k, k, d, Sk, Hkv, B, bn, fp16) ||
        !make_map(&p.tm_v, v, d, Sk, Hkv, B, bn, fp16) ||
        (d <= 128 && !make_map(&p.tm_o, o, d, Sq, H, B, 128, fp16)))
        return FA_ERR_CUDA;
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.kv_group = H / Hkv;
    p.Sq = Sq;
    p.Sk = Sk;
    p.mask_kind = mask_kind;
    p.window = (mask_kind == FA_MASK_SLIDING_WINDOW) ? window : 0;
    // The kernel needs a positive exponent scale: a hidden key is a score of
    // -inf, whose weight 2^(-inf * c - m) is 0 only for c > 0.  scale == 0
    // (and any scale whose product underflows) runs with c = 2^-126: for every
    // score below 2^100 in magnitude, s * c - m then lies within 2^-25 of 0,
    // so each visible weight is 1 to fp32 precision -- the uniform weights
    // of a zero scale.
    p.scale_log2 = std::fmax((float)((double)scale * 1.4426950408889634), FLT_MIN);
    p.o_vec8 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
    p.wait_limit_ns = fa::kWaitLimitNs;
    // Test hook: FA_DEBUG_STALL_MS=N makes the launch's first softmax wait
    // one that nothing completes, with N ms as the wait limit, so that the
    // bounded-wait path can be exercised without any fault.
    if (const char *e = std::getenv("FA_DEBUG_STALL_MS")) {
        const long ms = std::strtol(e, nullptr, 10);
        if (ms > 0 && ms <= 10000) {
            p.stall_test = 1;
            p.wait_limit_ns = (uint64_t)ms * 1000000ull;
        }
    }
    p.n_qtiles = (Sq + 127) / 128;
    p.n_units = B * H * p.n_qtiles;
    p.heads_per_group = heads_per_group(p, d, info->l2_bytes);
    p.sched = build_schedule(p, d, bn, p.n_units < info->num_sms ? p.n_units : info->num_sms) ? 1 : 0;

    if (log_enabled()) {
        char buf[256];
        fa_describe(d, mask_kind, dtype, buf, sizeof buf);
        std::fprintf(stderr, "[fa] %s B=%d H=%d Hkv=%d Sq=%d Sk=%d units=%d grid=%d\n", buf, B, H,
                     Hkv, Sq, Sk, p.n_units, p.n_units < info->num_sms ? p.n_units : info->num_sms);
    }

    switch (d) {
        case 64:
            return fp16 ? launch<64, true>(p, info->num_sms, *info, stream)
                        : launch<64, false>(p, info->num_sms, *info, stream);
        case 128:
            return fp16 ? launch<128, true>(p, info->num_sms, *info, stream)
                        : launch<128, false>(p, info->num_sms, *info, stream);
        case 256:
            return fp16 ? launch<256, true>(p, info->num_sms, *info, stream)
                        : launch<256, false>(p, info->num_sms, *info, stream);
        default:
            return FA_ERR_UNSUPPORTED;
    }
}

// ---------------------------------------------------------------- backward

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
    if (d > 128) return FA_ERR_UNSUPPORTED;  // dK and dV accumulators: 2 x d tensor-memory columns
    const long long kv_units = (long long)B * Hkv * (((long long)Sk + 127) / 128);
    if (kv_units > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

template <typename K>
fa_status set_smem(K kern, int bytes, bool &done) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!done) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
            cudaSuccess)
            return FA_ERR_CUDA;
        done = true;
    }
    return FA_OK;
}

// Every CTA of the two backward kernels allocates all 512 tensor-memory
// columns, so they request enough shared memory to run one CTA per SM.
constexpr int kBwdMinSmem = 120 * 1024;

template <int D, bool kFP16>
fa_status launch_bwd(const BwdParams &pkv, const BwdParams &pq, const void *o, const void *dout,
                     const float *lse, DeviceInfo &info, cudaStream_t stream) {
    const int slot = (D == 128 ? 2 : 0) + (kFP16 ? 1 : 0);
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
    kv<<<pkv.n_units, BwdKVCfg<D>::NUM_THREADS, kv_smem, stream>>>(pkv);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;

    auto kq = fa_bwd_dq_kernel<D, kFP16>;
    const int q_smem = std::max(BwdQCfg<D>::SMEM_BYTES, kBwdMinSmem);
    if (set_smem(kq, q_smem, info.attr_bwd[4 + slot]) != FA_OK) return FA_ERR_CUDA;
    kq<<<pq.n_units, BwdQCfg<D>::NUM_THREADS, q_smem, stream>>>(pq);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
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
    pq = pkv;
    pkv.n_tiles = (Sk + 127) / 128;
    pkv.n_units = B * Hkv * pkv.n_tiles;
    if (!make_map(&pq.tm_q, q, d, Sq, H, B, BwdQCfg<128>::BM, fp16) ||
        !make_map(&pq.tm_do, dout, d, Sq, H, B, BwdQCfg<128>::BM, fp16) ||
        !make_map(&pq.tm_k, k, d, Sk, Hkv, B, BwdQCfg<128>::BN, fp16) ||
        !make_map(&pq.tm_v, v, d, Sk, Hkv, B, BwdQCfg<128>::BN, fp16))
        return FA_ERR_CUDA;
    pq.n_tiles = (Sq + 127) / 128;
    pq.n_units = B * H * pq.n_tiles;

    if (log_enabled())
        std::fprintf(stderr, "[fa] fa_bwd d=%d %s B=%d H=%d Hkv=%d Sq=%d Sk=%d dkdv_ctas=%d dq_ctas=%d\n", d,
                     fp16 ? "fp16" : "bf16", B, H, Hkv, Sq, Sk, pkv.n_units, pq.n_units);
    switch (d) {
        case 64:
            return fp16 ? launch_bwd<64, true>(pkv, pq, o, dout, lse, *info, stream)
                        : launch_bwd<64, false>(pkv, pq, o, dout, lse, *info, stream);
        case 128:
            return fp16 ? launch_bwd<128, true>(pkv, pq, o, dout, lse, *info, stream)
                        : launch_bwd<128, false>(pkv, pq, o, dout, lse, *info, stream);
        default:
            return FA_ERR_UNSUPPORTED;
    }
}

// ---------------------------------------------------------------- paged decode

struct DecPlan {
    int n_splits = 1, tiles_per_split = 1;
    size_t part_o_bytes = 0, bytes = 0;
};

fa_status check_dec_sizes(int B, int H, int Hkv, int Sq, int d, int block_size, int max_blocks,
                          int num_blocks, int max_seq_len, int mask_kind, int dtype) {
    if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
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

// Key ranges per (request, K/V head): enough splits that about two CTAs per
// SM are in flight, never more than the longest request has 128-key tiles.
DecPlan plan_decode(int B, int H, int Hkv, int Sq, int d, int max_seq_len, int num_sms) {
    DecPlan pl;
    const long long tiles = (max_seq_len + 127) / 128;
    const long long base = (long long)B * Hkv;
    long long n = (2LL * num_sms + base - 1) / base;
    n = std::max(1LL, std::min(n, tiles));
    const long long per = (tiles + n - 1) / n;
    pl.tiles_per_split = (int)per;
    pl.n_splits = (int)((tiles + per - 1) / per);
    const size_t rows = (size_t)B * H * Sq;
    pl.part_o_bytes = ((size_t)pl.n_splits * rows * d * 4 + 255) / 256 * 256;
    pl.bytes = pl.part_o_bytes + (size_t)pl.n_splits * rows * 4;
    return pl;
}

template <int D, bool kFP16>
fa_status launch_decode(const DecParams &p, void *o, float *lse, DeviceInfo &info, cudaStream_t stream) {
    using C = DecCfg<D>;
    auto kern = fa_decode_kernel<D, kFP16>;
    const int slot = (D == 128 ? 2 : 0) + (kFP16 ? 1 : 0);
    const int smem = std::max(C::SMEM_BYTES, kBwdMinSmem);  // one CTA (and its 512 TMEM columns) per SM
    if (set_smem(kern, smem, info.attr_dec[slot]) != FA_OK) return FA_ERR_CUDA;
    const long long grid = (long long)p.B * p.Hkv * p.n_splits;
    kern<<<(unsigned)grid, C::NUM_THREADS, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    const int rows = p.B * p.H * p.Sq;
    fa_decode_combine_kernel<D, kFP16><<<(rows + 7) / 8, 256, 0, stream>>>(p.part_o, p.part_lse, o, lse,
                                                                          rows, p.n_splits);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

fa_status decode_impl(const void *q, const void *k_cache, const void *v_cache, const int *block_table,
                      const int *seq_lens, void *o, float *lse, void *workspace, size_t workspace_bytes,
                      int B, int H, int Hkv, int Sq, int d, int block_size, int max_blocks,
                      int num_blocks, int max_seq_len, float scale, int mask_kind, int dtype,
                      cudaStream_t stream) {
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
    int dev = 0;
    DeviceInfo *info = nullptr;
    st = device_info(&dev, &info);
    if (st != FA_OK) return st;
    const DecPlan pl = plan_decode(B, H, Hkv, Sq, d, max_seq_len, info->num_sms);
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
    DecParams p;
    std::memset(&p, 0, sizeof(p));
    if (!make_map(&p.tm_q, q, d, (int)rows, 1, 1, 128, fp16) ||
        !make_map(&p.tm_k, k_cache, d, block_size, Hkv, num_blocks, block_size, fp16) ||
        !make_map(&p.tm_v, v_cache, d, block_size, Hkv, num_blocks, block_size, fp16))
        return FA_ERR_CUDA;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.part_o = static_cast<float *>(workspace);
    p.part_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + pl.part_o_bytes);
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
    if (log_enabled())
        std::fprintf(stderr, "[fa] fa_decode_paged d=%d B=%d H=%d Hkv=%d Sq=%d bs=%d max_len=%d splits=%d x %d tiles\n",
                     d, B, H, Hkv, Sq, block_size, max_seq_len, pl.n_splits, pl.tiles_per_split);
    if (d == 64)
        return fp16 ? launch_decode<64, true>(p, o, lse, *info, stream)
                    : launch_decode<64, false>(p, o, lse, *info, stream);
    return fp16 ? launch_decode<128, true>(p, o, lse, *info, stream)
                : launch_decode<128, false>(p, o, lse, *info, stream);
}

// ---------------------------------------------------------------- 8-bit forward

fa_status fp8_impl(const void *q, const void *k, const void *vt, void *o, float *lse, int B, int H,
                   int Hkv, int Sq, int Sk, int d, float scale, float q_descale, float k_descale,
                   float v_descale, int mask_kind, int window, cudaStream_t stream) {
    if (d != 128) return FA_ERR_UNSUPPORTED;
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
    if (!make_map8(&p.tm_q, q, d, Sq, H, B, d, 128) || !make_map8(&p.tm_k, k, d, Sk, Hkv, B, d, 128) ||
        !make_map8(&p.tm_vt, vt, Sk, d, Hkv, B, 128, d))
        return FA_ERR_CUDA;
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
    const int smem = Fp8Cfg::SMEM_BYTES;
    if (set_smem(fa_fwd_fp8_kernel, smem, info->attr_fp8) != FA_OK) return FA_ERR_CUDA;
    fa_fwd_fp8_kernel<<<(unsigned)units, Fp8Cfg::NUM_THREADS, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                 int Sq, int Sk, int d, float scale, int mask_kind, int window,
                 fa_stream_t stream) {
    return fa::fwd_impl(q, k, v, o, lse, B, H, H, Sq, Sk, d, scale, mask_kind, window,
                        FA_DTYPE_BF16, reinterpret_cast<cudaStream_t>(stream));
}

fa_status fa_fwd_fp16(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                      int H, int Sq, int Sk, int d, float scale, int mask_kind, int window,
                      fa_stream_t stream) {
    return fa::fwd_impl(q, k, v, o, lse, B, H, H, Sq, Sk, d, scale, mask_kind, window,
                        FA_DTYPE_FP16, reinterpret_cast<cudaStream_t>(stream));
}

fa_status fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                     int H, int H_kv, int Sq, int Sk, int d, float scale, int mask_kind,
                     int window, int dtype, fa_stream_t stream) {
    return fa::fwd_impl(q, k, v, o, lse, B, H, H_kv, Sq, Sk, d, scale, mask_kind, window, dtype,
                        reinterpret_cast<cudaStream_t>(stream));
}

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
    {
        std::lock_guard<std::mutex> lock(fa::g_mutex);
        if (!info->noalloc_ws) {
            // first call on this device (which is current here): look the array up once
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, fa::g_noalloc_ws) != cudaSuccess || !addr)
                return FA_ERR_CUDA;
            info->noalloc_ws = addr;
        }
        ws = info->noalloc_ws;
    }
    // Nothing in the workspace has to start at zero: the row-statistics kernel
    // writes every entry the other two kernels read.
    return fa::bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, ws, fa::kNoAllocWsBytes, B, H, H_kv,
                        Sq, Sk, d, scale, mask_kind, window, dtype,
                        reinterpret_cast<cudaStream_t>(stream));
}

fa_status fa_fwd_fp8(const void *q, const void *k, const void *vt, void *o, float *lse, int B, int H,
                     int H_kv, int Sq, int Sk, int d, float scale, float q_descale,
                     float k_descale, float v_descale, int mask_kind, int window,
                     fa_stream_t stream) {
    return fa::fp8_impl(q, k, vt, o, lse, B, H, H_kv, Sq, Sk, d, scale, q_descale, k_descale,
                        v_descale, mask_kind, window, reinterpret_cast<cudaStream_t>(stream));
}

fa_status fa_decode_paged(const void *q, const void *k_cache, const void *v_cache,
                          const int *block_table, const int *seq_lens, void *o, float *lse,
                          void *workspace, size_t workspace_bytes, int B, int H, int H_kv, int Sq,
                          int d, int block_size, int max_blocks, int num_blocks, int max_seq_len,
                          float scale, int mask_kind, int dtype, fa_stream_t stream) {
    return fa::decode_impl(q, k_cache, v_cache, block_table, seq_lens, o, lse, workspace,
                           workspace_bytes, B, H, H_kv, Sq, d, block_size, max_blocks, num_blocks,
                           max_seq_len, scale, mask_kind, dtype, reinterpret_cast<cudaStream_t>(stream));
}

fa_status fa_decode_workspace_query(int B, int H, int H_kv, int Sq, int d, int block_size,
                                    int max_blocks, int num_blocks, int max_seq_len, int mask_kind,
                                    int dtype, size_t *bytes) {
    if (!bytes) return FA_ERR_INVALID_ARG;
    *bytes = 0;
    fa_status st = fa::check_dec_sizes(B, H, H_kv, Sq, d, block_size, max_blocks, num_blocks,
                                       max_seq_len, mask_kind, dtype);
    if (st != FA_OK) return st;
    int dev = 0;
    fa::DeviceInfo *info = nullptr;
    st = fa::device_info(&dev, &info);
    if (st == FA_OK) *bytes = fa::plan_decode(B, H, H_kv, Sq, d, max_seq_len, info->num_sms).bytes;
    return st;
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

fa_status fa_workspace_query(int B, int H, int Sq, int Sk, int d, int mask_kind, int window,
                             int dtype, size_t *bytes) {
    if (!bytes) return FA_ERR_INVALID_ARG;
    *bytes = 0;
    fa_status st = fa::check_sizes(B, H, Sq, Sk, d, mask_kind, window, dtype);
    if (st != FA_OK) return st;
    int dev = 0;
    fa::DeviceInfo *info = nullptr;
    return fa::device_info(&dev, &info);
}

const char *fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid size, pointer, window or scale";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dim, dtype, mask kind or GPU not supported";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED: q/k/v/o need 16-byte alignment, lse 4-byte";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call or the kernel launch failed";
        case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT: a kernel pipeline wait timed out";
        default: return "FA_ERR_UNKNOWN";
    }
}

fa_status fa_describe(int d, int mask_kind, int dtype, char *buf, size_t len) {
    if (!buf || len == 0) return FA_ERR_INVALID_ARG;
    fa_status st = fa::check_sizes(1, 1, 1, 1, d, mask_kind, 1, dtype);
    if (st != FA_OK) {
        std::snprintf(buf, len, "unsupported");
        return st;
    }
    static const char *masks[] = {"none", "causal", "sliding_window"};
    std::snprintf(buf, len,
                  "fa_fwd_kernel<d=%d,%s> sm_103a tcgen05+TMA: BM=128 BN=%d s_buffers=2 softmax_wgs=2 "
                  "k_slots=%d v_slots=%d threads=%d smem=%d mask=%s persistent",
                  d, dtype == FA_DTYPE_FP16 ? "fp16" : "bf16", fa::bn_for(d), fa::k_slots_for(d), fa::v_slots_for(d),
                  fa::Cfg<128>::NUM_THREADS,
                  d == 64 ? fa::Cfg<64>::SMEM_BYTES : d == 128 ? fa::Cfg<128>::SMEM_BYTES
                                                               : fa::Cfg<256>::SMEM_BYTES,
                  masks[mask_kind]);
    return FA_OK;
}

fa_status fa_get_device_error(void) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, fa::g_fa_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    if (v == 0) return FA_OK;
    const int zero = 0;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    return FA_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
