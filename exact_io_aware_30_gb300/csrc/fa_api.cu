// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument
// validation, TMA tensor-map encoding, kernel selection and launch.  This file
// holds the shared helpers and the forward (fa_fwd, fa_fwd_fp16, fa_fwd_gqa);
// the backward, paged decoding, the 8-bit forward and the forward from host
// memory are in fa_api_bwd.cuh, fa_api_decode.cuh, fa_api_fp8.cuh and
// fa_api_host.cuh, included at the end (one translation unit).
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
#include <atomic>
#include <queue>
#include <utility>
#include <vector>

#include "fa.h"
#include "fa_fwd_kernel.cuh"

namespace fa {

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int num_sms = 0;
    int l2_bytes = 0;
    bool attr_set[6] = {false, false, false, false, false, false};
    bool attr_bwd[12] = {};  // dK/dV then dQ kernels, d = 64, 128, 256 x bf16, fp16
    void *noalloc_ws = nullptr;  // device address of g_noalloc_ws in this device's context
    unsigned long long noalloc_ctx = 0;  // id of the context that address belongs to
    bool attr_dec[6] = {false, false, false, false, false, false};
    bool attr_fp8[3] = {false, false, false};  // 8-bit forward, d = 64, 128, 256
    bool attr_gemv[12] = {};  // few-row decode: d = 64, 128, 256 x bf16, fp16 x 1, 2 rows
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_probed = false;

// Test hook (fa_set_debug_stall_ms): while set to N ms, each launch's first
// softmax (or compute-warp) wait is one that nothing completes, with N ms as
// the limit of every wait, so that the bounded-wait path runs without any
// fault.  0 = off.
std::atomic<int> g_debug_stall_ms{0};

// The wait limit of the test hook in ns, 0 when the hook is off.
uint64_t debug_stall_ns() {
    const int ms = g_debug_stall_ms.load(std::memory_order_relaxed);
    return ms > 0 ? (uint64_t)ms * 1000000ull : 0;
}

// FA_LOG=1 in the environment logs each launch's configuration to stderr
// (read once, at the first call).
bool log_enabled() {
    static const bool on = [] {
        const char *e = std::getenv("FA_LOG");
        return e && e[0] && e[0] != '0';
    }();
    return on;
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

// Unique id of the calling thread's current CUDA context (0 if it cannot be
// told).  A device's context is destroyed and made anew by cudaDeviceReset;
// addresses of device symbols looked up in the old one are then stale.
unsigned long long current_ctx_id() {
    typedef CUresult (*GetCurrent)(CUcontext *);
    typedef CUresult (*GetId)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static bool probed = false;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!probed) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult qres;
            if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                                 &qres) == cudaSuccess &&
                qres == cudaDriverEntryPointSuccess)
                get_current = reinterpret_cast<GetCurrent>(fn);
            fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &qres) ==
                    cudaSuccess &&
                qres == cudaDriverEntryPointSuccess)
                get_id = reinterpret_cast<GetId>(fn);
            probed = true;
        }
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx &&
        get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
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
    if (const uint64_t ns = debug_stall_ns()) {  // test hook, off unless set
        p.stall_test = 1;
        p.wait_limit_ns = ns;
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
                  "fa_fwd_kernel<d=%d,%s> sm_103a tcgen05+TMA: BM=128 BN=%d s_buffers=%d softmax_wgs=2 "
                  "k_slots=%d v_slots=%d threads=%d smem=%d mask=%s persistent",
                  d, dtype == FA_DTYPE_FP16 ? "fp16" : "bf16", fa::bn_for(d),
                  d == 256 ? fa::Cfg<256>::NSB : d == 128 ? fa::Cfg<128>::NSB : fa::Cfg<64>::NSB,
                  fa::k_slots_for(d), fa::v_slots_for(d),
                  fa::Cfg<128>::NUM_THREADS,
                  d == 64 ? fa::Cfg<64>::SMEM_BYTES : d == 128 ? fa::Cfg<128>::SMEM_BYTES
                                                               : fa::Cfg<256>::SMEM_BYTES,
                  masks[mask_kind]);
    return FA_OK;
}

fa_status fa_set_debug_stall_ms(int ms) {
    if (ms < 0 || ms > 10000) return FA_ERR_INVALID_ARG;
    fa::g_debug_stall_ms.store(ms, std::memory_order_relaxed);
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

// The other entry points, each with its kernels: the backward, decoding over a
// paged cache, the 8-bit forward, and the forward from host memory.
#include "fa_api_bwd.cuh"
#include "fa_api_decode.cuh"
#include "fa_api_fp8.cuh"
#include "fa_api_host.cuh"
