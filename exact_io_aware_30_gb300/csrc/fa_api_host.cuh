// fa_api_host.cuh -- host side of fa_fwd_host and fa_fwd_host_workspace_query
// (included by fa_api.cu: one translation unit).
//
// The forward end to end from host memory: Q, K, V are copied into a device
// workspace the caller provides, the fused forward runs there, and O and lse
// are copied back.  The problem is cut into chunks of whole K/V heads (with
// the query heads that read them), and the chunks overlap: a copy-in stream
// moves chunk c+1's Q, K, V while chunk c's forward runs and a copy-out
// stream returns chunk c-1's O and lse.  The forwards go round-robin to
// kHostComputeStreams streams: a chunk of one or two heads has fewer query
// tiles than the GPU has SMs, and the next chunk's forward fills the SMs
// its predecessor leaves idle.  The time of a call then approaches the
// largest of the three totals rather than their sum.  Chunk c is an
// ordinary forward with B = 1: the flattened
// (batch, K/V head) pairs of a chunk are consecutive in every tensor, and
// query head (b, h) reads K/V pair (b * H + h) / (H / H_kv) of the flattened
// numbering, so the chunk's local heads keep their grouping.

namespace fa {
namespace {

// Chunks: the first chunk's copy-in and the last chunk's kernel and copy-out
// are not overlapped, so more chunks shorten that fill and drain, but every
// chunk adds five copies whose fixed costs add up: on GB300 8 chunks of at
// least 8 MB measured best (16 and 32 were 6 and 22 % slower on the causal
// 8k workload, 4 about 3 %).
constexpr int kHostMaxChunks = 8;
constexpr size_t kHostMinChunkBytes = 8u << 20;  // inputs per chunk worth a separate copy
constexpr int kHostComputeStreams = 4;

struct HostStreams {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaStream_t cmp[kHostComputeStreams] = {};
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t copied[kHostMaxChunks] = {};
    cudaEvent_t computed[kHostMaxChunks] = {};
};

HostStreams g_host[kMaxDevices];  // guarded by g_host_mutex
std::mutex g_host_mutex;          // serialises the enqueue of fa_fwd_host calls

// The copy streams and events of the current device, created by its first
// call (non-blocking streams, events without timing).
fa_status host_streams(int dev, HostStreams **hs) {
    HostStreams &h = g_host[dev];
    if (!h.ready) {
        const unsigned ef = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.start, ef) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.done, ef) == cudaSuccess;
        for (int c = 0; ok && c < kHostComputeStreams; ++c)
            ok = cudaStreamCreateWithFlags(&h.cmp[c], cudaStreamNonBlocking) == cudaSuccess;
        for (int c = 0; ok && c < kHostMaxChunks; ++c)
            ok = cudaEventCreateWithFlags(&h.copied[c], ef) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.computed[c], ef) == cudaSuccess;
        if (!ok) return FA_ERR_CUDA;  // what was created stays for the next attempt
        h.ready = true;
    }
    *hs = &h;
    return FA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace layout: Q | K | V | O | lse, each 256-byte aligned.
struct HostLayout {
    size_t q, k, v, o, lse, total;
};

HostLayout host_layout(int B, int H, int Hkv, int Sq, int Sk, int d) {
    HostLayout L;
    const size_t qo = (size_t)B * H * Sq * d * 2, kv = (size_t)B * Hkv * Sk * d * 2;
    L.q = 0;
    L.k = L.q + round256(qo);
    L.v = L.k + round256(kv);
    L.o = L.v + round256(kv);
    L.lse = L.o + round256(qo);
    L.total = L.lse + round256((size_t)B * H * Sq * 4);
    return L;
}

// Chunks of consecutive (batch, K/V head) pairs: as many as keep at least
// kHostMinChunkBytes of input each, at most kHostMaxChunks.  Pairs are spread
// in proportion to weights 1, 2, ..., 2, 1 (host_chunk_start): the first
// chunk's copy-in and the last chunk's forward and copy-out are the parts
// nothing overlaps, and halving those two chunks measured about 1 % faster
// end to end on every workload.
int host_chunks(long long pairs, size_t in_bytes) {
    long long n = (long long)(in_bytes / kHostMinChunkBytes);
    if (n > kHostMaxChunks) n = kHostMaxChunks;
    if (n > pairs) n = pairs;
    return n < 1 ? 1 : (int)n;
}

// Pairs before chunk c of n: pairs * (weights of chunks 0 .. c-1) / (all weights).
long long host_chunk_start(long long pairs, int c, int n) {
    auto weight_before = [n](int upto) {
        long long w = 0;
        for (int i = 0; i < upto; ++i) w += (n > 2 && (i == 0 || i == n - 1)) ? 1 : 2;
        return w;
    };
    return pairs * weight_before(c) / weight_before(n);
}

bool is_device_memory(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // unregistered host memory may report an error on older drivers
        return false;
    }
    return a.type == cudaMemoryTypeDevice;
}

fa_status fwd_host_impl(const void *q_h, const void *k_h, const void *v_h, void *o_h,
                        float *lse_h, void *ws, size_t ws_bytes, int B, int H, int Hkv, int Sq,
                        int Sk, int d, float scale, int mask_kind, int window, int dtype,
                        cudaStream_t stream) {
    fa_status st = check_sizes(B, H, Sq, Sk, d, mask_kind, window, dtype);
    if (st != FA_OK) return st;
    if (Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
    if (Sq == 0) return FA_OK;
    if (!q_h || !k_h || !v_h || !o_h || !lse_h || !ws) return FA_ERR_INVALID_ARG;
    const HostLayout L = host_layout(B, H, Hkv, Sq, Sk, d);
    if (ws_bytes < L.total) return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return FA_ERR_MISALIGNED;
    if (is_device_memory(q_h) || is_device_memory(k_h) || is_device_memory(v_h) ||
        is_device_memory(o_h) || is_device_memory(lse_h))
        return FA_ERR_INVALID_ARG;  // device tensors go to fa_fwd / fa_fwd_gqa
    int dev = 0;
    DeviceInfo *info = nullptr;
    st = device_info(&dev, &info);
    if (st != FA_OK) return st;

    const int G = H / Hkv;
    const long long pairs = (long long)B * Hkv;
    const size_t q_pair = (size_t)G * Sq * d * 2, kv_pair = (size_t)Sk * d * 2;
    const size_t lse_pair = (size_t)G * Sq * 4;
    const int n_chunks = host_chunks(pairs, (size_t)pairs * (q_pair + 2 * kv_pair));
    char *wsb = static_cast<char *>(ws);

    std::lock_guard<std::mutex> lock(g_host_mutex);
    HostStreams *hs = nullptr;
    st = host_streams(dev, &hs);
    if (st != FA_OK) return st;
    // The copies may start once the caller's earlier work (which may still
    // read or write the workspace) is done.
    if (cudaEventRecord(hs->start, stream) != cudaSuccess ||
        cudaStreamWaitEvent(hs->in, hs->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hs->out, hs->start, 0) != cudaSuccess)
        return FA_ERR_CUDA;
    for (int c = 0; c < n_chunks; ++c) {
        const long long p0 = host_chunk_start(pairs, c, n_chunks);
        const long long np = host_chunk_start(pairs, c + 1, n_chunks) - p0;
        if (np == 0) continue;  // few pairs: a half-weight chunk can be empty
        const size_t qoff = (size_t)p0 * q_pair, kvoff = (size_t)p0 * kv_pair;
        const size_t loff = (size_t)p0 * lse_pair;
        const size_t qn = (size_t)np * q_pair, kvn = (size_t)np * kv_pair, ln = (size_t)np * lse_pair;
        if (cudaMemcpyAsync(wsb + L.q + qoff, static_cast<const char *>(q_h) + qoff, qn,
                            cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
            cudaMemcpyAsync(wsb + L.k + kvoff, static_cast<const char *>(k_h) + kvoff, kvn,
                            cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
            cudaMemcpyAsync(wsb + L.v + kvoff, static_cast<const char *>(v_h) + kvoff, kvn,
                            cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
            cudaEventRecord(hs->copied[c], hs->in) != cudaSuccess)
            return FA_ERR_CUDA;
        // (the copy-in stream waited for the caller's earlier work, so the
        // compute streams inherit that through copied[c])
        cudaStream_t cs = hs->cmp[c % kHostComputeStreams];
        if (cudaStreamWaitEvent(cs, hs->copied[c], 0) != cudaSuccess) return FA_ERR_CUDA;
        st = fwd_impl(wsb + L.q + qoff, wsb + L.k + kvoff, wsb + L.v + kvoff, wsb + L.o + qoff,
                      reinterpret_cast<float *>(wsb + L.lse + loff), 1, (int)(np * G), (int)np,
                      Sq, Sk, d, scale, mask_kind, window, dtype, cs);
        if (st != FA_OK) return st;
        if (cudaEventRecord(hs->computed[c], cs) != cudaSuccess ||
            cudaStreamWaitEvent(hs->out, hs->computed[c], 0) != cudaSuccess ||
            cudaMemcpyAsync(static_cast<char *>(o_h) + qoff, wsb + L.o + qoff, qn,
                            cudaMemcpyDeviceToHost, hs->out) != cudaSuccess ||
            cudaMemcpyAsync(reinterpret_cast<char *>(lse_h) + loff, wsb + L.lse + loff, ln,
                            cudaMemcpyDeviceToHost, hs->out) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    // The caller's stream reaches its next work only once O and lse are on
    // the host (every forward finished before its chunk's copy-out).
    if (cudaEventRecord(hs->done, hs->out) != cudaSuccess ||
        cudaStreamWaitEvent(stream, hs->done, 0) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_fwd_host_workspace_query(int B, int H, int H_kv, int Sq, int Sk, int d,
                                      int mask_kind, int window, int dtype, size_t *bytes) {
    if (!bytes) return FA_ERR_INVALID_ARG;
    *bytes = 0;
    fa_status st = fa::check_sizes(B, H, Sq, Sk, d, mask_kind, window, dtype);
    if (st != FA_OK) return st;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    int dev = 0;
    fa::DeviceInfo *info = nullptr;
    st = fa::device_info(&dev, &info);
    if (st != FA_OK) return st;
    *bytes = Sq == 0 ? 0 : fa::host_layout(B, H, H_kv, Sq, Sk, d).total;
    return FA_OK;
}

fa_status fa_fwd_host(const void *q_host, const void *k_host, const void *v_host, void *o_host,
                      float *lse_host, void *workspace, size_t workspace_bytes, int B, int H,
                      int H_kv, int Sq, int Sk, int d, float scale, int mask_kind, int window,
                      int dtype, fa_stream_t stream) {
    return fa::fwd_host_impl(q_host, k_host, v_host, o_host, lse_host, workspace,
                             workspace_bytes, B, H, H_kv, Sq, Sk, d, scale, mask_kind, window,
                             dtype, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
