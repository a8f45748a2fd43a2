/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact attention forward library.
 *
 * The operation ("FlashAttention: IO-aware attention kernels", table "What
 * goes in, what comes out"; "FlashAttention: Why Tiling Attention Makes
 * Transformers Fast Without Changing the Result", section "The tiled forward
 * pass"): for every batch b and head h,
 *
 *     O   = softmax(scale * Q K^T  restricted to visible keys) V
 *     lse = per-row natural-log sum of exp(scale * q_i . k_j) over visible j
 *
 * computed in one fused pass: key/value tiles stream through on-chip memory
 * while each query row keeps a running max, a running sum and an
 * unnormalised accumulator; the S x S score and probability matrices are
 * never written to device memory.  The result is exact up to floating-point
 * rounding order: inputs are 16-bit, products accumulate in fp32, the
 * probabilities are rounded to the input type before the P V product, and O
 * is rounded to the input type once at the end.
 *
 * Masks (readings of the pages, which name causal and sliding-window masks
 * but not their alignment):
 *   FA_MASK_NONE            every key j < Sk is visible;
 *   FA_MASK_CAUSAL          key j visible to query i iff j <= i (top-left
 *                           aligned: query 0 sees key 0, also when Sq != Sk);
 *   FA_MASK_SLIDING_WINDOW  causal and j > i - window: `window` keys
 *                           including the diagonal.
 * A query row that sees no key (only possible with a window and Sq > Sk)
 * gets O = 0 and lse = -inf, never NaN.  Arbitrary boolean masks are not
 * supported and are rejected, never silently run another way.
 *
 * All entry points are plain C.  No entry point allocates device memory, and
 * none falls back to a slower path: an unsupported request returns an error.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t (struct CUstream_st*); NULL = legacy stream. */
typedef struct CUstream_st *fa_stream_t;

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,    /* sizes, pointers, mask/window or scale invalid  */
    FA_ERR_UNSUPPORTED = 2,    /* head dim, dtype, mask kind or GPU not supported */
    FA_ERR_MISALIGNED = 3,     /* q, k, v, o not 16-byte aligned or lse not 4    */
    FA_ERR_CUDA = 4,           /* a CUDA runtime/driver call or the launch failed */
    FA_ERR_DEVICE_TIMEOUT = 5  /* a kernel's pipeline wait ran out (device flag)  */
} fa_status;

enum { FA_MASK_NONE = 0, FA_MASK_CAUSAL = 1, FA_MASK_SLIDING_WINDOW = 2 };
enum { FA_DTYPE_BF16 = 0, FA_DTYPE_FP16 = 1 };
/* Kernel choice of fa_decode_paged / fa_decode_workspace_query. */
enum { FA_DECODE_AUTO = 0, FA_DECODE_TENSOR_CORES = 1, FA_DECODE_CUDA_CORES = 2 };

/*
 * fa_fwd -- fused attention forward, bf16 inputs and output.
 *
 *   q    device pointer, [B, H, Sq, d] bf16, contiguous row-major, 16-B aligned
 *   k, v device pointers, [B, H, Sk, d] bf16, contiguous, 16-B aligned
 *   o    device pointer, [B, H, Sq, d] bf16 output; must not overlap q, k, v
 *   lse  device pointer, [B, H, Sq] fp32 output (natural-log logsumexp of the
 *        scaled scores of each row), 4-B aligned; must not overlap the others
 *   B, H >= 1; Sk >= 1; Sq >= 0 (Sq == 0: FA_OK once the sizes, kinds and scale
 *        are valid; nothing is enqueued and the pointers are not examined)
 *   d    head dimension: 64, 128 or 256 (else FA_ERR_UNSUPPORTED)
 *   scale  multiplies Q K^T; finite and >= 0 (callers usually pass 1/sqrt(d))
 *   mask_kind  FA_MASK_NONE, FA_MASK_CAUSAL or FA_MASK_SLIDING_WINDOW
 *   window  keys per row for FA_MASK_SLIDING_WINDOW (>= 1); ignored otherwise
 *   stream  CUDA stream to enqueue on
 *
 * Ownership: every buffer belongs to the caller; the library keeps no pointer
 * after returning and allocates nothing.  The call validates its arguments
 * synchronously (nothing is enqueued on error), then enqueues one kernel
 * launch and returns; results are ready when the stream reaches that point.
 * Re-entrant: concurrent calls on different streams are independent.
 * A kernel whose internal pipeline wait exceeds its time limit (about 2 s)
 * stops early and raises a device flag read by fa_get_device_error().
 */
fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                 int B, int H, int Sq, int Sk, int d, float scale,
                 int mask_kind, int window, fa_stream_t stream);

/* fa_fwd_fp16 -- identical to fa_fwd with fp16 q, k, v and o. */
fa_status fa_fwd_fp16(const void *q, const void *k, const void *v, void *o, float *lse,
                      int B, int H, int Sq, int Sk, int d, float scale,
                      int mask_kind, int window, fa_stream_t stream);

/*
 * fa_fwd_gqa -- the same forward with grouped-query attention: K and V carry
 * H_kv heads and each run of H / H_kv consecutive query heads shares one, so
 * that query head h reads K/V head h / (H / H_kv).  (The pages name
 * grouped-query attention as a later variant of the method without defining
 * it -- "FlashAttention: Why Tiling...", section "Using it in practice"; this
 * grouping is the reading taken, the one PyTorch's enable_gqa uses.)
 * H_kv == H is fa_fwd / fa_fwd_fp16; H_kv == 1 is multi-query attention.
 *
 *   q, o  [B, H, Sq, d]; k, v [B, H_kv, Sk, d]; lse [B, H, Sq] fp32
 *   H_kv  >= 1 and dividing H, else FA_ERR_INVALID_ARG
 *   dtype FA_DTYPE_BF16 or FA_DTYPE_FP16 (q, k, v and o alike)
 * Every other argument, the ownership, the errors and the device flag are as
 * for fa_fwd; fa_workspace_query with (B, H, ...) answers for this call too
 * once H_kv divides H.  K/V tiles of a shared head are read by all of its
 * query heads from the L2, so DRAM reads of K and V shrink by H / H_kv.
 */
fa_status fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int H, int H_kv, int Sq, int Sk, int d, float scale,
                     int mask_kind, int window, int dtype, fa_stream_t stream);

/*
 * fa_bwd -- attention backward: dQ, dK, dV from Q, K, V, the forward's O and
 * lse, and dO = dLoss/dO ("FlashAttention: Why Tiling...", section "The
 * backward pass: recompute instead of storing").  Each score tile is
 * recomputed on chip from Q and K, its probabilities rebuilt from lse
 * (P = exp(scale q.k - lse)); then dV = P^T dO, dP = dO V^T, the softmax
 * Jacobian gives dS = P (dP - delta) with delta_i = dO_i . O_i, and
 * dQ = scale dS K, dK = scale dS^T Q.  No S x S matrix reaches device memory.
 * Deterministic: no atomics, the same inputs give the same bits.
 *
 *   q, o, dout  [B, H, Sq, d]; k, v [B, H_kv, Sk, d]; lse [B, H, Sq] fp32 as
 *               written by fa_fwd / fa_fwd_gqa for the same q, k, v, scale,
 *               mask and window (-inf marks a row that sees no key)
 *   dq          [B, H, Sq, d] output; dk, dv [B, H_kv, Sk, d] outputs (with
 *               shared K/V heads, summed over the query heads that read them)
 *   workspace   device scratch of at least fa_bwd_workspace_query() bytes,
 *               256-byte aligned; its contents on entry do not matter and on
 *               return are the per-row statistics of this call
 *   d           64, 128 or 256 (for 256 two CTAs share each 128-key tile,
 *               each accumulating half of the dK and dV columns)
 *   dtype       FA_DTYPE_BF16 or FA_DTYPE_FP16 for all 16-bit tensors
 *   the rest    as for fa_fwd_gqa
 * All tensors are contiguous and 16-byte aligned (lse 4-byte).  Outputs may
 * not overlap each other, the inputs or the workspace (FA_ERR_INVALID_ARG).
 * Sq == 0 sets dk and dv to zero; q, o, lse, dout, dq and the workspace are
 * then not examined.  Enqueues three kernels and returns; allocates
 * nothing.  The row statistics and dK/dV run on `stream`; dQ runs on a
 * library stream of the current device (created by the first call, never
 * destroyed), forked from `stream` after the statistics and joined back
 * before any later work on `stream`, both by events: synchronising `stream`
 * covers all three, and a stream capture on `stream` records the fork and
 * join as graph edges.  Calls may come from several host threads on several
 * streams (a lock serialises their enqueue); their dQ kernels then share the
 * library stream and run one after another.  Waits are bounded as in the
 * forward and report through fa_get_device_error().
 */
fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                 const void *dout, void *dq, void *dk, void *dv, void *workspace,
                 size_t workspace_bytes, int B, int H, int H_kv, int Sq, int Sk, int d,
                 float scale, int mask_kind, int window, int dtype, fa_stream_t stream);

/*
 * fa_bwd_noalloc -- fa_bwd for callers that cannot provide device memory:
 * the same computation and results, with the workspace taken from a fixed
 * 32 MiB array in the library's device memory instead of the caller.  The
 * pages have no counterpart to this entry point; it exists for the calling
 * convention only.
 *
 *   arguments   as for fa_bwd, without workspace and workspace_bytes
 *   limit       fa_bwd_workspace_query() bytes <= 32 MiB, i.e.
 *               B * H * ceil(Sq / 128) * 128 <= 4,194,304 query rows;
 *               larger problems return FA_ERR_INVALID_ARG (use fa_bwd)
 * The first call on a device looks up the array's device address (with that
 * device current) and should come before any stream capture: under capture
 * that lookup may fail, and the call then returns FA_ERR_CUDA having enqueued
 * nothing; a failed lookup is not remembered, so one plain call made before
 * the capture fixes it.  The address is looked up again in a new context of
 * the device (after cudaDeviceReset).  Nothing is allocated or freed by any
 * call.  Every call on a device uses the same array:
 * calls whose work overlaps in time on one device (another stream, another
 * host thread) race on it and give undefined results.
 */
fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dout, void *dq, void *dk, void *dv,
                         int B, int H, int H_kv, int Sq, int Sk, int d, float scale,
                         int mask_kind, int window, int dtype, fa_stream_t stream);

/*
 * fa_bwd_workspace_query -- workspace bytes fa_bwd needs (2 x 4 bytes per
 * query row, rows padded per head to a multiple of 128), and the status
 * fa_bwd would return for these sizes on the current device (pointer checks
 * aside).  bytes must be non-NULL; it is 0 whenever the status is not FA_OK.
 */
fa_status fa_bwd_workspace_query(int B, int H, int H_kv, int Sq, int Sk, int d, int mask_kind,
                                 int window, int dtype, size_t *bytes);

/*
 * fa_fwd_fp8 -- the fused forward with 8-bit inputs ("FlashAttention:
 * IO-aware attention kernels", section "Concept", names low-precision paths
 * as a later variant).  Q, K and V are e4m3 codes with one dequantisation
 * factor per tensor (value = code x descale); S = Q K^T and P V run on the
 * 8-bit tensor path with fp32 accumulation, the running max, sum and
 * rescaling are those of fa_fwd, P is rounded to e4m3 (weights of at most
 * 2^4, stored times 2^4) before P V, O is written as bf16 and lse (natural log of the scaled row sums) as
 * fp32.  Exact up to the rounding of P: each output element differs from the
 * exact attention of the dequantised inputs by at most about 2^-4 of
 * sum_j P_ij |v_jc|, plus its bf16 rounding.
 *
 *   q    [B, H, Sq, d] e4m3; k [B, H_kv, Sk, d] e4m3
 *   vt   V transposed, [B, H_kv, d, Sk] e4m3 (both tile products then read
 *        K-major operands); Sk a multiple of 16 (16-byte rows)
 *   o    [B, H, Sq, d] bf16; lse [B, H, Sq] fp32
 *   d    64, 128 or 256 (else FA_ERR_UNSUPPORTED)
 *   scale, q_descale, k_descale, v_descale: finite; descales > 0
 *   the rest as for fa_fwd_gqa (masks, window, H_kv grouping, errors)
 */
fa_status fa_fwd_fp8(const void *q, const void *k, const void *vt, void *o, float *lse, int B,
                     int H, int H_kv, int Sq, int Sk, int d, float scale, float q_descale,
                     float k_descale, float v_descale, int mask_kind, int window,
                     fa_stream_t stream);

/*
 * fa_decode_paged -- attention of the newest Sq rows of each request over its
 * paged K/V cache, as in decoding ("Flash attention and memory-efficient
 * attention variants", sections "A different bottleneck: the KV cache during
 * inference" and "PagedAttention: memory management borrowed from an
 * operating system").  The cache is a pool of physical blocks of block_size
 * tokens; request b's block table maps its logical block n (tokens
 * n*block_size .. (n+1)*block_size - 1) to a physical block.  Exact softmax
 * attention over the gathered tokens; each request's keys are cut into ranges
 * that run in parallel, and the partial results are merged by their lse.
 *
 *   q            [B, H, Sq, d] 16-bit: the new rows (Sq = 1 for one step)
 *   k_cache      [num_blocks, H_kv, block_size, d] 16-bit
 *   v_cache      same layout
 *   block_table  device int32 [B, max_blocks]; entries past a request's last
 *                block are not read; an entry outside [0, num_blocks) reads
 *                zeros
 *   seq_lens     device int32 [B]: cached tokens of each request, the last Sq
 *                of which are the new rows' own; must lie in
 *                [Sq, max_seq_len] (values outside are clamped into it)
 *   o, lse       [B, H, Sq, d] 16-bit and [B, H, Sq] fp32 outputs
 *   workspace    at least fa_decode_workspace_query() bytes, 256-byte aligned
 *   H_kv         K/V heads, dividing H; (H / H_kv) * Sq <= 128
 *   d            64, 128 or 256; block_size 16, 32, 64 or 128
 *   max_seq_len  host bound on seq_lens (it sizes the key ranges)
 *   mask_kind    FA_MASK_NONE (every cached token) or FA_MASK_CAUSAL: row i
 *                sits at position seq_lens[b] - Sq + i and sees tokens up to
 *                it (the reading for decoding: the new rows are the last)
 *   dtype        FA_DTYPE_BF16 or FA_DTYPE_FP16
 *   kernel       FA_DECODE_AUTO: with at most 2 rows per K/V head
 *                ((H / H_kv) * Sq <= 2) the key-range kernel runs on the CUDA
 *                cores (the products are matrix-vector ones), else on the
 *                tensor cores.  FA_DECODE_TENSOR_CORES / FA_DECODE_CUDA_CORES
 *                force one (CUDA cores: at most 2 rows, else
 *                FA_ERR_UNSUPPORTED); other values FA_ERR_UNSUPPORTED.  The
 *                two kernels split the keys differently, so pass the same
 *                choice to fa_decode_workspace_query.
 * Cache slots past a request's length may hold any values, inf and NaN
 * included: they are hidden and never reach O.  Errors and the device flag
 * are as for fa_fwd; the library allocates nothing.  Two launches: the
 * key-range kernel, then the merge.
 */
fa_status fa_decode_paged(const void *q, const void *k_cache, const void *v_cache,
                          const int *block_table, const int *seq_lens, void *o, float *lse,
                          void *workspace, size_t workspace_bytes, int B, int H, int H_kv,
                          int Sq, int d, int block_size, int max_blocks, int num_blocks,
                          int max_seq_len, float scale, int mask_kind, int dtype, int kernel,
                          fa_stream_t stream);

/*
 * fa_decode_workspace_query -- workspace bytes fa_decode_paged needs on the
 * current device with this kernel choice (partial rows of every key range:
 * (d + 1) x 4 bytes per row and range) and the status it would return for
 * these sizes.  bytes must be non-NULL; it is 0 whenever the status is not
 * FA_OK.
 */
fa_status fa_decode_workspace_query(int B, int H, int H_kv, int Sq, int d, int block_size,
                                    int max_blocks, int num_blocks, int max_seq_len,
                                    int mask_kind, int dtype, int kernel, size_t *bytes);

/*
 * fa_fwd_host -- the forward end to end from host memory: Q, K, V are
 * copied into a device workspace, the fused forward of fa_fwd_gqa runs there,
 * and O and lse are copied back to host memory.  The arithmetic and the
 * results are those of fa_fwd_gqa (the method's "what goes in, what comes
 * out" -- "FlashAttention: IO-aware attention kernels" -- with the host
 * copies around it).  The problem is cut into up to 8 chunks of whole K/V
 * heads (with the query heads that read them); chunk c+1's inputs are copied
 * in on a library stream while chunk c's forward runs on one of four library
 * compute streams (round robin, so a chunk too small to fill the GPU leaves
 * its idle SMs to the next one) and chunk c-1's outputs are copied out on a
 * further library stream, so the copies overlap the kernels and each other.
 *
 *   q_host, o_host  host pointers, [B, H, Sq, d] 16-bit (dtype)
 *   k_host, v_host  host pointers, [B, H_kv, Sk, d] 16-bit
 *   lse_host        host pointer, [B, H, Sq] fp32
 *                   Pinned (page-locked) host memory gives asynchronous
 *                   copies; pageable memory works but the copies then
 *                   serialise.  Device pointers are refused
 *                   (FA_ERR_INVALID_ARG): use fa_fwd / fa_fwd_gqa.
 *   workspace       device memory of at least fa_fwd_host_workspace_query()
 *                   bytes (Q, K, V, O and lse), 256-byte aligned; owned by
 *                   the caller; its contents on entry do not matter
 *   the rest        as for fa_fwd_gqa
 * The call returns once everything is enqueued; `stream` reaches its next
 * work only after O and lse have landed in host memory, so synchronising
 * `stream` is enough before reading them.  The host buffers and the
 * workspace must stay valid until then.  The library's copy and compute
 * streams and their events are created by the first call on a device (no
 * device memory is allocated); the enqueue of concurrent calls is
 * serialised by a lock.
 * Sq == 0: FA_OK, nothing is enqueued.  A CUDA error part way through the
 * enqueue returns FA_ERR_CUDA with the earlier chunks already enqueued.
 */
fa_status fa_fwd_host(const void *q_host, const void *k_host, const void *v_host,
                      void *o_host, float *lse_host, void *workspace, size_t workspace_bytes,
                      int B, int H, int H_kv, int Sq, int Sk, int d, float scale,
                      int mask_kind, int window, int dtype, fa_stream_t stream);

/*
 * fa_fwd_host_workspace_query -- device workspace bytes fa_fwd_host needs
 * (the 16-bit Q, K, V and O and the fp32 lse, each rounded up to 256 bytes)
 * and the status it would return for these sizes on the current device
 * (pointer checks aside).  bytes must be non-NULL; 0 unless FA_OK.
 */
fa_status fa_fwd_host_workspace_query(int B, int H, int H_kv, int Sq, int Sk, int d,
                                      int mask_kind, int window, int dtype, size_t *bytes);

/*
 * fa_workspace_query -- device scratch bytes fa_fwd needs for this problem
 * (always 0: the forward keeps every intermediate on chip, so its memory is
 * linear in the sequence length -- "FlashAttention: Why Tiling...", section
 * "The tiled forward pass").  Returns exactly the status fa_fwd would return
 * for these sizes on the current device (pointer checks aside), so it is also
 * the support probe: FA_OK means the fused kernel will run, never a fallback.
 * bytes must be non-NULL.
 */
fa_status fa_workspace_query(int B, int H, int Sq, int Sk, int d, int mask_kind,
                             int window, int dtype, size_t *bytes);

/* Human-readable name of a status code (static string, never NULL). */
const char *fa_status_string(fa_status status);

/*
 * fa_describe -- writes into buf (NUL-terminated, truncated to len) the kernel
 * and tile configuration fa_fwd selects for this head dim / mask / dtype, so
 * a caller can log which kernel ran.  FA_ERR_UNSUPPORTED if none would.
 */
fa_status fa_describe(int d, int mask_kind, int dtype, char *buf, size_t len);

/*
 * fa_get_device_error -- reads and clears the device status word of the
 * current device that kernels set when a pipeline wait times out.  The
 * caller synchronises the stream first.  FA_OK if no kernel raised it,
 * FA_ERR_DEVICE_TIMEOUT if one did, FA_ERR_CUDA if it cannot be read.
 * A kernel that times out stops its pipeline and finishes normally (its O
 * and lse are then undefined); the context stays usable.
 */
fa_status fa_get_device_error(void);

/*
 * fa_set_debug_stall_ms -- test hook for the timeout path.  With ms in
 * 1..10000, every later launch of every entry point makes its first softmax
 * (or compute-warp) wait one that nothing completes, with a limit of ms
 * instead of about 2 s: the wait runs out, the kernel winds down and raises
 * the device flag, without any fault.  0 turns the hook off (the default).
 * Process-wide; FA_ERR_INVALID_ARG outside 0..10000.
 */
fa_status fa_set_debug_stall_ms(int ms);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
