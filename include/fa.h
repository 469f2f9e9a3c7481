/*
 * fa.h -- C ABI of libfa.so: exact scaled dot-product attention on one GB300
 * (sm_103a), forward with the online-softmax recurrence and a recompute
 * backward.
 *
 * What is computed (per batch b and head h, rows of N x d matrices):
 *   S = scale * Q K^T, masked entries -inf   ("Transformer 入门", section
 *       "flash attention": S = QK^T/sqrt(d), m = rowmax(S), l = rowsum(exp(S-m)))
 *   P = softmax(S) row by row, O = P V        ("FlashAttention" notes,
 *       "Standard Attention Implementation")
 *   LSE_i = m_i + ln(l_i), natural log, stored instead of S and P
 *       ("FlashAttention" notes, "Tiling": keep (m, l) instead of S, P)
 *   dV = P^T dO, dP = dO V^T, D_i = dO_i . O_i, dS = P o (dP - D),
 *   dQ = scale * dS K, dK = scale * dS^T Q   ("FlashAttention" notes,
 *       "Backward Pass of flashattention", with the scale's chain rule)
 * The forward never writes S or P to memory; the backward recomputes P from
 * Q, K and the saved LSE.
 *
 * Layout and types (every tensor argument):
 *   q, k, v, o, dout, dq, dk, dv : bf16, contiguous [B, H, N, d], device memory
 *   lse                          : fp32, contiguous [B, H, N], device memory
 *   block_mask                   : uint8, contiguous [nb, nb] with nb = ceil(N/128), device
 *                                  memory, shared by every (b, h); nonzero keeps
 *                                  the 128 x 128 block (query block, key block)
 *   workspace                    : device memory of at least
 *                                  fa_bwd_workspace_bytes(B, H, N, d) bytes,
 *                                  256-byte aligned; its contents on entry do
 *                                  not matter.
 * Supported: d in {64, 128}; any N >= 1 (the last 128-row tile may be
 * partial); B, H >= 1; B * H * N * d < 2^31; scale finite and > 0; pointers
 * 16-byte aligned; a device of compute capability 10.3.  Block masks: N at
 * most 131072 (1024 tiles per row).
 *
 * Masks: causal keeps key j for query i iff j <= i (equal query and key
 * lengths); key tiles that a mask removes entirely are skipped, never loaded.
 * A query row with no visible key (possible only with a block mask whose
 * diagonal block is off) gets O = 0, LSE = -inf and zero gradients.
 *
 * Ownership: the caller allocates and frees every buffer and keeps it alive
 * until the enqueued work has finished.  The library holds no pointer after
 * a call returns; its only state is one status word per device (read through
 * fa_get_device_error()) and the wait timeout.
 *
 * Asynchrony and errors: every compute call validates its arguments on the
 * host, enqueues its kernels on `stream` and returns without waiting.  A
 * negative return value (an fa_status) means nothing was enqueued, except
 * FA_ERR_LAUNCH, which reports a launch failure from the CUDA runtime.  A
 * kernel whose internal wait exceeds the wait timeout (see
 * fa_set_wait_timeout_ns) records FA_ERR_TIMEOUT in the status word and
 * returns early; its outputs are then undefined.
 *
 * Stream capture: fa_fwd, fa_fwd_blocksparse, fa_fwd_dropout, fa_bwd,
 * fa_bwd_blocksparse, fa_bwd_dropout, the three backward stages
 * (fa_bwd_preprocess, fa_bwd_main, fa_bwd_dq_convert) and fa_decode enqueue
 * only kernel launches on `stream` -- no allocation, copy or
 * synchronisation -- so they can be captured into a CUDA graph and replayed.
 * The first call on a device sets up per-device state, so make one call
 * before capturing.  fa_get_device_error synchronises and the host-streamed
 * calls (fa_fwd_bwd_host, fa_fwd_host) use the library's own streams:
 * neither belongs in a capture.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the C ABI are exported from libfa.so; everything else is hidden. */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *fa_stream_t;

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID = -1,     /* bad argument: null pointer, size, alignment, scale */
  FA_ERR_UNSUPPORTED = -2, /* valid but not built: head dim other than 64/128, or a block mask longer than 1024 tiles */
  FA_ERR_ARCH = -3,        /* current device is not compute capability 10.3 */
  FA_ERR_LAUNCH = -4,      /* the CUDA runtime refused a launch or attribute call */
  FA_ERR_TIMEOUT = -5,     /* a kernel wait ran past the wait timeout (device status) */
  FA_ERR_CUDA = -6,        /* another CUDA runtime error (device query, descriptor) */
  FA_ERR_SCRATCH = -7,     /* fa_bwd_noalloc: the problem needs more than its static scratch */
  FA_ERR_BOUNDS = -8       /* debug build (libfa_debug.so) only: a device index check failed;
                              the access was skipped (reported by fa_get_device_error) */
} fa_status;

/* Library version, major * 10000 + minor * 100 + patch. */
FA_API int fa_version(void);

/* Human-readable name of an fa_status value; never NULL. */
FA_API const char *fa_status_string(int status);

/*
 * Forward: O and LSE from Q, K, V.  causal != 0 applies the lower-triangular
 * mask.  Cited: "FlashAttention" notes, "Tiling" and "Correctness"
 * (Theorem 1: the tiled recurrence yields softmax(S) V exactly);
 * "Как работает FlashAttention математически", sections 3-4 (online softmax
 * and output correction).
 */
FA_API int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int H, int N, int d, float scale, int causal, fa_stream_t stream);

/*
 * Forward with a 128 x 128 block mask (block-sparse attention, "FlashAttention"
 * notes, "Block-sparse Flashattention"): blocks whose mask byte is 0 are
 * skipped and add nothing to m, l or O.  causal != 0 also applies the causal
 * mask (key j visible to query i iff j <= i and the block is kept): with the
 * window masks below this is causal sliding-window or dilated attention.
 */
FA_API int fa_fwd_blocksparse(const void *q, const void *k, const void *v, void *o, float *lse,
                       const uint8_t *block_mask, int B, int H, int N, int d, float scale,
                       int causal, fa_stream_t stream);

/*
 * Bytes of device workspace that fa_bwd needs: an fp32 dQ accumulator
 * [B, H, N, d], then two fp32 vectors [B, H, npad] (npad = N rounded up to a
 * multiple of 128) holding -D and -LSE * log2(e), each region 256-byte
 * aligned.  Returns 0 when the sizes are invalid.
 */
FA_API size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward: dQ, dK, dV from Q, K, V, the forward's O and LSE, and dO.
 * Runs the three stages below in order on `stream`.  Cited: "FlashAttention"
 * notes, "Backward Pass of flashattention" (recompute P from the saved
 * statistics; D_i = do_i . o_i; masks are regenerated, not stored).
 */
FA_API int fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
           const float *lse, void *dq, void *dk, void *dv, void *workspace,
           int B, int H, int N, int d, float scale, int causal, fa_stream_t stream);

/* Backward with the block mask (and causal flag) of fa_fwd_blocksparse. */
FA_API int fa_bwd_blocksparse(const void *q, const void *k, const void *v, const void *o,
                       const void *dout, const float *lse, const uint8_t *block_mask,
                       void *dq, void *dk, void *dv, void *workspace,
                       int B, int H, int N, int d, float scale, int causal, fa_stream_t stream);

/*
 * Backward stage 1 of 3: D_i = sum_c dO[i,c] O[i,c] in fp32, stored as -D_i
 * next to -LSE_i * log2(e) (the form stage 2 consumes; zeros for the padding
 * rows past N), and the workspace's dQ accumulator set to zero.  lse is the
 * forward's output, read only here.
 */
FA_API int fa_bwd_preprocess(const void *o, const void *dout, const float *lse, void *workspace,
                      int B, int H, int N, int d, fa_stream_t stream);

/*
 * Backward stage 2 of 3: per 128-key tile, recompute P from Q, K and the
 * workspace's LSE, accumulate dK, dV (written as bf16) and add dS K into the
 * workspace's dQ accumulator.  Needs the workspace as stage 1 left it.
 * mask_kind: 0 none, 1 causal, 2 block (block_mask required), 3 causal and
 * block.  dropout_p, seed: as for fa_bwd_dropout (0 for none).
 */
FA_API int fa_bwd_main(const void *q, const void *k, const void *v, const void *dout,
                const uint8_t *block_mask, void *dk, void *dv,
                void *workspace, int B, int H, int N, int d, float scale, int mask_kind,
                float dropout_p, unsigned long long seed, fa_stream_t stream);

/* Backward stage 3 of 3: dQ = bf16(scale * accumulator). */
FA_API int fa_bwd_dq_convert(const void *workspace, void *dq, int B, int H, int N, int d,
                      float scale, fa_stream_t stream);

/*
 * Attention with dropout on the probabilities, the masks regenerated in the
 * backward instead of stored ("Как работает FlashAttention математически",
 * section 5: only the statistics and the random masks' generator state are
 * kept; "FlashAttention" notes, "Backward Pass of flashattention": masks are
 * regenerated).  O = (P o Z) V / (1 - p'), with P the softmax (LSE is P's),
 * Z the keep mask and p' the effective drop probability.
 *
 * Generator (the pages name none): Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11), key = seed (low
 * word first), counter = (j / 4, i / 4, h, b) for query i, key j; pair (i, j)
 * takes byte j % 4 of output word i % 4 and is kept iff that byte >= t with
 * t = round(256 dropout_p) (at most 255), so p' = t / 256 and kept values
 * are scaled by 256 / (256 - t).  The same (seed, dropout_p) in the forward
 * and the backward give the same mask.
 *
 * block_mask may be NULL (no block mask); causal as for fa_fwd.  dropout_p in
 * [0, 1), else FA_ERR_INVALID.  Everything else as for fa_fwd / fa_bwd.
 */
/*
 * The drop probability p' = round(256 dropout_p) / 256 (t at most 255) that
 * fa_fwd_dropout and fa_bwd_dropout apply for a requested dropout_p: the
 * requested value quantised to a multiple of 1/256 (0.1 runs as 26/256 =
 * 0.1015625).  A host function (no device work); -1 when dropout_p is not in
 * [0, 1).
 */
FA_API float fa_dropout_effective_p(float dropout_p);
FA_API int fa_fwd_dropout(const void *q, const void *k, const void *v, void *o, float *lse,
                          const uint8_t *block_mask, int B, int H, int N, int d, float scale,
                          int causal, float dropout_p, unsigned long long seed, fa_stream_t stream);
FA_API int fa_bwd_dropout(const void *q, const void *k, const void *v, const void *o,
                          const void *dout, const float *lse, const uint8_t *block_mask,
                          void *dq, void *dk, void *dv, void *workspace,
                          int B, int H, int N, int d, float scale, int causal,
                          float dropout_p, unsigned long long seed, fa_stream_t stream);

/*
 * Forward with 8-bit inputs: q, k, v hold e4m3 values (1 byte each, [B, H, N,
 * d] contiguous) whose real values are q * q_descale[b*H + h] (likewise k, v;
 * a NULL descale array means 1).  Both products run on the 8-bit tensor-core
 * path ("Как работает FlashAttention математически", section 9, names 8-bit
 * tensor-core arithmetic as the FlashAttention-3 extension; the pages give no
 * scaling convention, so the per-(b, h) descale is this library's):
 *   S = scale * dq * dk * (q k^T), softmax as for fa_fwd, P rounded to e4m3
 *   (scaled so a row's largest P is in [16, 256]), O = dv * (P8 v) / l with
 *   l the exact row sum, written as bf16 [B, H, N, d]; LSE (fp32) of the
 *   exact softmax.
 * The e4m3 rounding of P (3 mantissa bits) perturbs each attention weight by
 * at most 2^-4 relative, so |O - O_exact| <= 2^-4 * sum_j P_ij |v_j dv| plus
 * weights below 2^-14 of the row maximum and O's own bf16 rounding.  d must be 128.  workspace: device memory of
 * fa_fwd_fp8_workspace_bytes(B, H, N, d) bytes, 256-byte aligned (it receives
 * v transposed).  Other arguments, errors and asynchrony as for fa_fwd.
 */
FA_API size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d);
FA_API int fa_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse,
                      const float *q_descale, const float *k_descale, const float *v_descale,
                      int B, int H, int N, int d, float scale, int causal, void *workspace,
                      fa_stream_t stream);

/*
 * Block masks for the sparse patterns that block-sparse attention serves
 * ("Как работает FlashAttention математически", section 9: block-sparse
 * FlashAttention for sliding-window and dilated attention), at the 128 x 128
 * block granularity of fa_fwd_blocksparse.  Host functions: `mask` is HOST
 * memory of nb * nb bytes, nb = ceil(N / 128), row = query block, written
 * with 0 / 1; copy it to the device before use.  No GPU is touched.
 *
 * fa_block_mask_window: query block i keeps key block j iff
 *   i - left <= j <= i + right   (left, right >= 0, in blocks).
 *   right = 0 with causal = 1 in the attention call is causal sliding-window
 *   attention over the previous `left` blocks and the query's own block.
 * fa_block_mask_dilated: query block i keeps key block j iff
 *   j = i + t * dilation for an integer t with |t| <= window (t <= 0 when
 *   causal != 0)   (window >= 0, dilation >= 1; dilation 1 is the window).
 * Return FA_OK, FA_ERR_INVALID (null mask, N < 1, negative extents,
 * dilation < 1) or FA_ERR_UNSUPPORTED (nb > 1024, beyond the kernels' limit).
 */
FA_API int fa_block_mask_window(uint8_t *mask, int N, int left, int right);
FA_API int fa_block_mask_dilated(uint8_t *mask, int N, int window, int dilation, int causal);

/*
 * Decoding: the Nq newest query tokens of each (b, h) against a key/value
 * cache ("Как работает FlashAttention математически", section 9:
 * FlashDecoding -- K and V cached, Q the newest token).  The cache is split
 * into chunks processed in parallel; each chunk's O and LSE are merged with
 * the statistics merge of "FlashAttention" notes, "Tiling" (exact up to
 * rounding).
 *
 *   q, o        : bf16 [B, H, Nq, d] device memory; lse: fp32 [B, H, Nq]
 *   k, v        : bf16 [B, H, Nk, d] device memory, the cache's capacity Nk
 *   seqlens_k   : int32 [B] device memory, the valid cache rows of each batch
 *                 (clamped to [0, Nk]); NULL means all Nk rows are valid
 *   causal      : query i sits at position L - Nq + i of a cache of L valid
 *                 rows and sees keys 0 .. L - Nq + i; without it all L keys.
 *                 A query that sees no key gets O = 0, LSE = -inf.
 *   workspace   : device memory of fa_decode_workspace_bytes(B, H, Nq, Nk, d)
 *                 bytes, 256-byte aligned (may be NULL when that is 0)
 * Supported: 1 <= Nq <= 8, Nk >= 1, d in {64, 128}, B * H * Nk * d < 2^31.
 * Errors and asynchrony as for the other compute calls.
 */
FA_API size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d);
FA_API int fa_decode(const void *q, const void *k, const void *v, void *o, float *lse,
                     const int *seqlens_k, int B, int H, int Nq, int Nk, int d, float scale,
                     int causal, void *workspace, fa_stream_t stream);

/*
 * Size of the device scratch array behind fa_bwd_noalloc: 64 MiB per device.
 * fa_bwd_noalloc accepts a problem when fa_bwd_workspace_bytes(B, H, N, d) is
 * at most this: B * H * N * d up to about 16.5 million elements at d = 128
 * and 16.2 million at d = 64 (N a multiple of 128).
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * Backward that allocates nothing: the same computation and arguments as
 * fa_bwd, minus `workspace`.  (The attention pages have no counterpart to
 * this entry point; it exists for callers, not for the method.)
 *
 * Who needs it: callers that cannot call cudaMalloc on the compute path,
 * for example a serving process whose memory pool has reserved the device
 * up front, or a plugin inside a host framework that owns the allocator and
 * forbids side allocations.  They still pass every input and output buffer;
 * only the fp32 dQ accumulator and the D vector move into a file-scope
 * device array of FA_NOALLOC_SCRATCH_BYTES inside libfa.so.  The array is a
 * CUDA module of its own: under lazy module loading (the CUDA runtime's
 * default) a device holds it from the first call of this entry point there
 * until the process exits; with eager loading (CUDA_MODULE_LOADING=EAGER),
 * every device that loads the library holds it.
 *
 * Behaviour:
 *   - Returns FA_ERR_SCRATCH, without enqueuing anything, when
 *     fa_bwd_workspace_bytes(B, H, N, d) exceeds FA_NOALLOC_SCRATCH_BYTES;
 *     the other argument checks are those of fa_bwd, and q must live on
 *     the current device (FA_ERR_INVALID otherwise).
 *   - The first call on each device looks up the device address of the
 *     array (cudaGetSymbolAddress, with that device current).  Make that
 *     first call before any stream capture on that device.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Every call on a device shares the one array and leaves its last
 *     contents there; the first stage zeroes the dQ accumulator on every
 *     call.  Calls whose work overlaps on the GPU (other streams, other
 *     threads) race on the array: serialise them.
 */
FA_API int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                          const void *dout, const float *lse, void *dq, void *dk, void *dv,
                          int B, int H, int N, int d, float scale, int causal, fa_stream_t stream);

/*
 * Forward and backward of tensors that live in host memory: the call a
 * training step makes when its Q, K, V and dO arrive from the host and
 * O, LSE, dQ, dK and dV go back.  The same computation as fa_fwd followed by
 * fa_bwd (fa_fwd_blocksparse / fa_bwd_blocksparse when block_mask is given),
 * done in chunks of whole heads: the copies into the device of chunk c + 1,
 * the kernels of chunk c and the copies back of chunk c - 1 run at the same
 * time on three streams that the library owns (one set per device), through
 * two device buffer sets in `workspace`.  (A data-movement entry point for
 * callers; the attention pages do not describe it.)
 *
 *   q, k, v, dout   : bf16 [B, H, N, d] in host memory
 *   o, dq, dk, dv   : bf16 [B, H, N, d] in host memory, written
 *   lse             : fp32 [B, H, N] in host memory, written
 *   block_mask      : NULL, or device uint8 [N/128][N/128] as for
 *                     fa_fwd_blocksparse (combined with `causal`)
 *   workspace       : device memory, 256-byte aligned, of at least
 *                     fa_fwd_bwd_host_workspace_bytes(B, H, N, d) bytes
 *   workspace_size  : its size in bytes
 * Host buffers should be page-locked (cudaHostAlloc / pinned): the copies
 * then run asynchronously at full link speed.  Pageable buffers work, but
 * the copies stage through the driver and do not overlap.
 *
 * Ordering: the work starts after everything already queued on `stream` and
 * `stream` waits for its end (the last copy back), so a synchronisation of
 * `stream` makes the host outputs readable.  That holds for an error return
 * too: whatever was enqueued before the failing call finishes before
 * `stream` goes on.  The host inputs must stay
 * unchanged, and the outputs unread, until then.  Calls from several host
 * threads on one device are serialised while they enqueue; the workspace of
 * a call must not be in use by other work.
 * Returns FA_ERR_INVALID for a null pointer, an unaligned or too small
 * workspace, bad sizes or scale; FA_ERR_UNSUPPORTED as fa_fwd; FA_ERR_CUDA
 * when a stream, event or copy call fails.  Dropout is not offered here.
 */
FA_API size_t fa_fwd_bwd_host_workspace_bytes(int B, int H, int N, int d);
FA_API int fa_fwd_bwd_host(const void *q, const void *k, const void *v, const void *dout, void *o,
                           float *lse, void *dq, void *dk, void *dv, const uint8_t *block_mask,
                           void *workspace, size_t workspace_size, int B, int H, int N, int d,
                           float scale, int causal, fa_stream_t stream);

/*
 * The forward alone for host-resident tensors, streamed the same way as
 * fa_fwd_bwd_host: the same computation as fa_fwd (fa_fwd_blocksparse when
 * block_mask is given), in chunks of whole heads whose copies in, kernels
 * and copies back overlap on the library's three streams.
 *
 *   q, k, v         : bf16 [B, H, N, d] in host memory
 *   o               : bf16 [B, H, N, d] in host memory, written
 *   lse             : fp32 [B, H, N] in host memory, written
 *   block_mask      : NULL, or device uint8 [N/128][N/128] (with `causal`)
 *   workspace       : device memory, 256-byte aligned, of at least
 *                     fa_fwd_host_workspace_bytes(B, H, N, d) bytes
 * Host buffers, ordering, threads and errors: as for fa_fwd_bwd_host.
 */
FA_API size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d);
FA_API int fa_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                       const uint8_t *block_mask, void *workspace, size_t workspace_size,
                       int B, int H, int N, int d, float scale, int causal, fa_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word: FA_OK, or FA_ERR_TIMEOUT when a kernel wait gave up.  Returns
 * FA_ERR_CUDA when the synchronisation itself fails.
 */
FA_API int fa_get_device_error(fa_stream_t stream);

/*
 * Sets the limit, in nanoseconds, after which a kernel's wait on an on-chip
 * barrier gives up (default 2e9).  Applies to launches made after the call,
 * from any thread.  Returns FA_ERR_INVALID for 0.
 */
FA_API int fa_set_wait_timeout_ns(uint64_t ns);

/*
 * Self-test of the timeout path: launches one small kernel whose barrier wait
 * can never complete, with the given limit (nanoseconds, at most 1e9), waits
 * for it and returns what fa_get_device_error() then reports (FA_ERR_TIMEOUT
 * when the bounded wait works).  Faults nothing; the context stays usable.
 */
FA_API int fa_debug_wait_timeout(uint64_t timeout_ns, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
