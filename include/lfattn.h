/*
 * lfattn — Longformer sparse self-attention (forward) on one B300 GPU.
 *
 * The operation (sources are web pages, cited by title and section):
 *   "基于自注意力机制的长文本建模算法：Longformer详解" (Longformer explained)
 *       §2 sliding window, dilated sliding window and global attention;
 *       §4 the patterns combined under one attention.
 *   "基于Block-Sparse Attention的Longformer" (block-sparse Longformer)
 *       §3 sliding-window attention, §4 global attention.
 *   "Reformer哈希" §核心原理: Attention(Q,K,V) = softmax(QK^T/sqrt(d)) V.
 *
 * For head h with dilation d = dilation[h], one-sided window w, sequence
 * length L and sorted global positions G (n_global of them):
 *   band(i) = { i + d*t : |t| <= w, 0 <= i + d*t < L }
 *   K(i)    = [0, L)          if i is in G (global tokens see every key)
 *           = band(i) ∪ G     otherwise (every token sees the globals; each
 *                             key counted once)
 *   out_i   = sum_{j in K(i)} softmax_j(scale * q_i . k_j) v_j
 * with one softmax per query row over all of K(i).
 *
 * Conventions shared by every call:
 *   - Tensors are contiguous [B, H, L, D] (heads already split), row-major.
 *   - Tensor pointers are DEVICE pointers owned by the caller, unless the
 *     function says otherwise; they must be 16-byte aligned.
 *   - dilation[] and global_idx[] are HOST arrays read during the call.
 *   - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t;
 *     NULL = the legacy default stream); only lf_attn_get_status,
 *     lf_attn_pairs (which returns a count) and lf_attn_fwd_host block.
 *   - Library-owned state: a cache of per-shape plans (device work lists and
 *     the global-position table), the kernel parameters of recent calls, and
 *     one grow-only scratch buffer per (device, stream) taken from the
 *     stream-ordered allocator (cudaMallocAsync / cudaFreeAsync), reused by
 *     every later call on that stream.  A stream handle that is destroyed
 *     and reused by a new stream inherits the buffer: finish the old
 *     stream's work first.
 *   - Threads: the caches are locked, and calls from several host threads
 *     may overlap, with one exception.  A call that frees cached plans
 *     (lf_plan_cache_clear, and a call with a new extra-block table once 32
 *     are cached: see lf_attn_fwd_blocks) must not overlap calls of other
 *     threads that use the plans it frees.
 *   - No C++ exception crosses this interface.  A non-OK status leaves a
 *     message for lf_last_error() in the calling thread.
 *   - Device-side waits are bounded; a wait that runs out records a timeout
 *     that lf_attn_get_status reports (the kernel then returns cleanly and
 *     the outputs of that call are undefined).
 */
#ifndef LFATTN_H
#define LFATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LF_OK = 0,
  LF_ERR_INVALID_ARG = 1,   /* bad shape, pointer, alignment, index list or scale */
  LF_ERR_UNSUPPORTED = 2,   /* valid but not implemented (see each call) */
  LF_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  LF_ERR_NOMEM = 4,         /* device allocation failed */
  LF_ERR_TIMEOUT = 5        /* a device-side wait ran out (lf_attn_get_status) */
} lf_status;

typedef void* lf_stream_t; /* cudaStream_t */

#if defined(__GNUC__)
#define LF_API __attribute__((visibility("default")))
#else
#define LF_API
#endif

/*
 * lf_attn_fwd — sparse attention forward, bf16 in / bf16 out.
 *
 *   q, k, v   device, bf16 [B,H,L,D], read only.
 *   out       device, bf16 [B,H,L,D], written (every element).
 *   B, H, L   >= 1.  D in {64, 128}.  w >= 0 (one-sided window).
 *   dilation  host int32[H], each >= 1.  For d > 1, L % d must be 0
 *             (else LF_ERR_UNSUPPORTED).  At most 8 distinct values.
 *   global_idx host int32[n_global], strictly increasing, in [0, L);
 *             may be NULL when n_global == 0.  0 <= n_global <= L.
 *   scale     finite, > 0 (the configurations use 1/sqrt(D)).
 *   stream    cudaStream_t.
 *
 * Arithmetic: products in bf16 on the tensor cores with fp32 accumulation,
 * softmax in fp32, probabilities rounded to bf16 before the product with V,
 * output rounded to bf16 (round to nearest even).
 */
LF_API lf_status lf_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int H,
                      int L, int D, int w, const int32_t* dilation, const int32_t* global_idx,
                      int n_global, float scale, lf_stream_t stream);

/*
 * lf_attn_fwd_bias — lf_attn_fwd with a relative-position bias on the
 * window's scores.  Longformer explained, §5 (position-encoding adaptations), says
 * local attention is strengthened by a relative position bias but gives no
 * formula.  The form implemented: for a non-global row i and a key
 * j = i + d*t of its window (|t| <= w),
 *   s_ij = scale * q_i . k_j + rel_bias[h, t + w];
 * global keys outside the window and global rows carry no bias.
 *   rel_bias  device, fp32 [H, 2w+1], row-major, read only; values of
 *             magnitude up to 1e4 (-1e4 already removes a key: its weight
 *             falls below 2^-125).  Larger magnitudes are not checked and
 *             not supported: the exponentials take s*scale*log2(e) minus a
 *             rounded copy of the row maximum, and beyond about 2^30 the
 *             rounding alone overflows them.
 * Other arguments and errors as lf_attn_fwd; LF_ERR_INVALID_ARG also for a
 * null or misaligned rel_bias.  Two launches on `stream`: a copy of the table
 * scaled by 1/scale and zero-padded on both sides (into a workspace the
 * library keeps per device and stream, freed by lf_plan_cache_clear), then a
 * separate build of the attention kernel that adds it to the window's
 * scores; lf_attn_fwd's kernel is unchanged.
 */
LF_API lf_status lf_attn_fwd_bias(const void* q, const void* k, const void* v, void* out,
                                  const float* rel_bias, int B, int H, int L, int D, int w,
                                  const int32_t* dilation, const int32_t* global_idx,
                                  int n_global, float scale, lf_stream_t stream);

/*
 * lf_attn_fwd_blocks — lf_attn_fwd with extra key blocks per query tile:
 * BigBird's random blocks added to window + global attention, or a fixed
 * strided choice of blocks (the commentary on "Efficient Transformers: A
 * Survey", §3.1 fixed patterns and §3.2 combined patterns; neither gives a
 * block size or an indexing).  The form implemented, per head h with
 * dilation d: a query i with r = i mod d, t = i div d lies in tile
 * qt = t div 128 of residue class r; nqt = ceil(ceil(L/d) / 128) tiles per
 * class.  Row r*nqt + qt of xblocks[h] lists up to R key blocks kb (-1 for
 * none; duplicates allowed); block kb holds the keys r + d*t' with
 * 128*kb <= t' < 128*kb + 128 (clipped to [0, L)).  They join K(i) of every
 * non-global row of the tile, each key counted once (keys of the row's
 * window and global keys are not added twice).  Global rows still see all
 * keys.
 *   xblocks  host, int32 [H, T, R] row-major, read during the call only;
 *            T >= d*nqt for every head; entries in [-1, nqt).
 * Other arguments and errors as lf_attn_fwd; LF_ERR_INVALID_ARG for a table
 * of the wrong shape or an entry out of range.  The table is part of the
 * cached plan: a new table builds (and keeps) a new plan.  When 32 tables are
 * cached, the next new one first frees them all (their plans included), after
 * a cudaDeviceSynchronize; tables drawn anew every step therefore cost a
 * plan build per call and a device synchronization every 32 calls.
 */
LF_API lf_status lf_attn_fwd_blocks(const void* q, const void* k, const void* v, void* out,
                                    int B, int H, int L, int D, int w,
                                    const int32_t* dilation, const int32_t* global_idx,
                                    int n_global, const int32_t* xblocks, int T, int R,
                                    float scale, lf_stream_t stream);

/*
 * lf_attn_fwd_lse — lf_attn_fwd that also writes each row's log-sum-exp,
 *   lse[b,h,i] = ln( sum_{j in K(i)} exp(scale * q_i . k_j) )   (fp32),
 * the normaliser a backward pass needs (p_ij = exp(scale q_i.k_j - lse_i)).
 *   lse  device, fp32 [B,H,L], written (every element), 16-byte aligned.
 * Other arguments and errors as lf_attn_fwd.
 */
LF_API lf_status lf_attn_fwd_lse(const void* q, const void* k, const void* v, void* out,
                                 float* lse, int B, int H, int L, int D, int w,
                                 const int32_t* dilation, const int32_t* global_idx, int n_global,
                                 float scale, lf_stream_t stream);

/*
 * lf_attn_bwd — gradients of sum(out * dout) for out = lf_attn_fwd(q, k, v).
 *
 * With s_ij = scale q_i . k_j over K(i), p_ij = exp(s_ij - lse_i):
 *   dv_j = sum_i p_ij dout_i
 *   ds_ij = p_ij (dout_i . v_j - dout_i . out_i)
 *   dq_i = scale sum_j ds_ij k_j,   dk_j = scale sum_i ds_ij q_i
 * (the derivative of the forward's definition; the pages give no backward).
 *
 *   q, k, v, out, dout  device, bf16 [B,H,L,D], read only (out and lse from
 *                 the forward on the same q, k, v: lf_attn_fwd_lse).
 *   lse           device, fp32 [B,H,L], read only.
 *   dq, dk, dv    device, fp32 [B,H,L,D], written (every element).
 *   Other arguments and errors as lf_attn_fwd.
 *
 * Products in bf16 (p and ds are rounded to bf16 before their products) with
 * fp32 accumulation; contributions are summed with fp32 atomics, so the
 * low bits of the result depend on the order the hardware applies them.
 * Scratch: B*H*L*4 bytes in a third grow-only buffer per (device, stream).
 */
LF_API lf_status lf_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                             const float* lse, const void* dout, float* dq, float* dk, float* dv,
                             int B, int H, int L, int D, int w, const int32_t* dilation,
                             const int32_t* global_idx, int n_global, float scale,
                             lf_stream_t stream);

/*
 * lf_attn_fwd_f32 — same operation with fp32 q/k/v/out.  q, k and v are
 * rounded to bf16 (nearest even) on the device first; the output is written
 * in fp32 without the final bf16 rounding.  Same arguments and errors as
 * lf_attn_fwd, all tensors fp32.
 */
LF_API lf_status lf_attn_fwd_f32(const void* q, const void* k, const void* v, void* out, int B, int H,
                          int L, int D, int w, const int32_t* dilation,
                          const int32_t* global_idx, int n_global, float scale,
                          lf_stream_t stream);

/*
 * lf_layer_fwd — one Longformer layer forward, bf16 activations.
 *
 * The layer of "基于Block-Sparse Attention的Longformer" (block-sparse
 * Longformer) §6 "Longformer的整体架构", with its attention read as the
 * sparse attention above (one softmax per row over band(i) ∪ G, per head):
 *   [q | k | v] = x W_qkv^T + b_qkv, rounded to bf16, split into H heads
 *   a  = attention(q, k, v)      (lf_attn_fwd: D = hidden / H, w, dilation,
 *                                 global_idx, scale)
 *   x1 = bf16(LN1(x + a))         (a merged back to [B, L, hidden])
 *   y  = bf16(LN2(x1 + x1 W_ff^T + b_ff))
 * where LN(v) = (v - mean(v)) / sqrt(var(v) + eps) * gamma + beta over the
 * hidden axis (biased variance).  The page's feed-forward step is one linear
 * map (no activation); there is no output projection after the attention.
 *
 *   x      device, bf16 [B, L, hidden], read only.
 *   w_qkv  device, bf16 [3*hidden, hidden]: rows 0..hidden-1 map to q, then
 *          k, then v (the nn.Linear layout: out = x W^T + b).
 *   b_qkv  device, fp32 [3*hidden].
 *   w_ff   device, bf16 [hidden, hidden];  b_ff device, fp32 [hidden].
 *   ln1, ln2 device, fp32 [2*hidden]: gamma, then beta.
 *   out    device, bf16 [B, L, hidden], written (every element); may not
 *          alias x.
 *   hidden = H * D with D in {64, 128}; hidden in {64, 128, 256, 384, 512,
 *          768, 1024, 1536, 2048} (else LF_ERR_UNSUPPORTED).
 *   w, dilation, global_idx, n_global, scale: as for lf_attn_fwd.
 *   eps    finite, > 0.
 *
 * The two linear maps are this library's tcgen05 GEMMs (bf16 inputs, fp32
 * accumulation in tensor memory): the q/k/v map writes bf16(x W^T + b)
 * straight into per-head q, k, v; the feed-forward map applies its bias, the
 * residual and the second LayerNorm in its epilogue.  q, k, v, the attention
 * output, x1 and out are stored in bf16.  Scratch: a second grow-only buffer
 * per (device, stream), about B*L*hidden*10 bytes, apart from the
 * attention's.  Pointers must be 16-byte aligned (LF_ERR_INVALID_ARG).
 */
LF_API lf_status lf_layer_fwd(const void* x, const void* w_qkv, const float* b_qkv,
                              const void* w_ff, const float* b_ff, const float* ln1,
                              const float* ln2, void* out, int B, int L, int hidden, int H, int w,
                              const int32_t* dilation, const int32_t* global_idx, int n_global,
                              float scale, float eps, lf_stream_t stream);

/*
 * lf_attn_fwd_host — lf_attn_fwd (is_f32 == 0) or lf_attn_fwd_f32
 * (is_f32 != 0) on HOST buffers, same layout: copies q, k, v to device
 * memory it allocates on `stream`, runs the forward, copies the result into
 * the host buffer `out` and synchronises `stream` before returning.  The
 * work is split into chunks of whole heads of one batch element (about
 * eight chunks), pipelined over two streams of the library, so that the
 * copies in, the computation and the copies out of different chunks
 * overlap; those streams start after the work already queued on `stream`,
 * and `stream` continues after them.  Pinned host memory gives
 * asynchronous copies (pageable memory works, without the overlap).  One
 * host-buffer call runs at a time per process.
 */
LF_API lf_status lf_attn_fwd_host(const void* q, const void* k, const void* v, void* out, int is_f32,
                           int B, int H, int L, int D, int w, const int32_t* dilation,
                           const int32_t* global_idx, int n_global, float scale,
                           lf_stream_t stream);

/*
 * lf_attn_fwd_noalloc — lf_attn_fwd for callers that may not allocate
 * device memory.  The pages describe no such call; it exists for callers
 * that cannot let a library allocate: inference engines that plan all device
 * memory when they start and forbid allocation afterwards (for predictable
 * latency and no out-of-memory failure mid-run), and processes whose caching
 * allocator already holds the free device memory, where a direct allocation
 * would fail or fragment it.
 *
 * Same arguments, arithmetic and errors as lf_attn_fwd (bf16 in / bf16 out);
 * the output is the same.  It calls no cudaMalloc, cudaFree or other
 * allocating routine: its scratch (work list, global-position tables,
 * gathered global rows, global-row partials) lives in one fixed device array
 * of 32 MiB that the library declares.  A device holds the array from the
 * library's first use on it until the process exits: the library's device
 * code is loaded lazily, on the first call of any of its entry points on
 * that device, and the array is reserved then.  A caller whose allocator
 * will hold the device's free memory should therefore make one call per
 * device at start-up, before the allocator reserves its memory.  A problem
 * needing more scratch is rejected
 * with LF_ERR_UNSUPPORTED and a message giving both sizes (for example B=1,
 * H=16, L=65536, D=128 with 16 global tokens needs about 55 MiB).  Problems
 * without global tokens need only the work list and the global flags.
 *
 *   - The first call on a device looks up the array's device address there
 *     (one cudaGetSymbolAddress).
 *   - Every call uses the same array and overwrites what the previous call
 *     left in it; nothing in it needs to start at zero.  Calls whose work
 *     overlaps on the GPU (other streams, other threads) race on it: order
 *     them on one stream, or synchronise between them.
 *   - The per-kernel event tracing (lf_profile_*) does not record its
 *     launches; lf_launch_count counts them.
 */
LF_API lf_status lf_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, int B,
                                     int H, int L, int D, int w, const int32_t* dilation,
                                     const int32_t* global_idx, int n_global, float scale,
                                     lf_stream_t stream);

/*
 * lf_attn_pairs — the attended key lists, per (head, query), in CSR form.
 * Batch-independent (the pattern does not depend on b).
 *
 *   row_ptr   device int64[H*L + 1]: row (h, i) is index h*L + i; its keys
 *             are col_idx[row_ptr[r] .. row_ptr[r+1]) in increasing order.
 *             Always written.
 *   col_idx   device int32[cap], or NULL to only count.
 *   cap       capacity of col_idx in elements.
 *   total     host int64*, receives the number of pairs (row_ptr[H*L]).
 *
 * Blocks until the count is known.  Returns LF_ERR_INVALID_ARG (with *total
 * set) when col_idx is non-NULL and cap < total.  Same pattern arguments
 * and errors as lf_attn_fwd (L % d need not be 0 here).  The enumerator
 * uses the same key-set predicates as the attention kernel.
 */
LF_API lf_status lf_attn_pairs(int H, int L, int w, const int32_t* dilation, const int32_t* global_idx,
                        int n_global, int64_t* row_ptr, int32_t* col_idx, int64_t cap,
                        int64_t* total, lf_stream_t stream);

/* Message for the last non-OK status returned in this thread ("" if none).
 * The pointer stays valid until the thread's next lfattn call. */
LF_API const char* lf_last_error(void);

/*
 * Synchronises `stream`, then reports LF_ERR_TIMEOUT if a device-side wait
 * of any call on the current device ran out since the last check (and
 * clears that record), LF_ERR_CUDA if the stream holds an error, else LF_OK.
 */
LF_API lf_status lf_attn_get_status(lf_stream_t stream);

/*
 * lf_selftest_wait_timeout — exercises the device-side timeout path without
 * a fault: one thread waits, with the attention kernel's bounded wait, on a
 * barrier nothing completes; after about timeout_us microseconds (1 ..
 * 1000000) it records the timeout and the kernel returns.  The next
 * lf_attn_get_status on the stream then reports LF_ERR_TIMEOUT (and clears
 * it); the context stays usable.
 */
LF_API lf_status lf_selftest_wait_timeout(int timeout_us, lf_stream_t stream);

/* Frees every cached plan, cached call parameters and scratch buffer
 * (synchronises the device). */
LF_API void lf_plan_cache_clear(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads).  Lets callers count the kernels a region of work ran. */
LF_API uint64_t lf_launch_count(void);

/*
 * Per-kernel device-time tracing.  While enabled, every kernel launch of the
 * library is bracketed by two CUDA events recorded on the launch's stream.
 * lf_profile_query synchronises on those events and returns the summed
 * device time (ms) and number of launches of the kernels whose name
 * contains `name` (NULL or "" = all) since the last lf_profile_reset.
 * Kernel names: "attn_main", "gather_globals", "combine_globals",
 * "cast_f32_bf16", "pairs_count", "pairs_scan", "pairs_fill", and for the
 * layer "layer_gemm_qkv", "layer_split_qkv", "layer_merge_ln1",
 * "layer_gemm_ff", "layer_ln2".
 * Tracing adds two event records per traced launch (each costs the stream
 * about a microsecond); it is off by default.  lf_profile_only restricts it
 * to the kernels whose name contains `name` (NULL or "" = all, the default),
 * so that a timed loop brackets only the kernel it measures.
 */
LF_API void lf_profile_enable(int on);
LF_API void lf_profile_only(const char* name);
LF_API void lf_profile_reset(void);
LF_API lf_status lf_profile_query(const char* name, double* total_ms, uint64_t* launches);

/* Library version: major * 10000 + minor * 100 + patch. */
LF_API int lf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LFATTN_H */
