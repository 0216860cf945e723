/*
 * attn_gqa.h -- C ABI of libattn_gqa.so: grouped-query scaled-dot-product
 * attention computed in one tiled online-softmax pass on an NVIDIA GB300
 * (sm_103a).  The score matrix is never materialised.
 *
 * The operations are those of three published WGSL compute shaders:
 *   - meganeura 0.2.0, src/shaders/attention.wgsl         -> attn_forward
 *   - meganeura 0.2.0, src/shaders/cached_attention.wgsl  -> attn_decode_cached
 *   - cera, src/backend/shaders/attention_prefill.wgsl    -> attn_prefill
 * Argument lists follow the shaders' parameter lists; shader templating and
 * storage bindings become plain arguments.  Further entry points fill the
 * shaders' open hooks and named future work: sliding windows (*_window),
 * paged caches (*_paged), rotary embedding (*_rope), the backward pass,
 * and an append-and-decode step; each states its reading below.
 *
 * Common rules for every entry point
 *   Notation   H = num_heads, G = num_kv_heads, D = head_dim, gs = H / G.
 *   GQA map    query head h reads kv head g = h / gs (integer division); H
 *              must be a multiple of G (all three shaders divide this way).
 *   Scale      scores are scale * (q . k); forward and decode use
 *              scale = 1 / sqrt(D) (the meganeura shaders' inverseSqrt), prefill
 *              takes scale as an argument (the cera shader's params[5]).
 *   Data       fp32 in, fp32 out, row-major, all pointers are DEVICE memory
 *              owned by the caller.  The library keeps no pointer after a call
 *              returns.  Some calls need temporary scratch (the 16-bit K/V
 *              operand copies of the tensor-core paths, K turned for RoPE,
 *              the backward's per-row values; sizes from the
 *              attn_*_workspace_bytes queries).  With a workspace bound to the
 *              calling thread (attn_set_workspace) it is carved from that
 *              caller-owned buffer and the library allocates nothing.
 *              Otherwise it is stream-ordered on the call's stream, from a
 *              memory pool the library creates per device and keeps (freed
 *              blocks stay reserved for later calls; attn_release_scratch
 *              returns them).  Besides, every GPU that loads the library holds one
 *              fixed 4 MiB array for attn_decode_cached_noalloc (shared by
 *              all its calls on that device, kept until the process exits).
 *              The backward also runs one of its kernels on a library-owned
 *              stream per device, forked from and joined back into `stream`;
 *              all callers on a device share that stream, so concurrent
 *              backward calls on independent streams serialise there, and a
 *              backward must not be captured into CUDA graphs from two
 *              threads at once.
 *   Streams    every call is asynchronous on `stream` (a cudaStream_t; NULL is
 *              the legacy default stream).  Results are ready when the stream
 *              has reached the call.
 *   Errors     the return value is an attn status code.  Host-side checks run
 *              before anything is launched: on ATTN_ERR_INVALID_ARG or
 *              ATTN_ERR_UNSUPPORTED nothing is written.  ATTN_ERR_CUDA means a
 *              launch failed (the CUDA error is left in place for
 *              cudaGetLastError).  Conditions only the device can see (a
 *              device-resident kv_pos past the cache, a bounded wait that ran
 *              out) are recorded in a per-device status word; read it with
 *              attn_get_status.
 *   Empty      a window of zero keys writes zeros to the output rows and
 *              (-1e30, -1e30) to their LSE pair (attention.wgsl, fn main: the
 *              select() guards on sum_exp == 0).
 *   Precision  ATTN_FP32: fp32 CUDA-core arithmetic throughout.
 *              ATTN_TF32: both products on tcgen05 tensor cores with fp32
 *              accumulation and an fp32 softmax.  QK^T keeps Q to 22
 *              significant bits (two fp16 parts, hi + lo, under a power of
 *              two per query row) and K to 11 (fp16 under a power of two per
 *              128-key tile of a kv head): two products, the tensor time of
 *              one TF32 product.  PV takes TF32 operands (P and V with 11
 *              significant bits).  The scores feed an exponential, so their
 *              operand rounding sets the error: plain TF32 Q and K reach
 *              3.5e-3 of max|V| on scores of standard deviation 9, this
 *              scheme about 1.4e-3.
 *              ATTN_BF16: 16-bit operands at the full 16-bit tensor rate.
 *              QK^T takes fp16 operands (11 significant bits) under powers
 *              of two, one per query row and one per 128-key tile of a kv
 *              head, that keep every value below 2^15 whatever the fp32
 *              magnitudes; PV takes bf16 operands (P <= 2^24 and V; the
 *              fp32 accumulators carry |V| * keys * 2^24 below fp32's range
 *              for any |V| < 2^70).  K and V are converted by a pre-pass, Q
 *              and P on their way into the tensor core.
 *              Tensor-core precisions need D in {64, 128}, else they
 *              return ATTN_ERR_UNSUPPORTED.  Their kernels take
 *              1 <= gs <= 128 (a thread block packs 128/gs queries of gs
 *              heads; when gs does not divide 128 the remaining rows idle),
 *              16-byte aligned pointers, Q/out row strides that are
 *              multiples of 4 floats and K/V row strides that are multiples
 *              of 8 floats (paged caches: page_rows % 32 == 0); a call
 *              outside that runs on the fp32 CUDA-core kernel instead, whose
 *              results lie within every precision's bound.
 *              ATTN_FP32 accepts any 1 <= D <= 128.
 */
#ifndef ATTN_GQA_H
#define ATTN_GQA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; declared here so the header needs no
 * CUDA include. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
    ATTN_CAUSAL = 0, /* query at position p sees keys 0..p          (kv_seq == q_seq) */
    ATTN_FULL = 1,   /* every query sees keys 0..q_seq-1             (kv_seq == q_seq) */
    ATTN_CROSS = 2   /* every query sees keys 0..kv_seq-1 (any kv_seq, 0 allowed)      */
} attn_mask_t;

typedef enum { ATTN_FP32 = 0, ATTN_TF32 = 1, ATTN_BF16 = 2 } attn_prec_t;

enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,
    ATTN_ERR_UNSUPPORTED = 2,
    ATTN_ERR_CUDA = 3,
    ATTN_ERR_TIMEOUT = 4
};

/*
 * Self / cross attention forward with per-row (max, log-sum) output.
 * Source: meganeura attention.wgsl, fn main (variants causal kv_len = pos+1,
 * full kv_len = q_seq, cross kv_len = kv_seq; final store of
 * lse[(pos*H + head)*2 + {0,1}] = (max_score, log(sum_exp))).
 *
 *   q    [q_seq, H*D]     element (pos, h, d) at pos*H*D + h*D + d
 *   k, v [kv_seq, G*D]    element (t, g, d)   at t*G*D + g*D + d
 *   out  [q_seq, H*D]     same layout as q
 *   lse  [q_seq, H, 2]    (m, log l) with m the row's largest scaled score and
 *                         l = sum_t exp(s_t - m), so log-sum-exp = m + log l.
 *                         May be NULL (not written).
 *   mask ATTN_CAUSAL / ATTN_FULL need kv_seq == q_seq.
 *   prec ATTN_FP32, ATTN_TF32 or ATTN_BF16.
 * q_seq == 0 is a no-op (pointers may then be NULL).  Errors: INVALID_ARG for
 * NULL q/k/v/out (or k/v with kv_seq > 0), H % G != 0, G == 0, D == 0 or
 * D > 128, kv_seq != q_seq for causal/full, an unknown mask or precision;
 * UNSUPPORTED as described under Precision.
 */
ATTN_API int attn_forward(const float *q, const float *k, const float *v, float *out, float *lse,
                 uint32_t q_seq, uint32_t kv_seq, uint32_t num_heads, uint32_t num_kv_heads,
                 uint32_t head_dim, attn_mask_t mask, attn_prec_t prec, attn_stream_t stream);

/*
 * Bytes of device workspace attn_decode_cached needs for these sizes on the
 * current device (its SM count sets the number of KV splits).  Returns 0 for
 * sizes attn_decode_cached would reject.
 */
ATTN_API size_t attn_decode_workspace_bytes(uint32_t num_heads, uint32_t num_kv_heads, uint32_t head_dim,
                                   uint32_t max_seq);

/*
 * Cached single-token decode.  Source: meganeura cached_attention.wgsl,
 * fn main (Q = [1, H*D], K/V from a cache, kv_len = kv_pos_buf[0] + 1, so the
 * token attends to positions 0..kv_pos inclusive).
 *
 *   q                  [1, H*D]
 *   k_cache, v_cache   [max_seq, G*D]
 *   kv_pos_dev         one uint32 in DEVICE memory, read by the kernels (so a
 *                      CUDA graph can replay the call as the position grows)
 *   out                [1, H*D]
 *   max_seq            rows of the cache.  The window is cut at max_seq keys
 *                      (the cera prefill shader's defensive clamp); a kv_pos
 *                      >= max_seq also records ATTN_ERR_INVALID_ARG in the
 *                      device status word.
 *   workspace          device buffer of at least
 *                      attn_decode_workspace_bytes(H, G, D, max_seq) bytes,
 *                      16-byte aligned.  Zero it once (cudaMemset) before its
 *                      first use; each completed call leaves it ready for the
 *                      next.  Calls that share a workspace must not overlap on
 *                      the GPU.
 * The work is split over KV ranges; each split keeps its own (max, sum,
 * weighted V) and the last split of each kv head to finish merges them with
 * the log-sum-exp rule.  Errors: INVALID_ARG for NULL pointers, H % G != 0,
 * G == 0, D == 0 or D > 128, max_seq == 0, or a workspace that is too small
 * or misaligned.
 */
ATTN_API int attn_decode_cached(const float *q, const float *k_cache, const float *v_cache,
                       const uint32_t *kv_pos_dev, float *out, uint32_t num_heads,
                       uint32_t num_kv_heads, uint32_t head_dim, uint32_t max_seq,
                       void *workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * Cached decode of a new token that first appends its own K and V row: the
 * [G*D] rows k_new and v_new are written into row *kv_pos_dev
 * of k_cache and v_cache, then the call is attn_decode_cached over positions
 * 0..kv_pos (the new row included).  The pages leave filling the cache to
 * the host framework; this entry point saves a serving step the separate
 * copies into the cache (the split decode writes the row itself, in the
 * split that ends at kv_pos, before that split reads it).  A kv_pos >=
 * max_seq writes nothing and records ATTN_ERR_INVALID_ARG, as in
 * attn_decode_cached.  Arguments, workspace and errors otherwise as
 * attn_decode_cached, plus NULL k_new / v_new.
 *
 * Step I/O in host memory.  On the shapes the split decode covers (D in
 * {64, 128}, gs = H/G a power of two up to 32; the same holds for
 * attn_decode_cached), q, k_new, v_new, kv_pos_dev and out may also be
 * pinned host memory (cudaHostAlloc / cudaMallocHost, whose addresses are
 * valid on the device under unified addressing): the kernel reads the
 * step's inputs and writes its output across the host link itself, so a
 * serving step needs no staging copies.  The caches and the workspace must
 * be device memory.
 */
ATTN_API int attn_decode_append(const float *q, const float *k_new, const float *v_new, float *k_cache,
                                float *v_cache, const uint32_t *kv_pos_dev, float *out, uint32_t num_heads,
                                uint32_t num_kv_heads, uint32_t head_dim, uint32_t max_seq, void *workspace,
                                size_t workspace_bytes, attn_stream_t stream);

/*
 * Batched causal prefill against a KV cache.  Source: cera
 * attention_prefill.wgsl, fn attention_prefill (params n_heads, n_kv_heads,
 * head_dim, kv_dim, max_seq, scale, start_pos, q_stride, out_stride, q_base;
 * q_global = q_base + i; window min(start_pos + q_global + 1, max_seq)).
 *
 *   q_batch    query i of this call, head h, at (q_base+i)*q_stride + h*D
 *   k_cache,
 *   v_cache    [max_seq, kv_dim]; kv head g at column g*D
 *   out_batch  (q_base+i)*out_stride + h*D; other columns are not written
 *   n_queries  queries in this call (the shader's dispatch height)
 * n_queries == 0 is a no-op.  Errors: INVALID_ARG for NULL pointers,
 * H % G != 0, G == 0, D == 0 or D > 128, kv_dim < G*D, q_stride or
 * out_stride < H*D, start_pos + q_base + n_queries > max_seq (the shader's
 * host-side assertion), a non-finite scale or an unknown precision;
 * UNSUPPORTED as described under Precision.
 */
ATTN_API int attn_prefill(const float *q_batch, const float *k_cache, const float *v_cache,
                 float *out_batch, uint32_t n_queries, uint32_t n_heads, uint32_t n_kv_heads,
                 uint32_t head_dim, uint32_t kv_dim, uint32_t max_seq, float scale,
                 uint32_t start_pos, uint32_t q_stride, uint32_t out_stride, uint32_t q_base,
                 attn_prec_t prec, attn_stream_t stream);

/*
 * Sliding-window (local) attention: the three calls above with one more
 * argument, `window`, placed just before `stream`.  Every other argument,
 * layout, error and result is that of the call without the suffix.
 * Source: meganeura attention.wgsl, fn main -- the key loop of every variant
 * starts at a $KV_START placeholder that the page leaves to the host
 * framework.  This library reads it as a per-row lower bound: a row whose
 * window is keys [0, n) under the rules above attends keys
 *     [max(0, n - window), n)
 * i.e. its last `window` keys (window == 0: no lower bound, the call without
 * the suffix).  A window of 1 returns the V row of the last key; a window at
 * least n changes nothing.  The LSE pair of attn_forward_window describes
 * the kept keys only.  Key tiles that lie wholly before every row's window
 * are neither read nor computed, so the cost follows the window, not the
 * position.  No further errors.
 */
ATTN_API int attn_forward_window(const float *q, const float *k, const float *v, float *out, float *lse,
                                 uint32_t q_seq, uint32_t kv_seq, uint32_t num_heads, uint32_t num_kv_heads,
                                 uint32_t head_dim, attn_mask_t mask, attn_prec_t prec, uint32_t window, attn_stream_t stream);
ATTN_API int attn_decode_cached_window(const float *q, const float *k_cache, const float *v_cache,
                                       const uint32_t *kv_pos_dev, float *out, uint32_t num_heads,
                                       uint32_t num_kv_heads, uint32_t head_dim, uint32_t max_seq,
                                       void *workspace, size_t workspace_bytes, uint32_t window,
                                       attn_stream_t stream);
ATTN_API int attn_prefill_window(const float *q_batch, const float *k_cache, const float *v_cache,
                                 float *out_batch, uint32_t n_queries, uint32_t n_heads, uint32_t n_kv_heads,
                                 uint32_t head_dim, uint32_t kv_dim, uint32_t max_seq, float scale,
                                 uint32_t start_pos, uint32_t q_stride, uint32_t out_stride, uint32_t q_base,
                                 attn_prec_t prec, uint32_t window, attn_stream_t stream);

/*
 * Rotary position embedding (RoPE) fused into the forward.  The forward page
 * has hooks for it ($ROPE_DECL; $ROPE_Q_APPLY on the query value, and the key
 * expression $K_VAL_EXPR) whose bodies it leaves to the host framework.  This
 * library's convention: the pairs (d, d + D/2), d < D/2, of a row at position
 * p turn by the angle p * base^(-2d/D),
 *   x'[d]       = x[d] cos - x[d + D/2] sin
 *   x'[d + D/2] = x[d + D/2] cos + x[d] sin,
 * query row i at position i and key row t at position t; V is not turned.
 *
 * attn_rope_table fills a caller-owned DEVICE table [max_pos, head_dim] of
 * fp32: row p holds the cosines of the D/2 pair angles, then their sines,
 * computed in fp64 (base > 1, head_dim even and <= 128).
 *
 * attn_forward_rope is attn_forward_window with q and k turned first (inside
 * the kernels: the inputs are not modified); rope_table has table_rows >=
 * max(q_seq, kv_seq) rows from attn_rope_table for this head_dim.  Errors as
 * attn_forward_window, plus INVALID_ARG for an odd head_dim, a NULL or short
 * table, and UNSUPPORTED for head_dim % 8 != 0 or a table that is not
 * 16-byte aligned.
 */
ATTN_API int attn_rope_table(float *table, uint32_t max_pos, uint32_t head_dim, double base, attn_stream_t stream);
ATTN_API int attn_forward_rope(const float *q, const float *k, const float *v, float *out, float *lse,
                               uint32_t q_seq, uint32_t kv_seq, uint32_t num_heads, uint32_t num_kv_heads,
                               uint32_t head_dim, attn_mask_t mask, attn_prec_t prec, uint32_t window, const float *rope_table,
                               uint32_t table_rows, attn_stream_t stream);

/*
 * Paged KV cache: decode and prefill against a cache held in pages.  The
 * pages name paged KV only as future work for caches that overflow one buffer
 * (cera attention_prefill.wgsl, header comment); the layout here:
 *   k_pages, v_pages  pools of num_pages pages; page p holds page_rows
 *                     consecutive cache positions as rows
 *                     [p * page_rows, (p + 1) * page_rows) of a
 *                     [num_pages * page_rows, kv_dim] array (decode:
 *                     kv_dim = G*D)
 *   block_table       max_blocks uint32 in DEVICE memory: cache position t
 *                     is in pool page block_table[t / page_rows] at row
 *                     t % page_rows.  Entries may repeat (shared pages).
 * The cache's capacity is max_seq = page_rows * max_blocks; every other
 * argument, the window rule (with `window` as in the *_window calls), the
 * result and the errors are those of attn_decode_cached_window /
 * attn_prefill_window with that max_seq (decode's workspace:
 * attn_decode_workspace_bytes(H, G, D, max_seq)).  Only the block-table
 * entries of pages inside a row's window are read; an entry >= num_pages
 * reads as zeros and records ATTN_ERR_INVALID_ARG in the status word.  The
 * split decode and the tensor-core kernels need page_rows % 32 == 0
 * (otherwise decode, and a tensor-core prefill, run the fp32 CUDA-core
 * kernel).  The TF32 prefill reads named pages in
 * 32-row groups, so rows of such a group past the last attended position
 * must hold finite values.  Further errors: INVALID_ARG for a NULL
 * block_table, page_rows, num_pages or max_blocks of 0, or a capacity or
 * pool of 2^31 rows or more.
 */
ATTN_API int attn_decode_paged(const float *q, const float *k_pages, const float *v_pages,
                               const uint32_t *block_table, const uint32_t *kv_pos_dev, float *out,
                               uint32_t num_heads, uint32_t num_kv_heads, uint32_t head_dim, uint32_t page_rows,
                               uint32_t num_pages, uint32_t max_blocks, void *workspace, size_t workspace_bytes,
                               uint32_t window, attn_stream_t stream);
ATTN_API int attn_prefill_paged(const float *q_batch, const float *k_pages, const float *v_pages,
                                const uint32_t *block_table, float *out_batch, uint32_t n_queries, uint32_t n_heads,
                                uint32_t n_kv_heads, uint32_t head_dim, uint32_t kv_dim, uint32_t page_rows,
                                uint32_t num_pages, uint32_t max_blocks, float scale, uint32_t start_pos,
                                uint32_t q_stride, uint32_t out_stride, uint32_t q_base, attn_prec_t prec, uint32_t window,
                                attn_stream_t stream);

/*
 * Backward of attn_forward / attn_forward_window: the gradients of `out` with
 * respect to q, k and v for an upstream gradient dout.  The pages emit the
 * per-row (max, log-sum) pair for a backward pass (meganeura attention.wgsl:
 * header comment and the final LSE store) but print none; this is the plain
 * gradient of the forward definition, rebuilt from that pair:
 *   p_t  = exp(scale q.k_t - lse0 - lse1)      over the row's kept keys
 *   ds_t = p_t (dout.v_t - dout.out)
 *   dq   = scale sum_t ds_t k_t
 *   dk_t = scale sum over rows of ds_t q      (every query head of the kv head)
 *   dv_t = sum over rows of p_t dout
 * The LSE output is not differentiated (its gradient is taken as zero).
 *
 *   q, out, dout, dq   [q_seq, H*D]  (out and lse exactly as the forward wrote
 *   k, v, dk, dv       [kv_seq, G*D]  them for these q, k, v, mask, window)
 *   lse                [q_seq, H, 2]
 *   mask, window       as attn_forward_window (window 0 = none)
 *   prec               ATTN_FP32: CUDA cores, fp32 arithmetic.
 *                      ATTN_BF16: tensor cores; q, k, v, dout and the
 *                      P and dS tiles rounded to bf16, fp32 accumulation
 *                      (D in {64, 128}, else ATTN_ERR_UNSUPPORTED; a group
 *                      H/G that is not a power of two up to 128 runs the
 *                      fp32 backward instead).
 *                      ATTN_TF32 returns ATTN_ERR_UNSUPPORTED.
 * dq, dk and dv are written in full (keys no row attends get zero).  Each
 * element is computed by one thread block, without atomics, so repeated
 * calls give identical bits.  Needs D % 4 == 0 and 16-byte-aligned pointers,
 * else ATTN_ERR_UNSUPPORTED.  Scratch (8 bytes per (row, head); with
 * ATTN_BF16 also bf16 copies of q, dout, k and v) comes from the bound
 * workspace or the library pool (see the Data rule above).  q_seq == 0 is a
 * no-op; kv_seq == 0 zeroes
 * dq.  Errors otherwise as attn_forward, plus NULL out, dout, lse or
 * gradient pointers.
 */
ATTN_API int attn_backward(const float *q, const float *k, const float *v, const float *out, const float *dout,
                           const float *lse, float *dq, float *dk, float *dv, uint32_t q_seq, uint32_t kv_seq,
                           uint32_t num_heads, uint32_t num_kv_heads, uint32_t head_dim, attn_mask_t mask, attn_prec_t prec,
                           uint32_t window, attn_stream_t stream);

/*
 * Backward of attn_forward_rope: attn_backward's arguments plus the RoPE
 * table of that forward (rope_table, table_rows as there).  The gradients
 * are with respect to the unturned q and k: the plain gradient at the turned
 * q, k (turned into library scratch) is turned back.  out and lse are those
 * attn_forward_rope wrote.  Errors as attn_backward plus those of
 * attn_forward_rope's table checks.
 */
ATTN_API int attn_backward_rope(const float *q, const float *k, const float *v, const float *out, const float *dout,
                                const float *lse, float *dq, float *dk, float *dv, uint32_t q_seq, uint32_t kv_seq,
                                uint32_t num_heads, uint32_t num_kv_heads, uint32_t head_dim, attn_mask_t mask, attn_prec_t prec,
                                uint32_t window, const float *rope_table, uint32_t table_rows,
                                attn_stream_t stream);

/*
 * Cached single-token decode that allocates nothing and takes no workspace.
 * The shader pages have no counterpart to this entry point; it exists for
 * callers that cannot provide device scratch memory -- a plugin inside a
 * framework that owns every device allocation, or a serving loop that must
 * never call cudaMalloc (an allocation may synchronise the device and has no
 * latency bound).
 *
 * Arguments, layouts, the window rule and the result are those of
 * attn_decode_cached, minus the workspace.  In its place the library uses a
 * fixed 4 MiB array of device memory that is part of the library image: every
 * GPU that loads libattn_gqa.so holds it until the process exits.
 *   - Sizes whose split decode would need more than 4 MiB of scratch (about
 *     H * 2 * SMs / G * D * 4 bytes), shapes the split kernels do not cover
 *     (they take D in {64, 128} with gs = H/G a power of two up to 32) and
 *     pointers that are not 16-byte aligned return ATTN_ERR_UNSUPPORTED;
 *     nothing is launched.
 *   - All calls on a device share the one array, and it keeps what the last
 *     call left there; each call first clears the counters that must start
 *     at zero, on `stream`.  Calls that can overlap on the GPU (different
 *     streams without ordering between them) race on the array and give
 *     wrong results: order them on one stream.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.
 * Errors: as attn_decode_cached (INVALID_ARG for bad sizes or NULL pointers),
 * plus the UNSUPPORTED cases above.
 */
ATTN_API int attn_decode_cached_noalloc(const float *q, const float *k_cache, const float *v_cache,
                                        const uint32_t *kv_pos_dev, float *out, uint32_t num_heads,
                                        uint32_t num_kv_heads, uint32_t head_dim, uint32_t max_seq,
                                        attn_stream_t stream);

/*
 * Caller-owned scratch.  attn_set_workspace binds a DEVICE buffer of
 * workspace_bytes bytes (256-byte aligned) to the calling thread: from then
 * on every call this thread makes takes its temporary scratch from it, from
 * offset 0 each call, and allocates nothing; a call whose scratch does not
 * fit returns ATTN_ERR_INVALID_ARG before launching anything.
 * attn_set_workspace(NULL, 0) returns to the library pool.  The buffer is
 * read and written on the calls' streams: calls that share it must be
 * ordered on one stream (or synchronised), and it must stay allocated until
 * the last of them has run.  Errors: INVALID_ARG for a misaligned buffer.
 *
 * The queries give the bytes one call needs (0: none, or arguments the call
 * would reject); a bound workspace must hold the largest of the calls it
 * serves.
 *   attn_forward_workspace_bytes   attn_forward, attn_forward_window and, with
 *                                  rope != 0, attn_forward_rope
 *   attn_prefill_workspace_bytes   attn_prefill, attn_prefill_window and
 *                                  attn_prefill_paged (max_seq = page_rows *
 *                                  max_blocks)
 *   attn_backward_workspace_bytes  attn_backward and, with rope != 0,
 *                                  attn_backward_rope
 * Decode takes its workspace as an argument (attn_decode_workspace_bytes).
 */
ATTN_API int attn_set_workspace(void *workspace, size_t workspace_bytes);
ATTN_API size_t attn_forward_workspace_bytes(uint32_t q_seq, uint32_t kv_seq, uint32_t num_heads,
                                             uint32_t num_kv_heads, uint32_t head_dim, attn_mask_t mask,
                                             attn_prec_t prec, uint32_t window, int rope);
ATTN_API size_t attn_prefill_workspace_bytes(uint32_t n_queries, uint32_t n_heads, uint32_t n_kv_heads,
                                             uint32_t head_dim, uint32_t kv_dim, uint32_t max_seq,
                                             uint32_t start_pos, uint32_t q_base, attn_prec_t prec,
                                             uint32_t window);
ATTN_API size_t attn_backward_workspace_bytes(uint32_t q_seq, uint32_t kv_seq, uint32_t num_heads,
                                              uint32_t num_kv_heads, uint32_t head_dim, attn_prec_t prec, int rope);

/*
 * The library pool on the current device (the scratch of calls made without
 * a bound workspace): attn_scratch_reserved_bytes is the memory it holds;
 * attn_scratch_peak_bytes the most it has had in use at once since the last
 * reset (reset != 0 resets it to 0 after reading); attn_release_scratch
 * returns the reserved memory not in use (call it after synchronising the
 * streams that used the pool).  Errors: ATTN_ERR_CUDA if the pool is not
 * available.
 */
ATTN_API size_t attn_scratch_reserved_bytes(void);
ATTN_API size_t attn_scratch_peak_bytes(int reset);
ATTN_API int attn_release_scratch(void);

/*
 * Waits for `stream`, then returns and clears the current device's status
 * word: ATTN_OK, or the largest code a kernel recorded since the last read
 * (ATTN_ERR_INVALID_ARG for a decode kv_pos past the cache, ATTN_ERR_TIMEOUT
 * for a bounded device wait that gave up; its kernel returned early and its
 * output is not valid).  Returns ATTN_ERR_CUDA if the stream or the read
 * failed.
 */
ATTN_API int attn_get_status(attn_stream_t stream);

/*
 * Failure-path self test.  Launches one CTA that waits, with the bounded wait
 * every kernel of this library uses, on a barrier that nothing completes, but
 * with a limit of timeout_us microseconds (1 .. 1000000) instead of the usual
 * one second.  The wait gives up, the kernel records ATTN_ERR_TIMEOUT in the
 * device status word and returns normally: no fault, no hang, and the CUDA
 * context stays usable.  Read the outcome with attn_get_status.  Errors:
 * INVALID_ARG for a timeout outside the range.
 */
ATTN_API int attn_selftest_wait_timeout(uint32_t timeout_us, attn_stream_t stream);

/* Static, human-readable name of a status code. */
ATTN_API const char *attn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GQA_H */
