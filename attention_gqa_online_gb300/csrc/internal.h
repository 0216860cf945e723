// internal.h -- launchers shared between the C-ABI layer (api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn_gqa.h"

namespace attn {

// One flash-style attention launch.  Rows are (query i, head h) pairs; the
// query, key and value pointers already include every batch offset (q_base),
// so query 0 of the call is at q[0].
struct FlashArgs {
  const float* q;
  const float* k;
  const float* v;
  float* out;
  float* lse;                 // [n_q, H, 2] or nullptr
  long long q_row_stride;     // floats between consecutive query rows
  long long out_row_stride;   // floats between consecutive output rows
  long long kv_row_stride;    // floats between consecutive key/value rows
  int n_q, H, G, D;
  // Window of query i: keys [lo_i, n_i) with
  //   n_i = min(base_pos + i + 1, cap)  if causal
  //   n_i = n_all                       otherwise
  //   lo_i = first_key(n_i, window)
  int causal;
  long long base_pos;
  int cap;
  int n_all;
  int window;                 // sliding window length, 0 = none
  float scale;                // multiplies q . k
  // Decode through the generic kernel: when set, base_pos is read from
  // *kv_pos_dev on the device (n_q == 1, causal, cap = max_seq).
  const uint32_t* kv_pos_dev;
  unsigned* status;           // device status word
  // Paged K/V when block_table != nullptr: k and v are pools of num_pages
  // pages of page_rows rows, and key row t is pool row
  // block_table[t / page_rows] * page_rows + t % page_rows (see paged_row).
  const uint32_t* block_table;
  int page_rows;
  int num_pages;
  // Rotary position embedding when rope != nullptr: the [positions][D]
  // cos | sin table of launch_rope_table; q of query i is turned at position
  // base_pos + i and k of key row t at position t before the scores.
  const float* rope;
};

// Pool row of logical key row t in a paged cache, or -1 (and ATTN_ERR_INVALID_ARG
// in the status word) when the block table names a page outside the pool.
__device__ __forceinline__ long long paged_row(const uint32_t* table, int page_rows, int num_pages, int t,
                                               unsigned* status) {
  const uint32_t page = table[t / page_rows];
  if (page >= (uint32_t)num_pages) {
    atomicMax(status, (unsigned)ATTN_ERR_INVALID_ARG);
    return -1;
  }
  return (long long)page * page_rows + t % page_rows;
}

// First key of a window that ends at n (exclusive) under a sliding window of
// `window` keys (0 = unlimited): the window keeps the last `window` positions.
// Both bounds are non-decreasing in n, so over a block of consecutive queries
// the first query has the smallest bounds and the last the largest.
__host__ __device__ inline int first_key(int n, int window) { return (window > 0 && n > window) ? n - window : 0; }

// Launches `kernel` with programmatic stream serialization allowed, so it may
// start while the previous kernel in `s` finishes (the kernel itself waits
// for that kernel before touching global memory).
cudaError_t launch_pdl(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args);

// A non-blocking stream per device, created once, for work the library runs
// beside the caller's stream.
cudaStream_t side_stream();
// Runs two independent kernels with the same arguments concurrently: k1 on
// `s`, k2 on the side stream forked from `s` and joined back into it, so
// that work queued on `s` afterwards follows both.  Returns an ATTN_ status.
int launch_forked(cudaStream_t s, const void* k1, dim3 g1, size_t smem1, const void* k2, dim3 g2, size_t smem2,
                  dim3 block, void** args);

// Raises a kernel's dynamic shared memory limit to `bytes` on the current
// device; the attribute is set once per (kernel, device).
bool set_smem_limit(const void* kernel, size_t bytes);

// Encodes a tiled TMA tensor map.  dims[0] is the innermost (contiguous)
// extent in elements; strides_bytes has rank-1 entries (dims 1..rank-1);
// box is the tile copied per request.  fp32 or bf16 elements; out-of-bounds
// elements read as zero.  Swizzle: none, 128-byte rows with 16-byte chunks
// permuted, or 128-byte rows with 32-byte chunks permuted.
enum { kSwizzleNone = 0, kSwizzle128 = 1, kSwizzle128Atom32 = 2 };
bool make_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
               const uint32_t* box, bool bf16, int swizzle);

// K/V operand pre-pass of the tensor-core kernels (kv_prep.cu).  One block
// per (128-key tile T in [tile0, n_tiles), kv head g); rows at or past
// rows_end are not written.  Paged caches through table (as FlashArgs), RoPE
// on K through rope (the table of launch_rope_table).  out0 = K as fp16 times
// 2^(14 - E_T) (E_T: binary exponent of the tile's largest magnitude, per kv
// head), kfac[T * G + g] = 2^(E_T - 14); if out1 is set, out1 = V as bf16.
// Outputs keep the inputs' layout: rows of `stride` elements, head g at g*D.
struct PrepArgs {
  const float* k;
  const float* v;
  uint16_t* out0;
  uint16_t* out1;
  float* kfac;
  long long stride;
  int G, D;
  int tile0, n_tiles;
  long long rows_end;
  const float* rope;
  const uint32_t* table;
  int page_rows, num_pages;
  unsigned* status;
};
cudaError_t launch_kv_prep(const PrepArgs& p, cudaStream_t s);

// fp32 CUDA-core flash kernel; any 1 <= D <= 128.
int launch_flash_simt(const FlashArgs& a, cudaStream_t s);

// tcgen05 tensor-core flash kernel (prec = ATTN_TF32 or ATTN_BF16).
bool flash_tc_supported(const FlashArgs& a, int prec);
int launch_flash_tc(const FlashArgs& a, int prec, cudaStream_t s);
// bf16-operand kernel (flash_bf16.cu); the caller has checked
// flash_tc_supported(a, ATTN_BF16).
int launch_flash_bf16(const FlashArgs& a, cudaStream_t s);
// SM count of the current device (0 if it cannot be read).
int device_sm_count();

// Backward of the forward attention (fp32, CUDA cores).  Contiguous
// layouts: q, out, dout, dq [n_q][H*D]; k, v, dk, dv [n_kv][G*D]; lse
// [n_q][H][2] as the forward wrote it.  Windows follow the forward: query i
// sees keys [first_key(n_i, window), n_i) with n_i = min(i + 1, n_kv) if
// causal, else n_kv.  Needs n_kv >= 1, D % 4 == 0, 1 <= D <= 128 and
// 16-byte-aligned pointers (the caller checks).
struct BwdArgs {
  const float* q;
  const float* k;
  const float* v;
  const float* out;
  const float* dout;
  const float* lse;
  float* dq;
  float* dk;
  float* dv;
  int n_q, n_kv, H, G, D;
  int causal;
  int window;
  float scale;
  unsigned* status;  // device status word (bounded waits of the tensor-core kernels)
};
int launch_backward_simt(const BwdArgs& a, cudaStream_t s);
// The backward's first pass: delta[i*H + h] = dout . out and l2[i*H + h] =
// (lse0 + lse1) * log2(e) for every (row, head).
cudaError_t launch_bwd_prep(const BwdArgs& a, float* delta, float* l2, cudaStream_t s);
// tcgen05 backward with bf16 operands (bwd_tc.cu): D in {64, 128}, H/G a
// power of two up to 128, 16-byte-aligned pointers.
bool backward_bf16_supported(const BwdArgs& a);
int launch_backward_bf16(const BwdArgs& a, cudaStream_t s);

// RoPE helpers (rope.cu): fill table[max_pos][D] (cos of the D/2 pairs, then
// their sin; angles p * base^(-2d/D) in fp64), and write x ([rows][G*D], G
// heads, row t at position t) turned by the table (sgn = 1) or turned back
// (sgn = -1) into out (which may be x).  D % 8 == 0 for launch_rope_k;
// 16-byte-aligned pointers.
int launch_rope_table(float* table, int max_pos, int D, double base, cudaStream_t s);
cudaError_t launch_rope_k(const float* k, float* out, const float* table, long long rows, int G, int D, cudaStream_t s,
                          float sgn = 1.f);

// Split-KV decode.
struct DecodeArgs {
  const float* q;
  const float* k_cache;
  const float* v_cache;
  const uint32_t* kv_pos_dev;
  float* out;
  int H, G, D, max_seq;
  int window;  // sliding window length, 0 = none: keys [first_key(n, window), n)
  int kv_div;  // head groups per kv head (set by launch_decode_split)
  // Append (k_new != nullptr): the new token's K and V rows ([G*D] each) are
  // written into cache row kv_pos before it is attended.
  const float* k_new;
  const float* v_new;
  // Paged caches (block_table != nullptr): as FlashArgs; page_rows % 32 == 0.
  const uint32_t* block_table;
  int page_rows;
  int num_pages;
  void* workspace;
  unsigned* status;
};

// Head groups of the split decode (one CTA column each): G, or more when a kv
// head's query heads are split over several CTAs.
int decode_groups(int H, int G, int D);
// Number of KV splits per head group for `groups` groups on a device with
// sm_count SMs.
int decode_splits(int groups, int max_seq, int sm_count);
// Workspace bytes the split decode needs (0 if the fast path does not apply).
size_t decode_workspace_bytes(int H, int G, int D, int max_seq, int sm_count);
// True if the split-KV kernels handle these sizes (else the generic kernel runs).
bool decode_split_supported(int H, int G, int D);
int launch_decode_split(const DecodeArgs& a, int splits, cudaStream_t s);
// Writes k_new / v_new ([G*D] each) into row *kv_pos_dev of [max_seq][G*D]
// caches (nothing, and ATTN_ERR_INVALID_ARG in the status word, when the
// position is past the cache).
cudaError_t launch_cache_append(const float* k_new, const float* v_new, float* k_cache, float* v_cache,
                                const uint32_t* kv_pos_dev, int kv_dim, int max_seq, unsigned* status, cudaStream_t s);
// Bytes at the start of a split-decode workspace that must be zero when a
// call begins (the per-head-group arrival counters).
size_t decode_ticket_bytes(int groups);

// Device address of the current device's status word (nullptr on failure).
unsigned* device_status_word();

// Temporary scratch memory of a call.  With a workspace bound to the calling
// thread (scratch_bind; attn_set_workspace), allocations are carved from it
// in order, each start rounded up to 256 bytes, from offset 0 at every
// scratch_begin_call(); otherwise they are stream-ordered allocations from a
// library-owned pool on the current device that keeps freed memory reserved
// between calls.  scratch_free of workspace memory does nothing.
inline size_t scratch_round(size_t b) { return (b + 255) & ~size_t(255); }
void scratch_bind(void* ws, size_t bytes);
bool scratch_bound(size_t* bytes);
void scratch_begin_call();
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t s);
cudaError_t scratch_free(void* p, cudaStream_t s);
// The pool's reserved bytes (which = 0) or its high-water mark of bytes in
// use (which = 1; reset to 0 afterwards if `reset`); trimming returns the
// reserved memory that is not in use.
size_t scratch_pool_stat(int which, bool reset);
bool scratch_trim();

// Scratch bytes each launcher requests (a sum of scratch_round'ed sizes; 0
// when it needs none).  The launchers allocate exactly these.
size_t flash_tc_scratch_bytes(const FlashArgs& a);
size_t flash_bf16_scratch_bytes(const FlashArgs& a);
size_t flash_simt_scratch_bytes(const FlashArgs& a);
size_t backward_simt_scratch_bytes(const BwdArgs& a);
size_t backward_bf16_scratch_bytes(const BwdArgs& a);

}  // namespace attn
