// api.cu -- the C ABI of libattn_gqa.so (declared in include/attn_gqa.h):
// argument validation, kernel selection, and the device status word.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/attn_gqa.h"
#include "common.cuh"
#include "internal.h"

namespace attn {

__device__ unsigned int g_status_word = 0;

namespace {

constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
std::mutex g_mu;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

// Device address of this device's status word (looked up once per device).
unsigned* status_ptr() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

bool heads_ok(uint32_t H, uint32_t G, uint32_t D) {
  return H >= 1 && G >= 1 && H % G == 0 && D >= 1 && D <= 128 && H <= (1u << 20);
}

// A window longer than any key range is no limit at all.
int window_arg(uint32_t window) { return window > 0x7fffffffu ? 0x7fffffff : (int)window; }

bool valid_prec(int prec) { return prec == ATTN_FP32 || prec == ATTN_TF32 || prec == ATTN_BF16; }

// A tensor-core call that runs on the fp32 kernel instead (see run_flash)
// needs that kernel's scratch, so a tensor-core precision reports the larger.
size_t flash_scratch_bytes(const FlashArgs& a, int prec) {
  const size_t simt = flash_simt_scratch_bytes(a);
  if (prec == ATTN_FP32) return simt;
  const size_t tc = prec == ATTN_BF16 ? flash_bf16_scratch_bytes(a) : flash_tc_scratch_bytes(a);
  return tc > simt ? tc : simt;
}

// A workspace bound to this thread must hold the call's whole scratch; this
// is checked before anything is launched.
bool workspace_too_small(size_t need) {
  size_t have = 0;
  return scratch_bound(&have) && need > have;
}

int run_flash(const FlashArgs& a, int prec, cudaStream_t s) {
  scratch_begin_call();
  // The tensor-core precisions refuse only head_dim outside {64, 128}.  A
  // layout their kernels do not take (pointers not 16-byte aligned, row
  // strides off the TMA granule, more than 128 query heads per kv head, pages
  // the tiles cannot follow) runs on the fp32 kernel, whose results lie within
  // every precision's bound.
  if (prec != ATTN_FP32 && a.D != 64 && a.D != 128) return ATTN_ERR_UNSUPPORTED;
  if (workspace_too_small(flash_scratch_bytes(a, prec))) return ATTN_ERR_INVALID_ARG;
  if (prec != ATTN_FP32 && !flash_tc_supported(a, prec)) prec = ATTN_FP32;
  if (prec == ATTN_FP32) return launch_flash_simt(a, s);
  return launch_flash_tc(a, prec, s);
}

// Host-only stand-in for present K/V in size queries (never dereferenced).
const float kPresent = 0.f;

}  // namespace

unsigned* device_status_word() { return status_ptr(); }
int device_sm_count() { return sm_count(); }

}  // namespace attn

using namespace attn;

extern "C" int attn_forward_window(const float* q, const float* k, const float* v, float* out, float* lse,
                                   uint32_t q_seq, uint32_t kv_seq, uint32_t num_heads, uint32_t num_kv_heads,
                                   uint32_t head_dim, attn_mask_t mask, attn_prec_t prec, uint32_t window, attn_stream_t stream) {
  if (!heads_ok(num_heads, num_kv_heads, head_dim) || !valid_prec(prec)) return ATTN_ERR_INVALID_ARG;
  if (mask != ATTN_CAUSAL && mask != ATTN_FULL && mask != ATTN_CROSS) return ATTN_ERR_INVALID_ARG;
  if (mask != ATTN_CROSS && kv_seq != q_seq) return ATTN_ERR_INVALID_ARG;
  if (q_seq > 0x7fffffffu || kv_seq > 0x7fffffffu) return ATTN_ERR_INVALID_ARG;
  if (q_seq == 0) return ATTN_OK;
  if (q == nullptr || out == nullptr || (kv_seq > 0 && (k == nullptr || v == nullptr))) return ATTN_ERR_INVALID_ARG;
  FlashArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.q_row_stride = (long long)num_heads * head_dim;
  a.out_row_stride = a.q_row_stride;
  a.kv_row_stride = (long long)num_kv_heads * head_dim;
  a.n_q = (int)q_seq;
  a.H = (int)num_heads;
  a.G = (int)num_kv_heads;
  a.D = (int)head_dim;
  a.causal = (mask == ATTN_CAUSAL);
  a.base_pos = 0;
  a.cap = (int)kv_seq;
  a.n_all = (int)kv_seq;
  a.window = window_arg(window);
  a.scale = 1.0f / sqrtf((float)head_dim);
  a.kv_pos_dev = nullptr;
  a.status = status_ptr();
  if (a.status == nullptr) return ATTN_ERR_CUDA;
  // An empty key set is handled by the same kernels (no tiles, zero rows).
  return run_flash(a, prec, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int attn_rope_table(float* table, uint32_t max_pos, uint32_t head_dim, double base, attn_stream_t stream) {
  if (head_dim == 0 || head_dim > 128 || head_dim % 2 != 0 || !(base > 1.0) || !std::isfinite(base))
    return ATTN_ERR_INVALID_ARG;
  if ((uint64_t)max_pos * head_dim > 0x7fffffffu) return ATTN_ERR_INVALID_ARG;
  if (max_pos == 0) return ATTN_OK;
  if (table == nullptr) return ATTN_ERR_INVALID_ARG;
  return launch_rope_table(table, (int)max_pos, (int)head_dim, base, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int attn_forward_rope(const float* q, const float* k, const float* v, float* out, float* lse,
                                 uint32_t q_seq, uint32_t kv_seq, uint32_t num_heads, uint32_t num_kv_heads,
                                 uint32_t head_dim, attn_mask_t mask, attn_prec_t prec, uint32_t window, const float* rope_table,
                                 uint32_t table_rows, attn_stream_t stream) {
  if (!heads_ok(num_heads, num_kv_heads, head_dim) || !valid_prec(prec)) return ATTN_ERR_INVALID_ARG;
  if (mask != ATTN_CAUSAL && mask != ATTN_FULL && mask != ATTN_CROSS) return ATTN_ERR_INVALID_ARG;
  if (mask != ATTN_CROSS && kv_seq != q_seq) return ATTN_ERR_INVALID_ARG;
  if (q_seq > 0x7fffffffu || kv_seq > 0x7fffffffu) return ATTN_ERR_INVALID_ARG;
  if (head_dim % 2 != 0 || table_rows < q_seq || table_rows < kv_seq) return ATTN_ERR_INVALID_ARG;
  if (q_seq == 0) return ATTN_OK;
  if (q == nullptr || out == nullptr || rope_table == nullptr || (kv_seq > 0 && (k == nullptr || v == nullptr)))
    return ATTN_ERR_INVALID_ARG;
  // The table is read as float4 groups of pairs on every path.
  if (head_dim % 8 != 0 || (reinterpret_cast<uintptr_t>(rope_table) % 16) != 0) return ATTN_ERR_UNSUPPORTED;
  FlashArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.q_row_stride = (long long)num_heads * head_dim;
  a.out_row_stride = a.q_row_stride;
  a.kv_row_stride = (long long)num_kv_heads * head_dim;
  a.n_q = (int)q_seq;
  a.H = (int)num_heads;
  a.G = (int)num_kv_heads;
  a.D = (int)head_dim;
  a.causal = (mask == ATTN_CAUSAL);
  a.base_pos = 0;
  a.cap = (int)kv_seq;
  a.n_all = (int)kv_seq;
  a.window = window_arg(window);
  a.scale = 1.0f / sqrtf((float)head_dim);
  a.kv_pos_dev = nullptr;
  a.rope = rope_table;
  a.status = status_ptr();
  if (a.status == nullptr) return ATTN_ERR_CUDA;
  return run_flash(a, prec, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int attn_forward(const float* q, const float* k, const float* v, float* out, float* lse,
                            uint32_t q_seq, uint32_t kv_seq, uint32_t num_heads, uint32_t num_kv_heads,
                            uint32_t head_dim, attn_mask_t mask, attn_prec_t prec, attn_stream_t stream) {
  return attn_forward_window(q, k, v, out, lse, q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask, prec, 0,
                             stream);
}

extern "C" size_t attn_decode_workspace_bytes(uint32_t num_heads, uint32_t num_kv_heads, uint32_t head_dim,
                                              uint32_t max_seq) {
  if (!heads_ok(num_heads, num_kv_heads, head_dim) || max_seq == 0 || max_seq > 0x7fffffffu) return 0;
  const int sms = sm_count();
  if (sms <= 0) return 0;
  const size_t b = decode_workspace_bytes((int)num_heads, (int)num_kv_heads, (int)head_dim, (int)max_seq, sms);
  return b > 0 ? b : 256;  // the generic path needs none; report a token size
}

extern "C" int attn_decode_cached_window(const float* q, const float* k_cache, const float* v_cache,
                                         const uint32_t* kv_pos_dev, float* out, uint32_t num_heads,
                                         uint32_t num_kv_heads, uint32_t head_dim, uint32_t max_seq,
                                         void* workspace, size_t workspace_bytes, uint32_t window,
                                         attn_stream_t stream) {
  if (!heads_ok(num_heads, num_kv_heads, head_dim) || max_seq == 0 || max_seq > 0x7fffffffu)
    return ATTN_ERR_INVALID_ARG;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || kv_pos_dev == nullptr || out == nullptr)
    return ATTN_ERR_INVALID_ARG;
  const int H = (int)num_heads, G = (int)num_kv_heads, D = (int)head_dim, ms = (int)max_seq;
  unsigned* st = status_ptr();
  if (st == nullptr) return ATTN_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool aligned = ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
                         reinterpret_cast<uintptr_t>(v_cache)) % 16) == 0;
  if (decode_split_supported(H, G, D) && aligned) {
    const int sms = sm_count();
    if (sms <= 0) return ATTN_ERR_CUDA;
    const size_t need = decode_workspace_bytes(H, G, D, ms, sms);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % 16) != 0)
      return ATTN_ERR_INVALID_ARG;
    DecodeArgs d{};
    d.q = q;
    d.k_cache = k_cache;
    d.v_cache = v_cache;
    d.kv_pos_dev = kv_pos_dev;
    d.out = out;
    d.H = H;
    d.G = G;
    d.D = D;
    d.max_seq = ms;
    d.window = window_arg(window);
    d.workspace = workspace;
    d.status = st;
    return launch_decode_split(d, decode_splits(decode_groups(H, G, D), ms, sms), s);
  }
  // Other shapes: the generic flash kernel with one query row whose causal
  // position is read from kv_pos_dev.
  FlashArgs a{};
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.out = out;
  a.lse = nullptr;
  a.q_row_stride = (long long)H * D;
  a.out_row_stride = a.q_row_stride;
  a.kv_row_stride = (long long)G * D;
  a.n_q = 1;
  a.H = H;
  a.G = G;
  a.D = D;
  a.causal = 1;
  a.base_pos = 0;
  a.cap = ms;
  a.n_all = ms;
  a.window = window_arg(window);
  a.scale = 1.0f / sqrtf((float)D);
  a.kv_pos_dev = kv_pos_dev;
  a.status = st;
  return launch_flash_simt(a, s);
}

extern "C" int attn_decode_append(const float* q, const float* k_new, const float* v_new, float* k_cache,
                                  float* v_cache, const uint32_t* kv_pos_dev, float* out, uint32_t num_heads,
                                  uint32_t num_kv_heads, uint32_t head_dim, uint32_t max_seq, void* workspace,
                                  size_t workspace_bytes, attn_stream_t stream) {
  if (!heads_ok(num_heads, num_kv_heads, head_dim) || max_seq == 0 || max_seq > 0x7fffffffu)
    return ATTN_ERR_INVALID_ARG;
  if (q == nullptr || k_new == nullptr || v_new == nullptr || k_cache == nullptr || v_cache == nullptr ||
      kv_pos_dev == nullptr || out == nullptr)
    return ATTN_ERR_INVALID_ARG;
  const int H = (int)num_heads, G = (int)num_kv_heads, D = (int)head_dim, ms = (int)max_seq;
  unsigned* st = status_ptr();
  if (st == nullptr) return ATTN_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool aligned = ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
                         reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(k_new) |
                         reinterpret_cast<uintptr_t>(v_new)) % 16) == 0;
  if (decode_split_supported(H, G, D) && aligned) {
    // The split decode writes the row itself (the split ending at kv_pos).
    const int sms = sm_count();
    if (sms <= 0) return ATTN_ERR_CUDA;
    const size_t need = decode_workspace_bytes(H, G, D, ms, sms);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % 16) != 0)
      return ATTN_ERR_INVALID_ARG;
    DecodeArgs d{};
    d.q = q;
    d.k_cache = k_cache;
    d.v_cache = v_cache;
    d.kv_pos_dev = kv_pos_dev;
    d.out = out;
    d.H = H;
    d.G = G;
    d.D = D;
    d.max_seq = ms;
    d.k_new = k_new;
    d.v_new = v_new;
    d.workspace = workspace;
    d.status = st;
    return launch_decode_split(d, decode_splits(decode_groups(H, G, D), ms, sms), s);
  }
  if (launch_cache_append(k_new, v_new, k_cache, v_cache, kv_pos_dev, G * D, ms, st, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return attn_decode_cached(q, k_cache, v_cache, kv_pos_dev, out, num_heads, num_kv_heads, head_dim, max_seq,
                            workspace, workspace_bytes, stream);
}

extern "C" int attn_decode_cached(const float* q, const float* k_cache, const float* v_cache,
                                  const uint32_t* kv_pos_dev, float* out, uint32_t num_heads,
                                  uint32_t num_kv_heads, uint32_t head_dim, uint32_t max_seq, void* workspace,
                                  size_t workspace_bytes, attn_stream_t stream) {
  return attn_decode_cached_window(q, k_cache, v_cache, kv_pos_dev, out, num_heads, num_kv_heads, head_dim, max_seq,
                                   workspace, workspace_bytes, 0, stream);
}

extern "C" int attn_prefill_window(const float* q_batch, const float* k_cache, const float* v_cache,
                                   float* out_batch, uint32_t n_queries, uint32_t n_heads, uint32_t n_kv_heads,
                                   uint32_t head_dim, uint32_t kv_dim, uint32_t max_seq, float scale,
                                   uint32_t start_pos, uint32_t q_stride, uint32_t out_stride, uint32_t q_base,
                                   attn_prec_t prec, uint32_t window, attn_stream_t stream) {
  if (!heads_ok(n_heads, n_kv_heads, head_dim) || !valid_prec(prec)) return ATTN_ERR_INVALID_ARG;
  if ((uint64_t)kv_dim < (uint64_t)n_kv_heads * head_dim) return ATTN_ERR_INVALID_ARG;
  if ((uint64_t)q_stride < (uint64_t)n_heads * head_dim || (uint64_t)out_stride < (uint64_t)n_heads * head_dim)
    return ATTN_ERR_INVALID_ARG;
  if ((uint64_t)start_pos + q_base + n_queries > max_seq || max_seq > 0x7fffffffu) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (n_queries == 0) return ATTN_OK;
  if (q_batch == nullptr || k_cache == nullptr || v_cache == nullptr || out_batch == nullptr)
    return ATTN_ERR_INVALID_ARG;
  FlashArgs a{};
  a.q = q_batch + (size_t)q_base * q_stride;
  a.k = k_cache;
  a.v = v_cache;
  a.out = out_batch + (size_t)q_base * out_stride;
  a.lse = nullptr;
  a.q_row_stride = q_stride;
  a.out_row_stride = out_stride;
  a.kv_row_stride = kv_dim;
  a.n_q = (int)n_queries;
  a.H = (int)n_heads;
  a.G = (int)n_kv_heads;
  a.D = (int)head_dim;
  a.causal = 1;
  a.base_pos = (long long)start_pos + q_base;
  a.cap = (int)max_seq;
  a.n_all = (int)max_seq;
  a.window = window_arg(window);
  a.scale = scale;
  a.kv_pos_dev = nullptr;
  a.status = status_ptr();
  if (a.status == nullptr) return ATTN_ERR_CUDA;
  return run_flash(a, prec, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int attn_prefill(const float* q_batch, const float* k_cache, const float* v_cache, float* out_batch,
                            uint32_t n_queries, uint32_t n_heads, uint32_t n_kv_heads, uint32_t head_dim,
                            uint32_t kv_dim, uint32_t max_seq, float scale, uint32_t start_pos, uint32_t q_stride,
                            uint32_t out_stride, uint32_t q_base, attn_prec_t prec, attn_stream_t stream) {
  return attn_prefill_window(q_batch, k_cache, v_cache, out_batch, n_queries, n_heads, n_kv_heads, head_dim, kv_dim,
                             max_seq, scale, start_pos, q_stride, out_stride, q_base, prec, 0, stream);
}

// Paged-cache checks shared by the two paged entry points: the logical
// capacity page_rows * max_blocks and the pool page_rows * num_pages rows must
// fit in an int.
static bool paged_sizes_ok(uint32_t page_rows, uint32_t num_pages, uint32_t max_blocks) {
  return page_rows >= 1 && num_pages >= 1 && max_blocks >= 1 &&
         (uint64_t)page_rows * max_blocks <= 0x7fffffffu && (uint64_t)page_rows * num_pages <= 0x7fffffffu;
}

extern "C" int attn_decode_paged(const float* q, const float* k_pages, const float* v_pages,
                                 const uint32_t* block_table, const uint32_t* kv_pos_dev, float* out,
                                 uint32_t num_heads, uint32_t num_kv_heads, uint32_t head_dim, uint32_t page_rows,
                                 uint32_t num_pages, uint32_t max_blocks, void* workspace, size_t workspace_bytes,
                                 uint32_t window, attn_stream_t stream) {
  if (!heads_ok(num_heads, num_kv_heads, head_dim) || !paged_sizes_ok(page_rows, num_pages, max_blocks))
    return ATTN_ERR_INVALID_ARG;
  if (q == nullptr || k_pages == nullptr || v_pages == nullptr || block_table == nullptr || kv_pos_dev == nullptr ||
      out == nullptr)
    return ATTN_ERR_INVALID_ARG;
  const int H = (int)num_heads, G = (int)num_kv_heads, D = (int)head_dim;
  const int ms = (int)(page_rows * max_blocks);
  unsigned* st = status_ptr();
  if (st == nullptr) return ATTN_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool aligned = ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_pages) |
                         reinterpret_cast<uintptr_t>(v_pages)) % 16) == 0;
  if (decode_split_supported(H, G, D) && aligned && page_rows % 32 == 0) {
    const int sms = sm_count();
    if (sms <= 0) return ATTN_ERR_CUDA;
    const size_t need = decode_workspace_bytes(H, G, D, ms, sms);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % 16) != 0)
      return ATTN_ERR_INVALID_ARG;
    DecodeArgs d{};
    d.q = q;
    d.k_cache = k_pages;
    d.v_cache = v_pages;
    d.kv_pos_dev = kv_pos_dev;
    d.out = out;
    d.H = H;
    d.G = G;
    d.D = D;
    d.max_seq = ms;
    d.window = window_arg(window);
    d.block_table = block_table;
    d.page_rows = (int)page_rows;
    d.num_pages = (int)num_pages;
    d.workspace = workspace;
    d.status = st;
    return launch_decode_split(d, decode_splits(decode_groups(H, G, D), ms, sms), s);
  }
  FlashArgs a{};
  a.q = q;
  a.k = k_pages;
  a.v = v_pages;
  a.out = out;
  a.lse = nullptr;
  a.q_row_stride = (long long)H * D;
  a.out_row_stride = a.q_row_stride;
  a.kv_row_stride = (long long)G * D;
  a.n_q = 1;
  a.H = H;
  a.G = G;
  a.D = D;
  a.causal = 1;
  a.base_pos = 0;
  a.cap = ms;
  a.n_all = ms;
  a.window = window_arg(window);
  a.scale = 1.0f / sqrtf((float)D);
  a.kv_pos_dev = kv_pos_dev;
  a.status = st;
  a.block_table = block_table;
  a.page_rows = (int)page_rows;
  a.num_pages = (int)num_pages;
  return launch_flash_simt(a, s);
}

extern "C" int attn_prefill_paged(const float* q_batch, const float* k_pages, const float* v_pages,
                                  const uint32_t* block_table, float* out_batch, uint32_t n_queries, uint32_t n_heads,
                                  uint32_t n_kv_heads, uint32_t head_dim, uint32_t kv_dim, uint32_t page_rows,
                                  uint32_t num_pages, uint32_t max_blocks, float scale, uint32_t start_pos,
                                  uint32_t q_stride, uint32_t out_stride, uint32_t q_base, attn_prec_t prec, uint32_t window,
                                  attn_stream_t stream) {
  if (!heads_ok(n_heads, n_kv_heads, head_dim) || !valid_prec(prec)) return ATTN_ERR_INVALID_ARG;
  if (!paged_sizes_ok(page_rows, num_pages, max_blocks)) return ATTN_ERR_INVALID_ARG;
  const uint64_t max_seq = (uint64_t)page_rows * max_blocks;
  if ((uint64_t)kv_dim < (uint64_t)n_kv_heads * head_dim) return ATTN_ERR_INVALID_ARG;
  if ((uint64_t)q_stride < (uint64_t)n_heads * head_dim || (uint64_t)out_stride < (uint64_t)n_heads * head_dim)
    return ATTN_ERR_INVALID_ARG;
  if ((uint64_t)start_pos + q_base + n_queries > max_seq) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (n_queries == 0) return ATTN_OK;
  if (q_batch == nullptr || k_pages == nullptr || v_pages == nullptr || block_table == nullptr || out_batch == nullptr)
    return ATTN_ERR_INVALID_ARG;
  FlashArgs a{};
  a.q = q_batch + (size_t)q_base * q_stride;
  a.k = k_pages;
  a.v = v_pages;
  a.out = out_batch + (size_t)q_base * out_stride;
  a.lse = nullptr;
  a.q_row_stride = q_stride;
  a.out_row_stride = out_stride;
  a.kv_row_stride = kv_dim;
  a.n_q = (int)n_queries;
  a.H = (int)n_heads;
  a.G = (int)n_kv_heads;
  a.D = (int)head_dim;
  a.causal = 1;
  a.base_pos = (long long)start_pos + q_base;
  a.cap = (int)max_seq;
  a.n_all = (int)max_seq;
  a.window = window_arg(window);
  a.scale = scale;
  a.kv_pos_dev = nullptr;
  a.status = status_ptr();
  if (a.status == nullptr) return ATTN_ERR_CUDA;
  a.block_table = block_table;
  a.page_rows = (int)page_rows;
  a.num_pages = (int)num_pages;
  return run_flash(a, prec, reinterpret_cast<cudaStream_t>(stream));
}

// Scratch of one backward call: q and k turned (RoPE), then the backward's own.
static size_t backward_scratch_bytes(const BwdArgs& a, int prec, bool rope) {
  const size_t turned = rope ? scratch_round(((size_t)a.n_q * a.H + (size_t)a.n_kv * a.G) * a.D * sizeof(float)) : 0;
  if (a.n_kv == 0) return 0;
  const size_t simt = backward_simt_scratch_bytes(a);
  if (prec != ATTN_BF16) return turned + simt;
  // A bf16 call that runs on the fp32 backward (see backward_impl) needs that
  // kernel's scratch: report the larger.
  const size_t tc = backward_bf16_scratch_bytes(a);
  return turned + (tc > simt ? tc : simt);
}

// The backward behind attn_backward and attn_backward_rope; rope_table (or
// nullptr) turns q and k first and the gradients back afterwards.
static int backward_impl(const float* q, const float* k, const float* v, const float* out, const float* dout,
                         const float* lse, float* dq, float* dk, float* dv, uint32_t q_seq, uint32_t kv_seq,
                         uint32_t num_heads, uint32_t num_kv_heads, uint32_t head_dim, int mask, int prec,
                         uint32_t window, const float* rope_table, uint32_t table_rows, attn_stream_t stream) {
  if (!heads_ok(num_heads, num_kv_heads, head_dim) || !valid_prec(prec)) return ATTN_ERR_INVALID_ARG;
  if (mask != ATTN_CAUSAL && mask != ATTN_FULL && mask != ATTN_CROSS) return ATTN_ERR_INVALID_ARG;
  if (mask != ATTN_CROSS && kv_seq != q_seq) return ATTN_ERR_INVALID_ARG;
  if (q_seq > 0x7fffffffu || kv_seq > 0x7fffffffu) return ATTN_ERR_INVALID_ARG;
  const bool rope = rope_table != nullptr;
  if (rope && (head_dim % 2 != 0 || table_rows < q_seq || table_rows < kv_seq)) return ATTN_ERR_INVALID_ARG;
  if (q_seq == 0) return ATTN_OK;
  if (q == nullptr || dout == nullptr || dq == nullptr || out == nullptr || lse == nullptr) return ATTN_ERR_INVALID_ARG;
  if (kv_seq > 0 && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (prec == ATTN_TF32) return ATTN_ERR_UNSUPPORTED;
  const uintptr_t al = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out) |
                       reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                       reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv) |
                       reinterpret_cast<uintptr_t>(rope_table);
  if (head_dim % 4 != 0 || al % 16 != 0 || (rope && head_dim % 8 != 0)) return ATTN_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (kv_seq == 0)  // no keys: out was all zeros and every gradient is zero
    return cudaMemsetAsync(dq, 0, (size_t)q_seq * num_heads * head_dim * sizeof(float), s) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
  BwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.n_q = (int)q_seq;
  a.n_kv = (int)kv_seq;
  a.H = (int)num_heads;
  a.G = (int)num_kv_heads;
  a.D = (int)head_dim;
  a.causal = (mask == ATTN_CAUSAL);
  a.window = window_arg(window);
  a.scale = 1.0f / sqrtf((float)head_dim);
  a.status = status_ptr();
  if (a.status == nullptr) return ATTN_ERR_CUDA;
  if (prec == ATTN_BF16 && !backward_bf16_supported(a)) {
    // bf16 operands refuse only head_dim outside {64, 128}; other groups
    // (not a power of two up to 128) run the fp32 backward.
    if (a.D != 64 && a.D != 128) return ATTN_ERR_UNSUPPORTED;
    prec = ATTN_FP32;
  }
  scratch_begin_call();
  if (workspace_too_small(backward_scratch_bytes(a, prec, rope))) return ATTN_ERR_INVALID_ARG;
  // RoPE: the gradient of the plain attention at the turned q and k, turned
  // back (the rotations are orthogonal); q and k are turned into scratch.
  void* scratch = nullptr;
  const size_t qe = (size_t)q_seq * num_heads * head_dim, ke = (size_t)kv_seq * num_kv_heads * head_dim;
  if (rope) {
    if (scratch_alloc(&scratch, (qe + ke) * sizeof(float), s) != cudaSuccess) return ATTN_ERR_CUDA;
    float* qt = static_cast<float*>(scratch);
    float* kt = qt + qe;  // qe is a multiple of 8 floats: 32-byte aligned
    if (launch_rope_k(q, qt, rope_table, q_seq, a.H, a.D, s) != cudaSuccess ||
        launch_rope_k(k, kt, rope_table, kv_seq, a.G, a.D, s) != cudaSuccess) {
      scratch_free(scratch, s);
      return ATTN_ERR_CUDA;
    }
    a.q = qt;
    a.k = kt;
  }
  int rc = prec == ATTN_BF16 ? launch_backward_bf16(a, s) : launch_backward_simt(a, s);
  if (rope && rc == ATTN_OK &&
      (launch_rope_k(dq, dq, rope_table, q_seq, a.H, a.D, s, -1.f) != cudaSuccess ||
       launch_rope_k(dk, dk, rope_table, kv_seq, a.G, a.D, s, -1.f) != cudaSuccess))
    rc = ATTN_ERR_CUDA;
  if (scratch != nullptr && scratch_free(scratch, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
  return rc;
}

extern "C" int attn_backward(const float* q, const float* k, const float* v, const float* out, const float* dout,
                             const float* lse, float* dq, float* dk, float* dv, uint32_t q_seq, uint32_t kv_seq,
                             uint32_t num_heads, uint32_t num_kv_heads, uint32_t head_dim, attn_mask_t mask, attn_prec_t prec,
                             uint32_t window, attn_stream_t stream) {
  return backward_impl(q, k, v, out, dout, lse, dq, dk, dv, q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask,
                       prec, window, nullptr, 0, stream);
}

extern "C" int attn_backward_rope(const float* q, const float* k, const float* v, const float* out, const float* dout,
                                  const float* lse, float* dq, float* dk, float* dv, uint32_t q_seq, uint32_t kv_seq,
                                  uint32_t num_heads, uint32_t num_kv_heads, uint32_t head_dim, attn_mask_t mask, attn_prec_t prec,
                                  uint32_t window, const float* rope_table, uint32_t table_rows,
                                  attn_stream_t stream) {
  if (rope_table == nullptr) return ATTN_ERR_INVALID_ARG;
  return backward_impl(q, k, v, out, dout, lse, dq, dk, dv, q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask,
                       prec, window, rope_table, table_rows, stream);
}

extern "C" int attn_set_workspace(void* workspace, size_t workspace_bytes) {
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) % 256) != 0) return ATTN_ERR_INVALID_ARG;
  scratch_bind(workspace, workspace_bytes);
  return ATTN_OK;
}

extern "C" size_t attn_forward_workspace_bytes(uint32_t q_seq, uint32_t kv_seq, uint32_t num_heads,
                                               uint32_t num_kv_heads, uint32_t head_dim, attn_mask_t mask,
                                               attn_prec_t prec, uint32_t window, int rope) {
  if (!heads_ok(num_heads, num_kv_heads, head_dim) || !valid_prec(prec)) return 0;
  if (mask != ATTN_CAUSAL && mask != ATTN_FULL && mask != ATTN_CROSS) return 0;
  if ((mask != ATTN_CROSS && kv_seq != q_seq) || q_seq > 0x7fffffffu || kv_seq > 0x7fffffffu) return 0;
  FlashArgs a{};
  a.k = a.v = kv_seq > 0 ? &kPresent : nullptr;
  a.q_row_stride = a.out_row_stride = (long long)num_heads * head_dim;
  a.kv_row_stride = (long long)num_kv_heads * head_dim;
  a.n_q = (int)q_seq;
  a.H = (int)num_heads;
  a.G = (int)num_kv_heads;
  a.D = (int)head_dim;
  a.causal = (mask == ATTN_CAUSAL);
  a.cap = a.n_all = (int)kv_seq;
  a.window = window_arg(window);
  a.rope = rope ? &kPresent : nullptr;
  return flash_scratch_bytes(a, prec);
}

extern "C" size_t attn_prefill_workspace_bytes(uint32_t n_queries, uint32_t n_heads, uint32_t n_kv_heads,
                                               uint32_t head_dim, uint32_t kv_dim, uint32_t max_seq,
                                               uint32_t start_pos, uint32_t q_base, attn_prec_t prec,
                                               uint32_t window) {
  if (!heads_ok(n_heads, n_kv_heads, head_dim) || !valid_prec(prec)) return 0;
  if ((uint64_t)kv_dim < (uint64_t)n_kv_heads * head_dim || max_seq > 0x7fffffffu) return 0;
  if ((uint64_t)start_pos + q_base + n_queries > max_seq) return 0;
  FlashArgs a{};
  a.k = a.v = &kPresent;
  a.q_row_stride = a.out_row_stride = (long long)n_heads * head_dim;
  a.kv_row_stride = kv_dim;
  a.n_q = (int)n_queries;
  a.H = (int)n_heads;
  a.G = (int)n_kv_heads;
  a.D = (int)head_dim;
  a.causal = 1;
  a.base_pos = (long long)start_pos + q_base;
  a.cap = a.n_all = (int)max_seq;
  a.window = window_arg(window);
  return flash_scratch_bytes(a, prec);
}

extern "C" size_t attn_backward_workspace_bytes(uint32_t q_seq, uint32_t kv_seq, uint32_t num_heads,
                                                uint32_t num_kv_heads, uint32_t head_dim, attn_prec_t prec, int rope) {
  if (!heads_ok(num_heads, num_kv_heads, head_dim) || !valid_prec(prec) || q_seq > 0x7fffffffu ||
      kv_seq > 0x7fffffffu)
    return 0;
  BwdArgs a{};
  a.n_q = (int)q_seq;
  a.n_kv = (int)kv_seq;
  a.H = (int)num_heads;
  a.G = (int)num_kv_heads;
  a.D = (int)head_dim;
  return q_seq == 0 ? 0 : backward_scratch_bytes(a, prec, rope != 0);
}

extern "C" size_t attn_scratch_reserved_bytes(void) { return scratch_pool_stat(0, false); }

extern "C" size_t attn_scratch_peak_bytes(int reset) { return scratch_pool_stat(1, reset != 0); }

extern "C" int attn_release_scratch(void) { return scratch_trim() ? ATTN_OK : ATTN_ERR_CUDA; }

extern "C" int attn_get_status(attn_stream_t stream) {
  unsigned* st = status_ptr();
  if (st == nullptr) return ATTN_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, st, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpy(st, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  return (int)v;
}

extern "C" const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape, precision or alignment";
    case ATTN_ERR_CUDA: return "CUDA launch or runtime error";
    case ATTN_ERR_TIMEOUT: return "a bounded device wait ran out";
    default: return "unknown status";
  }
}
