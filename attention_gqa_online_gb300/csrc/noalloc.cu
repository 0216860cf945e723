// noalloc.cu -- attn_decode_cached_noalloc: the split-KV decode with its
// scratch in a fixed device array that is part of the library image, so a
// call allocates no memory at all.
//
// Some callers cannot hand the library a workspace: code running under an
// allocator or host framework that owns all device memory and exposes none
// to plugins, or a latency-bound serving loop that must not call cudaMalloc
// (an allocation can synchronise the device and has no latency bound).  This
// entry point serves them.  Its cost is a fixed kScratchBytes of device
// memory held on every GPU that loads the library, until the process exits.
#include <mutex>

#include "../../include/attn_gqa.h"
#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

// Largest workspace the fixed scratch can stand in for.  The split decode
// needs about H * splits * D * 4 bytes (splits ~ 2 * SMs / G), i.e. about
// 0.6 MiB for 32 heads over 8 kv heads at D = 128 on a 152-SM GPU.
constexpr size_t kScratchBytes = size_t(4) << 20;

// The scratch itself.  Host code must not use this name as an address: on the
// host it is only a stand-in for the symbol.  The device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_dev_addr[kMaxDev] = {};
int g_scratch_sms[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of the scratch and the SM count of the current device,
// looked up on the first call on each device (with that device current).
int scratch_setup(void** addr, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_dev_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return ATTN_ERR_CUDA;
    g_scratch_dev_addr[dev] = p;
    g_scratch_sms[dev] = n;
  }
  *addr = g_scratch_dev_addr[dev];
  *sms = g_scratch_sms[dev];
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_decode_cached_noalloc(const float* q, const float* k_cache, const float* v_cache,
                                          const uint32_t* kv_pos_dev, float* out, uint32_t num_heads,
                                          uint32_t num_kv_heads, uint32_t head_dim, uint32_t max_seq,
                                          attn_stream_t stream) {
  if (num_heads == 0 || num_kv_heads == 0 || num_heads % num_kv_heads != 0 || head_dim == 0 || head_dim > 128 ||
      max_seq == 0 || max_seq > 0x7fffffffu)
    return ATTN_ERR_INVALID_ARG;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || kv_pos_dev == nullptr || out == nullptr)
    return ATTN_ERR_INVALID_ARG;
  const int H = (int)num_heads, G = (int)num_kv_heads, D = (int)head_dim, ms = (int)max_seq;
  const bool aligned = ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
                         reinterpret_cast<uintptr_t>(v_cache)) % 16) == 0;
  if (!decode_split_supported(H, G, D) || !aligned) return ATTN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  int sms = 0;
  int rc = scratch_setup(&scratch, &sms);
  if (rc != ATTN_OK) return rc;
  const size_t need = decode_workspace_bytes(H, G, D, ms, sms);
  if (need == 0 || need > kScratchBytes) return ATTN_ERR_UNSUPPORTED;
  unsigned* status = device_status_word();
  if (status == nullptr) return ATTN_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The scratch keeps whatever the previous call left; the per-kv-head
  // arrival counters at its start must read zero when the kernel begins.
  if (cudaMemsetAsync(scratch, 0, decode_ticket_bytes(decode_groups(H, G, D)), s) != cudaSuccess) return ATTN_ERR_CUDA;
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
  d.workspace = scratch;
  d.status = status;
  return launch_decode_split(d, decode_splits(decode_groups(H, G, D), ms, sms), s);
}
