// tma.cu -- host-side construction of TMA tensor maps (cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point so the library does not
// link libcuda directly).
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace attn {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void resolve() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

bool make_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
               const uint32_t* box, bool bf16, int swizzle) {
  std::call_once(g_once, resolve);
  if (g_encode == nullptr || rank < 1 || rank > 5) return false;
  uint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                              (cuuint32_t)rank, const_cast<void*>(base), dims, strides_bytes, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle == kSwizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B
                              : swizzle == kSwizzle128Atom32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B
                                                             : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {
struct SmemAttr {
  const void* kernel;
  int device;
  size_t bytes;
};
constexpr int kAttrSlots = 256;
SmemAttr g_attr[kAttrSlots];
int g_attr_n = 0;
std::mutex g_attr_mu;
}  // namespace

cudaError_t launch_pdl(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kernel, args);
}

namespace {
// One stream-ordered memory pool per device for kernel scratch.  Its release
// threshold is unbounded, so memory freed at the end of a call stays
// reserved for the next one instead of being returned (and re-mapped) at
// every synchronisation.
constexpr int kMaxDevices = 64;
cudaMemPool_t g_pool[kMaxDevices] = {};
std::mutex g_pool_mu;

cudaMemPool_t scratch_pool() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  if (g_pool[dev] == nullptr) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
    uint64_t keep = ~0ull;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return nullptr;
    }
    g_pool[dev] = pool;
  }
  return g_pool[dev];
}

// A caller-owned workspace bound to this thread (attn_set_workspace): every
// call's scratch is carved from it, from offset 0 at the start of each call
// (calls on one stream run in order, so they can reuse the same bytes).
thread_local void* t_ws = nullptr;
thread_local size_t t_ws_bytes = 0;
thread_local size_t t_ws_used = 0;

}  // namespace

void scratch_bind(void* ws, size_t bytes) {
  t_ws = ws;
  t_ws_bytes = ws != nullptr ? bytes : 0;
  t_ws_used = 0;
}

bool scratch_bound(size_t* bytes) {
  if (bytes != nullptr) *bytes = t_ws_bytes;
  return t_ws != nullptr;
}

void scratch_begin_call() { t_ws_used = 0; }

cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t s) {
  if (t_ws != nullptr) {
    const size_t off = scratch_round(t_ws_used);
    if (off > t_ws_bytes || bytes > t_ws_bytes - off) return cudaErrorMemoryAllocation;
    *p = static_cast<char*>(t_ws) + off;
    t_ws_used = off + bytes;
    return cudaSuccess;
  }
  cudaMemPool_t pool = scratch_pool();
  if (pool == nullptr) return cudaErrorMemoryAllocation;
  return cudaMallocFromPoolAsync(p, bytes, pool, s);
}

cudaError_t scratch_free(void* p, cudaStream_t s) {
  if (t_ws != nullptr && p >= t_ws && p < static_cast<char*>(t_ws) + t_ws_bytes) return cudaSuccess;
  return cudaFreeAsync(p, s);
}

size_t scratch_pool_stat(int which, bool reset) {
  cudaMemPool_t pool = scratch_pool();
  if (pool == nullptr) return 0;
  cudaMemPoolAttr attr = which == 0 ? cudaMemPoolAttrReservedMemCurrent : cudaMemPoolAttrUsedMemHigh;
  uint64_t v = 0;
  if (cudaMemPoolGetAttribute(pool, attr, &v) != cudaSuccess) return 0;
  if (reset && which == 1) {
    uint64_t zero = 0;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &zero);
  }
  return (size_t)v;
}

bool scratch_trim() {
  cudaMemPool_t pool = scratch_pool();
  return pool != nullptr && cudaMemPoolTrimTo(pool, 0) == cudaSuccess;
}

cudaStream_t side_stream() {
  static cudaStream_t streams[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (streams[dev] == nullptr && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess)
    streams[dev] = nullptr;
  return streams[dev];
}

int launch_forked(cudaStream_t s, const void* k1, dim3 g1, size_t smem1, const void* k2, dim3 g2, size_t smem2,
                  dim3 block, void** args) {
  cudaStream_t side = side_stream();
  cudaEvent_t fork = nullptr, join = nullptr;
  if (side == nullptr || cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
    if (fork != nullptr) cudaEventDestroy(fork);
    return ATTN_ERR_CUDA;
  }
  int rc = ATTN_OK;
  if (cudaEventRecord(fork, s) != cudaSuccess || cudaStreamWaitEvent(side, fork, 0) != cudaSuccess ||
      launch_pdl(k2, g2, block, smem2, side, args) != cudaSuccess || launch_pdl(k1, g1, block, smem1, s, args) != cudaSuccess ||
      cudaEventRecord(join, side) != cudaSuccess || cudaStreamWaitEvent(s, join, 0) != cudaSuccess)
    rc = ATTN_ERR_CUDA;
  cudaEventDestroy(fork);  // released once the recorded work has completed
  cudaEventDestroy(join);
  return rc;
}

bool set_smem_limit(const void* kernel, size_t bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  {
    std::lock_guard<std::mutex> lock(g_attr_mu);
    for (int i = 0; i < g_attr_n; ++i)
      if (g_attr[i].kernel == kernel && g_attr[i].device == dev && g_attr[i].bytes >= bytes) return true;
  }
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
    return false;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (g_attr_n < kAttrSlots) g_attr[g_attr_n++] = SmemAttr{kernel, dev, bytes};
  return true;
}

}  // namespace attn
