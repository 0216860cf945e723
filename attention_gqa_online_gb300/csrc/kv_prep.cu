// kv_prep.cu -- K/V operand pre-pass of the tensor-core flash kernels.
//
// One block per (128-key tile T, kv head g) for K and, on the 16-bit path, two
// per tile for V (64 rows each: V needs no tile-wide reduction, and the
// smaller blocks leave the SMs sooner), 512 threads; a row of
// one head is D/4 consecutive threads' float4 groups, so every load and store
// is a coalesced row run.  Rows [128 T, 128 T + 128) at or past `rows_end`
// are not written (the attention kernels' tensor maps end there).  Paged
// caches (table != nullptr): logical row t is read from its pool row; a page
// outside the pool reads as zeros and records ATTN_ERR_INVALID_ARG.  RoPE
// (rope != nullptr): K row t is turned at position t first.  Outputs keep the
// inputs' layout (rows of `stride` elements, head g at column g * D).
//
// Operands: K as fp16 times 2^(14 - E_T), E_T the binary exponent of the
// tile's (this head's) largest magnitude, so its values lie below 2^15, inside
// fp16's range; kfac[T * G + g] = 2^(E_T - 14).  With out1 set, blocks of the
// second grid layer (z = 1) also write V as bf16 (the 16-bit kernel's P V
// operand; the TF32-class kernel reads V as it is).
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace attn {
namespace {

constexpr int kPrepThreads = 512;

template <int D>
__global__ void __launch_bounds__(kPrepThreads, 2) kv_prep_kernel(const PrepArgs p) {
  constexpr int kPerRow = D / 4;                       // float4 groups per row of one head
  constexpr int kRowsPerPass = kPrepThreads / kPerRow;  // rows of the tile per pass of the block
  constexpr int kPasses = 128 / kRowsPerPass;
  // The attention kernel that follows may start once every block is past this
  // wait: it reads Q (and the RoPE table, a block table) before waiting for
  // this grid, and those were written, if at all, by kernels this wait covers.
  grid_dependency_wait();
  allow_dependent_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y;
  if (blockIdx.z > 0) {
    // V as bf16, half a tile per block (no reduction over the tile).
    constexpr int kHalf = kPasses / 2;
    const long long t0 = (long long)(p.tile0 + blockIdx.x) * 128 + 64 * (blockIdx.z - 1);
    const int c4v = tid % kPerRow, rsv = tid / kPerRow;
    const long long colv = (long long)g * D + 4 * c4v;
    float4 xv[kHalf];
    if (p.table == nullptr && t0 + 64 <= p.rows_end) {
#pragma unroll
      for (int i = 0; i < kHalf; ++i)
        xv[i] = *reinterpret_cast<const float4*>(p.v + (t0 + i * kRowsPerPass + rsv) * p.stride + colv);
    } else {
#pragma unroll
      for (int i = 0; i < kHalf; ++i) {
        const long long t = t0 + i * kRowsPerPass + rsv;
        xv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < p.rows_end) {
          long long row = t;
          if (p.table != nullptr) row = paged_row(p.table, p.page_rows, p.num_pages, (int)t, p.status);
          if (row >= 0) xv[i] = *reinterpret_cast<const float4*>(p.v + row * p.stride + colv);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kHalf; ++i) {
      const long long t = t0 + i * kRowsPerPass + rsv;
      if (t < p.rows_end)
        *reinterpret_cast<uint2*>(p.out1 + t * p.stride + colv) =
            make_uint2(tc::pack_bf16(xv[i].x, xv[i].y), tc::pack_bf16(xv[i].z, xv[i].w));
    }
    return;
  }
  const long long t_first = (long long)(p.tile0 + blockIdx.x) * 128;
  const int c4 = tid % kPerRow;  // float4 group within the row
  const int rsub = tid / kPerRow;
  const float* src = p.k;
  const long long col = (long long)g * D + 4 * c4;
  float4 x[kPasses];
  float mx = 0.f;
  if (p.table == nullptr && t_first + 128 <= p.rows_end) {
    // A whole contiguous tile: every load is issued before any is used.
#pragma unroll
    for (int i = 0; i < kPasses; ++i)
      x[i] = *reinterpret_cast<const float4*>(src + (t_first + i * kRowsPerPass + rsub) * p.stride + col);
  } else {
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
      const long long t = t_first + i * kRowsPerPass + rsub;
      x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < p.rows_end) {
        long long row = t;
        if (p.table != nullptr) row = paged_row(p.table, p.page_rows, p.num_pages, (int)t, p.status);
        if (row >= 0) x[i] = *reinterpret_cast<const float4*>(src + row * p.stride + col);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    if (p.rope != nullptr) {
      // Pair (d, d + D/2): the partner float4 is D/8 lanes away in the same row.
      const float4 y =
          make_float4(__shfl_xor_sync(0xffffffffu, x[i].x, D / 8), __shfl_xor_sync(0xffffffffu, x[i].y, D / 8),
                      __shfl_xor_sync(0xffffffffu, x[i].z, D / 8), __shfl_xor_sync(0xffffffffu, x[i].w, D / 8));
      const long long t = t_first + i * kRowsPerPass + rsub;
      if (t < p.rows_end) {
        const int e = 4 * c4;
        const bool first = e < D / 2;
        const int dd = first ? e : e - D / 2;
        const float4 cv = *reinterpret_cast<const float4*>(p.rope + t * D + dd);
        const float4 sv = *reinterpret_cast<const float4*>(p.rope + t * D + D / 2 + dd);
        const float sg = first ? -1.f : 1.f;
        x[i] = make_float4(fmaf(sg * y.x, sv.x, x[i].x * cv.x), fmaf(sg * y.y, sv.y, x[i].y * cv.y),
                           fmaf(sg * y.z, sv.z, x[i].z * cv.z), fmaf(sg * y.w, sv.w, x[i].w * cv.w));
      }
    }
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x[i].x), fabsf(x[i].y)), fmaxf(fabsf(x[i].z), fabsf(x[i].w))));
  }
  // Largest magnitude of the tile: warp maxima, then the block's.
  __shared__ float wmax[kPrepThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) wmax[warp] = mx;
  __syncthreads();
  mx = 0.f;
#pragma unroll
  for (int w = 0; w < kPrepThreads / 32; ++w) mx = fmaxf(mx, wmax[w]);
  const int et = pow2_scale_exp(mx);
  const float up = pow2f(14 - et);
  if (tid == 0) p.kfac[(long long)(p.tile0 + blockIdx.x) * p.G + g] = pow2f(et - 14);
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const long long t = t_first + i * kRowsPerPass + rsub;
    if (t < p.rows_end)
      *reinterpret_cast<uint2*>(p.out0 + t * p.stride + col) =
          make_uint2(tc::pack_f16(x[i].x * up, x[i].y * up), tc::pack_f16(x[i].z * up, x[i].w * up));
  }
}

template <int D>
cudaError_t launch_d(const PrepArgs& p, cudaStream_t s) {
  PrepArgs pp = p;
  void* args[] = {&pp};
  const dim3 grid((unsigned)(p.n_tiles - p.tile0), (unsigned)p.G, p.out1 != nullptr ? 3u : 1u);
  return launch_pdl(reinterpret_cast<const void*>(kv_prep_kernel<D>), grid, dim3(kPrepThreads), 0, s, args);
}

}  // namespace

cudaError_t launch_kv_prep(const PrepArgs& p, cudaStream_t s) {
  if (p.n_tiles <= p.tile0) return cudaSuccess;
  if (p.D == 128) return launch_d<128>(p, s);
  if (p.D == 64) return launch_d<64>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace attn
