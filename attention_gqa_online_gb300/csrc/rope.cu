// rope.cu -- rotary position embedding helpers: the cos/sin table and the
// rotation of K rows ahead of the tensor-core forward.
//
// Convention (the forward page leaves its RoPE hooks to the host framework;
// this library's reading): the pairs (d, d + D/2), d < D/2, of a row at
// position p turn by the angle p * base^(-2d/D):
//   x'[d]       = x[d] cos - x[d + D/2] sin
//   x'[d + D/2] = x[d + D/2] cos + x[d] sin
// Table row p holds (cos of pairs 0..D/2-1, sin of pairs 0..D/2-1) in fp32,
// computed in fp64 (an fp32 angle p * theta would be off by up to p * 2^-24
// rad, 1e-3 at p = 16384).
#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

__global__ void __launch_bounds__(256) rope_table_kernel(float* table, int max_pos, int D, double base) {
  const int half = D / 2;
  const long long idx = (long long)blockIdx.x * 256 + threadIdx.x;
  if (idx >= (long long)max_pos * half) return;
  const int p = (int)(idx / half), d = (int)(idx % half);
  const double a = (double)p * pow(base, -2.0 * (double)d / (double)D);
  double s, c;
  sincos(a, &s, &c);
  table[(long long)p * D + d] = (float)c;
  table[(long long)p * D + half + d] = (float)s;
}

// Rows [0, rows) of x ([rows][G*D], G heads): each thread turns one float4
// pair (4 dims d..d+3 and d+D/2..d+D/2+3) of one head of one row, by the
// angle (sgn = 1) or back (sgn = -1).  out may be x itself.
__global__ void __launch_bounds__(256) rope_k_kernel(const float* k, float* out, const float* __restrict__ table,
                                                     long long rows, int G, int D, float sgn) {
  allow_dependent_launch();
  grid_dependency_wait();
  const int half4 = D / 8;  // float4 groups per half row of one head
  const long long idx = (long long)blockIdx.x * 256 + threadIdx.x;
  if (idx >= rows * G * half4) return;
  const long long t = idx / ((long long)G * half4);
  const int rem = (int)(idx % ((long long)G * half4));
  const int g = rem / half4, d = 4 * (rem % half4);
  const long long base = t * G * D + (long long)g * D;
  const float4 lo = *reinterpret_cast<const float4*>(k + base + d);
  const float4 hi = *reinterpret_cast<const float4*>(k + base + D / 2 + d);
  const float4 c = *reinterpret_cast<const float4*>(table + t * D + d);
  float4 s = *reinterpret_cast<const float4*>(table + t * D + D / 2 + d);
  s = make_float4(sgn * s.x, sgn * s.y, sgn * s.z, sgn * s.w);
  *reinterpret_cast<float4*>(out + base + d) =
      make_float4(lo.x * c.x - hi.x * s.x, lo.y * c.y - hi.y * s.y, lo.z * c.z - hi.z * s.z, lo.w * c.w - hi.w * s.w);
  *reinterpret_cast<float4*>(out + base + D / 2 + d) =
      make_float4(hi.x * c.x + lo.x * s.x, hi.y * c.y + lo.y * s.y, hi.z * c.z + lo.z * s.z, hi.w * c.w + lo.w * s.w);
}

}  // namespace

int launch_rope_table(float* table, int max_pos, int D, double base, cudaStream_t s) {
  const long long n = (long long)max_pos * (D / 2);
  if (n == 0) return ATTN_OK;
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(table, max_pos, D, base);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

cudaError_t launch_rope_k(const float* k, float* out, const float* table, long long rows, int G, int D,
                          cudaStream_t s, float sgn) {
  const long long n = rows * G * (D / 8);
  if (n == 0) return cudaSuccess;
  void* args[] = {&k, &out, &table, &rows, &G, &D, &sgn};
  return launch_pdl(reinterpret_cast<const void*>(rope_k_kernel), dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s,
                    args);
}

}  // namespace attn
