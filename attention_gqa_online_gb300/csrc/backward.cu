// backward.cu -- fp32 CUDA-core backward of the forward attention.
//
// The forward page emits, per (query row, head), the pair (max score, log of
// the exponential sum) so that a backward pass can rebuild the softmax without
// a second reduction (meganeura attention.wgsl: header comment and the final
// LSE store).  The pages print no backward; this one computes the plain
// gradient of out = softmax(scale * q K^T) V for an upstream gradient dout:
//
//   p_t  = 2^(scale*log2(e) * q.k_t - L),  L = (slot0 + slot1) * log2(e)
//   D    = dout . out                      (= sum_t p_t dout.v_t)
//   ds_t = p_t * (dout . v_t - D)
//   dv_t += p_t dout,   dk_t += scale ds_t q,   dq = scale sum_t ds_t k_t
//
// Three kernels:
//   bwd_prep_kernel   one warp per (row, head): D and L (fp32 scratch).
//   bwd_dkdv_kernel   one CTA per (64-key block, kv head g): K, V of the
//                     block stay in shared memory and dK, dV in registers,
//                     while the packed (query, head) rows of every query
//                     head of g whose window touches the block stream by in
//                     blocks of 64; each block rebuilds P and dS.
//   bwd_dq_kernel     one CTA per (64 packed rows, kv head g): Q, dout and
//                     dQ stay, key tiles of the rows' windows stream by.
// Every output element is written by exactly one CTA (no atomics), so the
// result does not depend on scheduling.  Rows and windows are those of the
// forward (causal / full / cross, optional sliding window).
//
// Thread layout (256 threads): rg = tid / 16, cl = tid % 16.  Score tiles:
// rows 4rg..4rg+3 x keys cl + 16j.  Gradient tiles: 4 rows (or keys)
// 4rg..4rg+3 x dims 4cl + 64jj.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

constexpr int BM = 64;   // packed rows per block
constexpr int BN = 64;   // keys per block
constexpr int NT = 256;  // threads per CTA
constexpr int PS = BN + 4;  // row stride of the P / dS tiles (floats)

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

// rows x DMAX fp32 tile into shared memory (row stride STRIDE floats), zero
// fill for rows >= valid_rows and columns >= D; src(r) is row r's address.
// D % 4 == 0 and every row address is 16-byte aligned.
template <int DMAX, int STRIDE, typename SrcFn>
__device__ __forceinline__ void load_rows(float* dst, int rows, int valid_rows, int D, SrcFn src) {
  constexpr int F = DMAX / 4;
  for (int idx = threadIdx.x; idx < rows * F; idx += NT) {
    const int r = idx / F, f = idx % F;
    const bool ok = r < valid_rows && 4 * f < D;
    cp_async16(dst + r * STRIDE + 4 * f, ok ? src(r) + 4 * f : src(0), ok ? 16u : 0u);
  }
}

// Window of query i (forward rules): keys [lo, n).
__device__ __forceinline__ void query_window(const BwdArgs& a, long long i, int* n, int* lo) {
  int w = 0;
  if (i >= 0 && i < a.n_q) w = a.causal ? (int)min((long long)a.n_kv, i + 1) : a.n_kv;
  *n = w;
  *lo = first_key(w, a.window);
}

// S[4][4] += rows r0..r0+3 of A . rows cl+16j of B (both [64][STRIDE] tiles),
// products summed in groups of 8 before they join the running sum.
template <int DMAX, int STRIDE>
__device__ __forceinline__ void score_tile(const float* A, const float* B, int r0, int cl, float s[4][4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 2
  for (int d = 0; d < DMAX; d += 8) {
    float4 x[4][2], y[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[i][0] = *reinterpret_cast<const float4*>(&A[(r0 + i) * STRIDE + d]);
      x[i][1] = *reinterpret_cast<const float4*>(&A[(r0 + i) * STRIDE + d + 4]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      y[j][0] = *reinterpret_cast<const float4*>(&B[(cl + 16 * j) * STRIDE + d]);
      y[j][1] = *reinterpret_cast<const float4*>(&B[(cl + 16 * j) * STRIDE + d + 4]);
    }
    // Each 8-product group as two chains (even and odd elements) of paired
    // fmas on the register pairs the float4 loads fill.
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float e0 = 0.f, e1 = 0.f;
        fma2_acc(e0, e1, x[i][0].x, x[i][0].y, y[j][0].x, y[j][0].y);
        fma2_acc(e0, e1, x[i][0].z, x[i][0].w, y[j][0].z, y[j][0].w);
        fma2_acc(e0, e1, x[i][1].x, x[i][1].y, y[j][1].x, y[j][1].y);
        fma2_acc(e0, e1, x[i][1].z, x[i][1].w, y[j][1].z, y[j][1].w);
        s[i][j] += e0 + e1;
      }
  }
}

// ------------------------------------------------------------------ prep
// delta[i*H + h] = dout . out; l2[i*H + h] = (lse0 + lse1) * log2(e).
__global__ void __launch_bounds__(256) bwd_prep_kernel(const BwdArgs a, float* delta, float* l2) {
  allow_dependent_launch();
  grid_dependency_wait();
  const long long pair = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (pair >= (long long)a.n_q * a.H) return;
  const long long off = pair * a.D;  // (i, h) row of out / dout
  float acc = 0.f;
  for (int d = 4 * lane; d < a.D; d += 128) {
    const float4 o = *reinterpret_cast<const float4*>(a.out + off + d);
    const float4 g = *reinterpret_cast<const float4*>(a.dout + off + d);
    acc = dot4(o, g, acc);
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (lane == 0) {
    delta[pair] = acc;
    l2[pair] = (a.lse[2 * pair] + a.lse[2 * pair + 1]) * kLog2e;
  }
}

// ------------------------------------------------------------------ dK, dV
template <int DMAX>
struct KvSmem {
  static constexpr int QS = DMAX + 4;
  float k[BN * QS];
  float v[BN * QS];
  float q[BM * QS];
  float g[BM * QS];  // dout rows
  float p[BM * PS];  // [row][key]
  float ds[BM * PS];
  float l2[BM];
  float delta[BM];
  int row_n[BM];
  int row_lo[BM];
};

template <int DMAX>
__global__ void __launch_bounds__(NT, 1)
    bwd_dkdv_kernel(const BwdArgs a, const float* __restrict__ delta, const float* __restrict__ l2) {
  using Smem = KvSmem<DMAX>;
  constexpr int QS = Smem::QS;
  constexpr int OC = DMAX / 64;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  allow_dependent_launch();
  grid_dependency_wait();
  const int tid = threadIdx.x, rg = tid >> 4, cl = tid & 15, r0 = 4 * rg;
  const int g = blockIdx.y, gs = a.H / a.G, D = a.D;
  const int k0 = blockIdx.x * BN;
  const int k_valid = min(BN, a.n_kv - k0);
  const long long row_stride = (long long)a.H * D, kv_stride = (long long)a.G * D;
  const float sl2 = a.scale * kLog2e;

  load_rows<DMAX, QS>(sm.k, BN, k_valid, D, [&](int r) { return a.k + (k0 + r) * kv_stride + (long long)g * D; });
  load_rows<DMAX, QS>(sm.v, BN, k_valid, D, [&](int r) { return a.v + (k0 + r) * kv_stride + (long long)g * D; });
  cp_async_commit();

  // Queries whose window meets keys [k0, k0 + BN): windows [lo_i, n_i) with
  // both bounds non-decreasing in i.
  long long i_begin = 0, i_end = a.n_q;
  if (a.causal) {
    i_begin = k0;  // n_i = i + 1 > k0
    if (a.window > 0) i_end = min((long long)a.n_q, (long long)k0 + BN - 1 + a.window);  // lo_i < k0 + BN
  } else if (first_key(a.n_kv, a.window) >= k0 + BN) {
    i_end = 0;
  }
  const long long row_first = i_begin * gs, row_last = max(i_begin, i_end) * gs;  // packed rows [first, last)

  float dk[4][OC * 4], dv[4][OC * 4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < OC * 4; ++c) dk[i][c] = dv[i][c] = 0.f;

  for (long long rb = row_first; rb < row_last; rb += BM) {
    const int rows = (int)min((long long)BM, row_last - rb);
    auto row_src = [&](const float* base) {
      return [=](int r) {
        const long long pk = rb + r;
        return base + (pk / gs) * row_stride + (long long)(g * gs + (int)(pk % gs)) * D;
      };
    };
    __syncthreads();  // the previous block's tiles are no longer read
    load_rows<DMAX, QS>(sm.q, BM, rows, D, row_src(a.q));
    load_rows<DMAX, QS>(sm.g, BM, rows, D, row_src(a.dout));
    cp_async_commit();
    if (tid < BM) {
      const long long pk = rb + tid;
      const long long i = pk / gs;
      int n = 0, lo = 0;
      if (tid < rows) query_window(a, i, &n, &lo);
      sm.row_n[tid] = n;
      sm.row_lo[tid] = lo;
      const long long pair = i * a.H + g * gs + (int)(pk % gs);
      sm.l2[tid] = tid < rows ? l2[pair] : 0.f;
      sm.delta[tid] = tid < rows ? delta[pair] : 0.f;
    }
    cp_async_wait<0>();
    __syncthreads();

    // P and dS for rows r0..r0+3, keys cl + 16j.
    float s[4][4], dp[4][4];
    score_tile<DMAX, QS>(sm.q, sm.k, r0, cl, s);
    score_tile<DMAX, QS>(sm.g, sm.v, r0, cl, dp);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + i;
      const int n = sm.row_n[r], lo = sm.row_lo[r];
      const float lr = sm.l2[r], dr = sm.delta[r];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int t = k0 + cl + 16 * j;
        const float p = (t >= lo && t < n) ? ex2(fmaf(s[i][j], sl2, -lr)) : 0.f;
        sm.p[r * PS + cl + 16 * j] = p;
        sm.ds[r * PS + cl + 16 * j] = p * (dp[i][j] - dr);
      }
    }
    __syncthreads();

    // dV[key][d] += sum_r P[r][key] dout[r][d];  dK[key][d] += sum_r dS[r][key] q[r][d]
    // for keys r0..r0+3 (as key indices) and dims 4cl + 64jj.
#pragma unroll 2
    for (int r = 0; r < BM; ++r) {
      const float4 pv = *reinterpret_cast<const float4*>(&sm.p[r * PS + r0]);
      const float4 sv = *reinterpret_cast<const float4*>(&sm.ds[r * PS + r0]);
      const float pk[4] = {pv.x, pv.y, pv.z, pv.w};
      const float sk[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
      for (int jj = 0; jj < OC; ++jj) {
        const int col = 4 * cl + 64 * jj;
        const float4 gv = *reinterpret_cast<const float4*>(&sm.g[r * QS + col]);
        const float4 qv = *reinterpret_cast<const float4*>(&sm.q[r * QS + col]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          fma2_acc(dv[i][4 * jj + 0], dv[i][4 * jj + 1], pk[i], pk[i], gv.x, gv.y);  // same order per column
          fma2_acc(dv[i][4 * jj + 2], dv[i][4 * jj + 3], pk[i], pk[i], gv.z, gv.w);
          fma2_acc(dk[i][4 * jj + 0], dk[i][4 * jj + 1], sk[i], sk[i], qv.x, qv.y);
          fma2_acc(dk[i][4 * jj + 2], dk[i][4 * jj + 3], sk[i], sk[i], qv.z, qv.w);
        }
      }
    }
  }
  cp_async_wait<0>();  // a block with no query rows still owns its K/V copies

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int key = r0 + i;
    if (key >= k_valid) continue;
    float* dkr = a.dk + (k0 + key) * kv_stride + (long long)g * D;
    float* dvr = a.dv + (k0 + key) * kv_stride + (long long)g * D;
#pragma unroll
    for (int jj = 0; jj < OC; ++jj) {
      const int col = 4 * cl + 64 * jj;
      if (col < D) {
        *reinterpret_cast<float4*>(dkr + col) = make_float4(dk[i][4 * jj] * a.scale, dk[i][4 * jj + 1] * a.scale,
                                                            dk[i][4 * jj + 2] * a.scale, dk[i][4 * jj + 3] * a.scale);
        *reinterpret_cast<float4*>(dvr + col) =
            make_float4(dv[i][4 * jj], dv[i][4 * jj + 1], dv[i][4 * jj + 2], dv[i][4 * jj + 3]);
      }
    }
  }
}

// ------------------------------------------------------------------ dQ
template <int DMAX>
struct QSmem {
  static constexpr int QS = DMAX + 4;
  float q[BM * QS];
  float g[BM * QS];
  float k[BN * QS];
  float v[BN * QS];
  float dst[BN * PS];  // dS transposed: [key][row]
  float l2[BM];
  float delta[BM];
  int row_n[BM];
  int row_lo[BM];
};

template <int DMAX>
__global__ void __launch_bounds__(NT, 1)
    bwd_dq_kernel(const BwdArgs a, const float* __restrict__ delta, const float* __restrict__ l2) {
  using Smem = QSmem<DMAX>;
  constexpr int QS = Smem::QS;
  constexpr int OC = DMAX / 64;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  allow_dependent_launch();
  grid_dependency_wait();
  const int tid = threadIdx.x, rg = tid >> 4, cl = tid & 15, r0 = 4 * rg;
  const int g = blockIdx.y, gs = a.H / a.G, D = a.D;
  const long long rb = (long long)(gridDim.x - 1 - blockIdx.x) * BM;  // latest (longest) causal rows first
  const int rows = (int)min((long long)BM, (long long)a.n_q * gs - rb);
  const long long row_stride = (long long)a.H * D, kv_stride = (long long)a.G * D;
  const float sl2 = a.scale * kLog2e;

  auto row_src = [&](const float* base) {
    return [=](int r) {
      const long long pk = rb + r;
      return base + (pk / gs) * row_stride + (long long)(g * gs + (int)(pk % gs)) * D;
    };
  };
  load_rows<DMAX, QS>(sm.q, BM, rows, D, row_src(a.q));
  load_rows<DMAX, QS>(sm.g, BM, rows, D, row_src(a.dout));
  cp_async_commit();
  if (tid < BM) {
    const long long pk = rb + tid;
    const long long i = pk / gs;
    int n = 0, lo = 0;
    if (tid < rows) query_window(a, i, &n, &lo);
    sm.row_n[tid] = n;
    sm.row_lo[tid] = lo;
    const long long pair = i * a.H + g * gs + (int)(pk % gs);
    sm.l2[tid] = tid < rows ? l2[pair] : 0.f;
    sm.delta[tid] = tid < rows ? delta[pair] : 0.f;
  }
  __syncthreads();
  int n_max = 0, lo_min = INT_MAX;
  for (int r = 0; r < BM; ++r) {
    n_max = max(n_max, sm.row_n[r]);
    if (sm.row_n[r] > 0) lo_min = min(lo_min, sm.row_lo[r]);
  }
  const int t_begin = n_max > 0 ? lo_min / BN * BN : 0;

  float dq[4][OC * 4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < OC * 4; ++c) dq[i][c] = 0.f;

  for (int t0 = t_begin; t0 < n_max; t0 += BN) {
    const int valid = min(BN, n_max - t0);
    __syncthreads();  // the previous tile is no longer read
    load_rows<DMAX, QS>(sm.k, BN, valid, D, [&](int r) { return a.k + (t0 + r) * kv_stride + (long long)g * D; });
    load_rows<DMAX, QS>(sm.v, BN, valid, D, [&](int r) { return a.v + (t0 + r) * kv_stride + (long long)g * D; });
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    float s[4][4], dp[4][4];
    score_tile<DMAX, QS>(sm.q, sm.k, r0, cl, s);
    score_tile<DMAX, QS>(sm.g, sm.v, r0, cl, dp);
    float ds[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + i;
      const int n = sm.row_n[r], lo = sm.row_lo[r];
      const float lr = sm.l2[r], dr = sm.delta[r];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int t = t0 + cl + 16 * j;
        const float p = (t >= lo && t < n) ? ex2(fmaf(s[i][j], sl2, -lr)) : 0.f;
        ds[i][j] = p * (dp[i][j] - dr);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<float4*>(&sm.dst[(cl + 16 * j) * PS + r0]) = make_float4(ds[0][j], ds[1][j], ds[2][j], ds[3][j]);
    __syncthreads();

    // dQ[r][d] += sum_key dS[r][key] K[key][d] for rows r0..r0+3, dims 4cl + 64jj.
#pragma unroll 4
    for (int kk = 0; kk < BN; ++kk) {
      const float4 sv = *reinterpret_cast<const float4*>(&sm.dst[kk * PS + r0]);
      const float sr[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
      for (int jj = 0; jj < OC; ++jj) {
        const float4 kv = *reinterpret_cast<const float4*>(&sm.k[kk * QS + 4 * cl + 64 * jj]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          fma2_acc(dq[i][4 * jj + 0], dq[i][4 * jj + 1], sr[i], sr[i], kv.x, kv.y);  // same order per column
          fma2_acc(dq[i][4 * jj + 2], dq[i][4 * jj + 3], sr[i], sr[i], kv.z, kv.w);
        }
      }
    }
  }
  cp_async_wait<0>();

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + i;
    if (r >= rows) continue;
    const long long pk = rb + r;
    float* dst = a.dq + (pk / gs) * row_stride + (long long)(g * gs + (int)(pk % gs)) * D;
#pragma unroll
    for (int jj = 0; jj < OC; ++jj) {
      const int col = 4 * cl + 64 * jj;
      if (col < D)
        *reinterpret_cast<float4*>(dst + col) = make_float4(dq[i][4 * jj] * a.scale, dq[i][4 * jj + 1] * a.scale,
                                                            dq[i][4 * jj + 2] * a.scale, dq[i][4 * jj + 3] * a.scale);
    }
  }
}

template <int DMAX>
int launch_d(const BwdArgs& a, float* delta, float* l2, cudaStream_t s) {
  const int gs = a.H / a.G;
  const size_t kv_smem = sizeof(KvSmem<DMAX>), q_smem = sizeof(QSmem<DMAX>);
  auto kv_kern = bwd_dkdv_kernel<DMAX>;
  auto q_kern = bwd_dq_kernel<DMAX>;
  if (!set_smem_limit(reinterpret_cast<const void*>(kv_kern), kv_smem) ||
      !set_smem_limit(reinterpret_cast<const void*>(q_kern), q_smem))
    return ATTN_ERR_CUDA;
  BwdArgs aa = a;
  float* d = delta;
  float* l = l2;
  void* args[] = {&aa, &d, &l};
  const long long kb = (a.n_kv + BN - 1) / BN;
  const long long qb = ((long long)a.n_q * gs + BM - 1) / BM;
  // dK/dV and dQ are independent: they run concurrently (dQ on a side stream).
  return launch_forked(s, reinterpret_cast<const void*>(kv_kern), dim3((unsigned)kb, (unsigned)a.G), kv_smem,
                       reinterpret_cast<const void*>(q_kern), dim3((unsigned)qb, (unsigned)a.G), q_smem, dim3(NT),
                       args);
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdArgs& a, float* delta, float* l2, cudaStream_t s) {
  const long long pairs = (long long)a.n_q * a.H;
  BwdArgs aa = a;
  void* pargs[] = {&aa, &delta, &l2};
  return launch_pdl(reinterpret_cast<const void*>(bwd_prep_kernel), dim3((unsigned)((pairs + 7) / 8)), dim3(256), 0, s,
                    pargs);
}

// delta and the base-2 log-sum-exp per (row, head).
size_t backward_simt_scratch_bytes(const BwdArgs& a) {
  return scratch_round((size_t)a.n_q * a.H * 2 * sizeof(float));
}

int launch_backward_simt(const BwdArgs& a, cudaStream_t s) {
  const long long pairs = (long long)a.n_q * a.H;
  if (pairs == 0) return ATTN_OK;
  if (a.G > 65535 || (pairs + 7) / 8 > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (scratch_alloc(&scratch, backward_simt_scratch_bytes(a), s) != cudaSuccess) return ATTN_ERR_CUDA;
  float* delta = static_cast<float*>(scratch);
  float* l2 = delta + pairs;
  int rc = launch_bwd_prep(a, delta, l2, s) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  if (rc == ATTN_OK) rc = a.D <= 64 ? launch_d<64>(a, delta, l2, s) : launch_d<128>(a, delta, l2, s);
  if (scratch_free(scratch, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
  return rc;
}

}  // namespace attn
