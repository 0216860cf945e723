// bwd_tc.cu -- tcgen05 backward with bf16 operands and fp32 accumulation.
//
// The same gradient as backward.cu (the plain chain rule through the forward,
// the softmax rebuilt from the forward's (max, log-sum) pair; see there), with
// the five products on the tensor cores.  A pre-pass writes Q, dout, K and V
// as bf16 (same layouts) and the per-row D = dout . out and base-2
// log-sum-exp L; then two kernels:
//
//   bwd_dkdv_tc_kernel  one CTA per (128-key block, kv head g).  K and V of
//                       the block stay in shared memory; dV and dK accumulate
//                       in tensor memory while 128-row blocks of the packed
//                       (query, head) rows whose windows meet the block come
//                       by (every query head of g, so the GQA sum happens in
//                       the accumulators):
//                         S^T  = K Q^T,   dP^T = V dout^T       (SS MMAs)
//                         P^T  = 2^(S^T scale log2(e) - L),  dS^T = P^T (dP^T - D)
//                         dV  += P^T dout,   dK += dS^T Q       (A from TMEM)
//   bwd_dq_tc_kernel    one CTA per (128 packed rows, kv head g): Q and dout
//                       stay, the key tiles of the rows' windows come by:
//                         S = Q K^T,  dP = dout V^T,  dS = P (dP - D),  dQ += dS K
//
// Warp roles (256 threads): warp 0 issues the TMA copies, warp 1 allocates
// tensor memory and issues every MMA (its loop runs warp-uniformly, one
// elected lane issues), warps 4-7 hold one TMEM lane (key or row) per thread
// and do the elementwise step.  The chain per block is serial (products, then
// the elementwise step, then the next products); bf16 tiles are read both
// K-major and MN-major from the same 128-byte-swizzled copy.  Every wait is
// bounded; a CTA whose pipeline breaks drains its copies and MMAs first.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace attn {
namespace {

constexpr int kR = 128;                // keys per key block / packed rows per row block
constexpr int kThreads = 256;
constexpr int kChunkBytes = kR * 128;  // one 64-element column chunk of a 128-row bf16 tile
constexpr int kColS = 0, kColP = 128, kColAcc = 256;  // TMEM: S, dP (then P, dS as bf16), accumulators

template <int D>
struct Tile {
  static constexpr int kChunks = D / 64;
  static constexpr int kBytes = kChunks * kChunkBytes;
};

struct RowInfo {
  float l2, delta;
  int n, lo;  // window [lo, n); n = 0 for rows outside the call
};

template <int D>
struct __align__(1024) KvTcSmem {
  unsigned char k[Tile<D>::kBytes];
  unsigned char v[Tile<D>::kBytes];
  unsigned char q[2][Tile<D>::kBytes];
  unsigned char g[2][Tile<D>::kBytes];  // dout
  RowInfo rows[2][kR];
  uint64_t kv_full, q_full[2], q_empty[2], s_full, p_ready[2], pv_done, drain;  // p_ready: rows 0-63, 64-127
  uint32_t tmem_base;
  int abort;
};

template <int D>
struct __align__(1024) QTcSmem {
  unsigned char q[Tile<D>::kBytes];
  unsigned char g[Tile<D>::kBytes];
  unsigned char k[2][Tile<D>::kBytes];
  unsigned char v[2][Tile<D>::kBytes];
  uint64_t q_full, kv_full[2], kv_empty[2], s_full, p_ready[2], pv_done, drain;  // p_ready: keys 0-63, 64-127
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ int query_n(const BwdArgs& a, long long i) {
  return a.causal ? (int)min((long long)a.n_kv, i + 1) : a.n_kv;
}

// The elementwise step for one thread's TMEM lane: 128 columns of S and dP
// (at kColS / kColP) become bf16 P (over S, if write_p) and dS (over dP).
// info(c) gives the column's l2, delta and whether it is inside the window.
// half_done() runs once the first 64 columns are written (the products that
// read them may start while the other 64 are worked on).
template <typename InfoFn, typename HalfFn>
__device__ __forceinline__ void elementwise(uint32_t lane_tmem, float sl2, bool write_p, InfoFn info,
                                            HalfFn half_done) {
#pragma unroll 1
  for (int cc = 0; cc < kR / 32; ++cc) {
    if (cc == 2) {
      tc::tmem_st_wait();
      half_done();
    }
    uint32_t s[32], dp[32];
    tc::tmem_ld32(lane_tmem + kColS + 32 * cc, s);
    tc::tmem_ld32(lane_tmem + kColP + 32 * cc, dp);
    tc::tmem_ld_wait();
    tc::reg_fence(s);
    tc::reg_fence(dp);
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float p2[2], d2[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float l2, delta;
        const bool in = info(32 * cc + e + u, &l2, &delta);
        const float p = in ? ex2(fmaf(__uint_as_float(s[e + u]), sl2, -l2)) : 0.f;
        p2[u] = p;
        d2[u] = p * (__uint_as_float(dp[e + u]) - delta);
      }
      s[e >> 1] = tc::pack_bf16(p2[0], p2[1]);
      dp[e >> 1] = tc::pack_bf16(d2[0], d2[1]);
    }
    // Column 16 cc onwards: the loads of later chunks read columns >= 32 (cc + 1).
    if (write_p) tc::tmem_st16(lane_tmem + kColS + 16 * cc, s);
    tc::tmem_st16(lane_tmem + kColP + 16 * cc, dp);
  }
  tc::tmem_st_wait();
}

// Stores one thread's TMEM row of D fp32 accumulator columns, times `mul`.
template <int D>
__device__ __forceinline__ void store_row(uint32_t taddr, float* dst, float mul, bool ok) {
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t v[32];
    tc::tmem_ld32(taddr + 32 * c, v);
    tc::tmem_ld_wait();
    tc::reg_fence(v);
    if (ok) {
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4*>(dst + 32 * c + e) =
            make_float4(__uint_as_float(v[e]) * mul, __uint_as_float(v[e + 1]) * mul, __uint_as_float(v[e + 2]) * mul,
                        __uint_as_float(v[e + 3]) * mul);
    }
  }
}

// ------------------------------------------------------------------ dK, dV
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_tc_kernel(const BwdArgs a, const float* __restrict__ delta, const float* __restrict__ l2,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_g) {
  using T = Tile<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  KvTcSmem<D>& sm = *reinterpret_cast<KvTcSmem<D>*>(smem_raw + ((1024u - (raw & 1023u)) & 1023u));
  allow_dependent_launch();
  grid_dependency_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, gs = a.H / a.G;
  const int k0 = blockIdx.x * kR;
  const int k_valid = min(kR, a.n_kv - k0);
  // Queries whose window meets keys [k0, k0 + 128) (both window bounds grow with i).
  long long i_begin = 0, i_end = a.n_q;
  if (a.causal) {
    i_begin = k0;
    if (a.window > 0) i_end = min((long long)a.n_q, (long long)k0 + kR - 1 + a.window);
  } else if (first_key(a.n_kv, a.window) >= k0 + kR) {
    i_end = 0;
  }
  if (i_end < i_begin) i_end = i_begin;
  const long long row_first = i_begin * gs;
  const int nqb = (int)(((i_end - i_begin) * gs + kR - 1) / kR);

  if (tid == 0) {
    mbar_init(&sm.kv_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.q_full[b], 1);
      mbar_init(&sm.q_empty[b], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_ready[0], 4);
    mbar_init(&sm.p_ready[1], 4);
    mbar_init(&sm.pv_done, 1);
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(&sm.tmem_base, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (nqb > 0) {
      if (lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_g);
        mbar_arrive_expect_tx(&sm.kv_full, 2u * T::kBytes);
#pragma unroll
        for (int c = 0; c < T::kChunks; ++c) {
          tma_load_2d(sm.k + c * kChunkBytes, &tm_k, g * D + 64 * c, k0, &sm.kv_full);
          tma_load_2d(sm.v + c * kChunkBytes, &tm_v, g * D + 64 * c, k0, &sm.kv_full);
        }
      }
      int issued = 0;
      for (int j = 0; j < nqb; ++j) {
        const int b = j & 1;
        if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait_bounded(&sm.q_empty[b], ((j - 2) >> 1) & 1, a.status,
                                                                  &sm.abort)))
          break;
        const long long rb = row_first + (long long)j * kR;
        for (int c = lane; c < kR; c += 32) {
          const long long pk = rb + c, i = pk / gs;
          RowInfo ri{0.f, 0.f, 0, 0};
          if (i < i_end) {
            ri.n = query_n(a, i);
            ri.lo = first_key(ri.n, a.window);
            const long long pair = i * a.H + g * gs + (int)(pk % gs);
            ri.l2 = l2[pair];
            ri.delta = delta[pair];
          }
          sm.rows[b][c] = ri;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&sm.q_full[b], 2u * T::kBytes);
#pragma unroll
          for (int c = 0; c < T::kChunks; ++c) {
            tma_load_3d(sm.q[b] + c * kChunkBytes, &tm_q, 64 * c, g * gs, (int)(rb / gs), &sm.q_full[b]);
            tma_load_3d(sm.g[b] + c * kChunkBytes, &tm_g, 64 * c, g * gs, (int)(rb / gs), &sm.q_full[b]);
          }
        }
        __syncwarp();
        issued = j + 1;
      }
      // No copy may still be landing in shared memory when the CTA exits.
      if (lane == 0) {
        mbar_wait_bounded(&sm.kv_full, 0, a.status);
        for (int j = max(0, issued - 2); j < issued; ++j) mbar_wait_bounded(&sm.q_full[j & 1], (j >> 1) & 1, a.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (nqb > 0) {
      constexpr uint32_t idesc_ss = tc::idesc_f32acc(tc::kFmtBF16, false, kR, kR);
      constexpr uint32_t idesc_ts = tc::idesc_f32acc(tc::kFmtBF16, true, kR, D);
      constexpr uint64_t st = (16 * 128) >> 4;  // one K step of an MN-major operand: 16 rows
      const uint64_t dk = tc::sdesc_sw128(smem_u32(sm.k), 16, 1024);
      const uint64_t dv = tc::sdesc_sw128(smem_u32(sm.v), 16, 1024);
      auto wait = [&](uint64_t* bar, int phase) {
        return __all_sync(0xffffffffu, mbar_wait_bounded(bar, (unsigned)(phase & 1), a.status, &sm.abort));
      };
      bool ok = wait(&sm.kv_full, 0);
      for (int j = 0; ok && j < nqb; ++j) {
        const int b = j & 1;
        ok = wait(&sm.q_full[b], j >> 1) && (j == 0 || wait(&sm.pv_done, j - 1));
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t qa = smem_u32(sm.q[b]), ga = smem_u32(sm.g[b]);
        const uint64_t dq = tc::sdesc_sw128(qa, 16, 1024), dg = tc::sdesc_sw128(ga, 16, 1024);
        // S^T = K Q^T and dP^T = V dout^T (M = 128 keys, N = 128 rows, K = D).
#pragma unroll
        for (int c4 = 0; c4 < T::kChunks; ++c4) {
          const uint64_t c = (uint64_t)((c4 * kChunkBytes) >> 4);
          tc::mma4_f16_ss(tmem + kColS, dk + c, dk + c + 2, dk + c + 4, dk + c + 6, dq + c, dq + c + 2, dq + c + 4,
                          dq + c + 6, idesc_ss, c4 > 0 ? 1u : 0u);
          tc::mma4_f16_ss(tmem + kColP, dv + c, dv + c + 2, dv + c + 4, dv + c + 6, dg + c, dg + c + 2, dg + c + 4,
                          dg + c + 6, idesc_ss, c4 > 0 ? 1u : 0u);
        }
        tc::commit_elect(&sm.s_full);
        // dV += P^T dout and dK += dS^T Q (M = 128 keys, N = D, K = 128 rows;
        // A bf16 in TMEM, 8 columns per 16-row step; B MN-major), in two
        // halves of 64 rows, each as soon as its P and dS are written.
        const uint64_t gm = tc::sdesc_sw128(ga, kChunkBytes, 1024), qm = tc::sdesc_sw128(qa, kChunkBytes, 1024);
#pragma unroll 1
        for (int c4 = 0; c4 < kR / 64; ++c4) {
          ok = wait(&sm.p_ready[c4], j);
          if (!ok) break;
          tc::fence_after_sync();
          const uint64_t c = 4 * st * c4;
          const uint32_t pa = tmem + kColS + 32 * c4, sa = tmem + kColP + 32 * c4;
          const uint32_t acc = (j > 0 || c4 > 0) ? 1u : 0u;
          tc::mma4_f16_ts(tmem + kColAcc, pa, pa + 8, pa + 16, pa + 24, gm + c, gm + c + st, gm + c + 2 * st,
                          gm + c + 3 * st, idesc_ts, acc);
          tc::mma4_f16_ts(tmem + kColAcc + D, sa, sa + 8, sa + 16, sa + 24, qm + c, qm + c + st, qm + c + 2 * st,
                          qm + c + 3 * st, idesc_ts, acc);
        }
        if (!ok) break;
        tc::commit_elect(&sm.pv_done);
        tc::commit_elect(&sm.q_empty[b]);
      }
      // Every MMA has finished before tensor memory is released.
      tc::commit_elect(&sm.drain);
      mbar_wait_bounded(&sm.drain, 0, a.status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ elementwise / epilogue
    const int row = 32 * (warp & 3) + lane;  // key row == TMEM lane
    const int key = k0 + row;
    const uint32_t lane_tmem = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const float sl2 = a.scale * kLog2e;
    for (int j = 0; j < nqb; ++j) {
      const int b = j & 1;
      mbar_wait_bounded(&sm.s_full, (unsigned)(j & 1), a.status, &sm.abort);
      tc::fence_after_sync();
      auto ready = [&](int half) {
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_ready[half]);
      };
      elementwise(
          lane_tmem, sl2, true,
          [&](int c, float* lv, float* dv) {
            const RowInfo ri = sm.rows[b][c];
            *lv = ri.l2;
            *dv = ri.delta;
            return key >= ri.lo && key < ri.n;
          },
          [&] { ready(0); });
      ready(1);
    }
    if (nqb > 0) mbar_wait_bounded(&sm.pv_done, (unsigned)((nqb - 1) & 1), a.status, &sm.abort);
    tc::fence_after_sync();
    const long long off = (long long)key * a.G * D + (long long)g * D;
    if (nqb > 0) {
      store_row<D>(lane_tmem + kColAcc, a.dv + off, 1.f, row < k_valid);
      store_row<D>(lane_tmem + kColAcc + D, a.dk + off, a.scale, row < k_valid);
    } else if (row < k_valid) {  // no query attends these keys
      for (int d = 0; d < D; d += 4) {
        *reinterpret_cast<float4*>(a.dv + off + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(a.dk + off + d) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
    tc::tmem_relinquish();
  }
}

// ------------------------------------------------------------------ dQ
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_tc_kernel(const BwdArgs a, const float* __restrict__ delta, const float* __restrict__ l2,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_g) {
  using T = Tile<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  QTcSmem<D>& sm = *reinterpret_cast<QTcSmem<D>*>(smem_raw + ((1024u - (raw & 1023u)) & 1023u));
  allow_dependent_launch();
  grid_dependency_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, gs = a.H / a.G;
  const int blk = gridDim.x - 1 - blockIdx.x;  // latest (longest) causal rows first
  const int qpb = kR / gs;
  const long long i0 = (long long)blk * qpb;
  const long long i1 = min((long long)a.n_q, i0 + qpb) - 1;
  const int n_min = query_n(a, i0), n_max = query_n(a, i1);
  const int jt0 = first_key(n_min, a.window) / kR;
  const int nt = (n_max + kR - 1) / kR - jt0;

  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.kv_full[b], 1);
      mbar_init(&sm.kv_empty[b], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_ready[0], 4);
    mbar_init(&sm.p_ready[1], 4);
    mbar_init(&sm.pv_done, 1);
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(&sm.tmem_base, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    if (lane == 0 && nt > 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_g);
      mbar_arrive_expect_tx(&sm.q_full, 2u * T::kBytes);
#pragma unroll
      for (int c = 0; c < T::kChunks; ++c) {
        tma_load_3d(sm.q + c * kChunkBytes, &tm_q, 64 * c, g * gs, (int)i0, &sm.q_full);
        tma_load_3d(sm.g + c * kChunkBytes, &tm_g, 64 * c, g * gs, (int)i0, &sm.q_full);
      }
      int issued = 0;
      for (int t = 0; t < nt; ++t) {
        const int b = t & 1;
        if (t >= 2 && !mbar_wait_bounded(&sm.kv_empty[b], ((t - 2) >> 1) & 1, a.status, &sm.abort)) break;
        mbar_arrive_expect_tx(&sm.kv_full[b], 2u * T::kBytes);
        const int y = (jt0 + t) * kR;
#pragma unroll
        for (int c = 0; c < T::kChunks; ++c) {
          tma_load_2d(sm.k[b] + c * kChunkBytes, &tm_k, g * D + 64 * c, y, &sm.kv_full[b]);
          tma_load_2d(sm.v[b] + c * kChunkBytes, &tm_v, g * D + 64 * c, y, &sm.kv_full[b]);
        }
        issued = t + 1;
      }
      mbar_wait_bounded(&sm.q_full, 0, a.status);
      for (int t = max(0, issued - 2); t < issued; ++t) mbar_wait_bounded(&sm.kv_full[t & 1], (t >> 1) & 1, a.status);
    }
  } else if (warp == 1) {
    if (nt > 0) {
      constexpr uint32_t idesc_ss = tc::idesc_f32acc(tc::kFmtBF16, false, kR, kR);
      constexpr uint32_t idesc_ts = tc::idesc_f32acc(tc::kFmtBF16, true, kR, D);
      constexpr uint64_t st = (16 * 128) >> 4;
      const uint64_t dq = tc::sdesc_sw128(smem_u32(sm.q), 16, 1024);
      const uint64_t dg = tc::sdesc_sw128(smem_u32(sm.g), 16, 1024);
      auto wait = [&](uint64_t* bar, int phase) {
        return __all_sync(0xffffffffu, mbar_wait_bounded(bar, (unsigned)(phase & 1), a.status, &sm.abort));
      };
      bool ok = wait(&sm.q_full, 0);
      for (int t = 0; ok && t < nt; ++t) {
        const int b = t & 1;
        ok = wait(&sm.kv_full[b], t >> 1) && (t == 0 || wait(&sm.pv_done, t - 1));
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t ka = smem_u32(sm.k[b]), va = smem_u32(sm.v[b]);
        const uint64_t dk = tc::sdesc_sw128(ka, 16, 1024), dv = tc::sdesc_sw128(va, 16, 1024);
        // S = Q K^T and dP = dout V^T (M = 128 rows, N = 128 keys, K = D).
#pragma unroll
        for (int c4 = 0; c4 < T::kChunks; ++c4) {
          const uint64_t c = (uint64_t)((c4 * kChunkBytes) >> 4);
          tc::mma4_f16_ss(tmem + kColS, dq + c, dq + c + 2, dq + c + 4, dq + c + 6, dk + c, dk + c + 2, dk + c + 4,
                          dk + c + 6, idesc_ss, c4 > 0 ? 1u : 0u);
          tc::mma4_f16_ss(tmem + kColP, dg + c, dg + c + 2, dg + c + 4, dg + c + 6, dv + c, dv + c + 2, dv + c + 4,
                          dv + c + 6, idesc_ss, c4 > 0 ? 1u : 0u);
        }
        tc::commit_elect(&sm.s_full);
        // dQ += dS K (M = 128 rows, N = D, K = 128 keys; B = K tile MN-major),
        // in two halves of 64 keys, each as soon as its dS is written.
        const uint64_t km = tc::sdesc_sw128(ka, kChunkBytes, 1024);
#pragma unroll 1
        for (int c4 = 0; c4 < kR / 64; ++c4) {
          ok = wait(&sm.p_ready[c4], t);
          if (!ok) break;
          tc::fence_after_sync();
          const uint64_t c = 4 * st * c4;
          const uint32_t sa = tmem + kColP + 32 * c4;
          tc::mma4_f16_ts(tmem + kColAcc, sa, sa + 8, sa + 16, sa + 24, km + c, km + c + st, km + c + 2 * st,
                          km + c + 3 * st, idesc_ts, (t > 0 || c4 > 0) ? 1u : 0u);
        }
        if (!ok) break;
        tc::commit_elect(&sm.pv_done);
        tc::commit_elect(&sm.kv_empty[b]);
      }
      tc::commit_elect(&sm.drain);
      mbar_wait_bounded(&sm.drain, 0, a.status);
    }
  } else if (warp >= 4) {
    const int row = 32 * (warp & 3) + lane;  // packed row == TMEM lane
    const long long pk = (long long)blk * kR + row;
    const long long qi = pk / gs;
    const int h = g * gs + (int)(pk % gs);
    const bool row_ok = qi < a.n_q;
    const int n_r = row_ok ? query_n(a, qi) : 0;
    const int lo_r = first_key(n_r, a.window);
    const long long pair = qi * a.H + h;
    const float lr = row_ok ? l2[pair] : 0.f, dr = row_ok ? delta[pair] : 0.f;
    const uint32_t lane_tmem = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const float sl2 = a.scale * kLog2e;
    for (int t = 0; t < nt; ++t) {
      mbar_wait_bounded(&sm.s_full, (unsigned)(t & 1), a.status, &sm.abort);
      tc::fence_after_sync();
      const int key0 = (jt0 + t) * kR;
      auto ready = [&](int half) {
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_ready[half]);
      };
      elementwise(
          lane_tmem, sl2, false,
          [&](int c, float* lv, float* dv) {
            *lv = lr;
            *dv = dr;
            return key0 + c >= lo_r && key0 + c < n_r;
          },
          [&] { ready(0); });
      ready(1);
    }
    if (nt > 0) mbar_wait_bounded(&sm.pv_done, (unsigned)((nt - 1) & 1), a.status, &sm.abort);
    tc::fence_after_sync();
    float* dst = a.dq + qi * a.H * D + (long long)h * D;
    if (nt > 0) {
      store_row<D>(lane_tmem + kColAcc, dst, a.scale, row_ok);
    } else if (row_ok) {
      for (int d = 0; d < D; d += 4) *reinterpret_cast<float4*>(dst + d) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
    tc::tmem_relinquish();
  }
}

// Two fp32 arrays of n4 float4 groups to bf16 (same layout).
__global__ void __launch_bounds__(256) pair_to_bf16_kernel(const float4* __restrict__ x, const float4* __restrict__ y,
                                                           uint2* __restrict__ x16, uint2* __restrict__ y16, long long n4) {
  allow_dependent_launch();
  grid_dependency_wait();
  for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < n4; i += (long long)gridDim.x * 256) {
    const float4 a = x[i], b = y[i];
    x16[i] = make_uint2(tc::pack_bf16(a.x, a.y), tc::pack_bf16(a.z, a.w));
    y16[i] = make_uint2(tc::pack_bf16(b.x, b.y), tc::pack_bf16(b.z, b.w));
  }
}

cudaError_t to_bf16(const float* x, const float* y, uint16_t* x16, uint16_t* y16, long long elems, cudaStream_t s) {
  const float4* x4 = reinterpret_cast<const float4*>(x);
  const float4* y4 = reinterpret_cast<const float4*>(y);
  uint2* x2 = reinterpret_cast<uint2*>(x16);
  uint2* y2 = reinterpret_cast<uint2*>(y16);
  long long n4 = elems / 4;
  void* args[] = {&x4, &y4, &x2, &y2, &n4};
  const long long blocks = min((n4 + 255) / 256, 152LL * 16);
  return launch_pdl(reinterpret_cast<const void*>(pair_to_bf16_kernel), dim3((unsigned)max(blocks, 1LL)), dim3(256), 0,
                    s, args);
}

template <int D>
int launch_d(const BwdArgs& a, const float* delta, const float* l2, const uint16_t* q16, const uint16_t* g16,
             const uint16_t* k16, const uint16_t* v16, cudaStream_t s) {
  const int gs = a.H / a.G;
  CUtensorMap tm_k, tm_v, tm_q, tm_g;
  // K, V: [n_kv][G*D] bf16, boxes of 64 elements x 128 keys.
  const uint64_t kdims[2] = {(uint64_t)a.G * D, (uint64_t)a.n_kv};
  const uint64_t kstr[1] = {(uint64_t)a.G * D * 2};
  const uint32_t kbox[2] = {64, (uint32_t)kR};
  // Q, dout: [n_q][H][D] bf16; a block is 64 elements x gs heads x 128/gs queries.
  const uint64_t qdims[3] = {(uint64_t)D, (uint64_t)a.H, (uint64_t)a.n_q};
  const uint64_t qstr[2] = {(uint64_t)D * 2, (uint64_t)a.H * D * 2};
  const uint32_t qbox[3] = {64, (uint32_t)gs, (uint32_t)(kR / gs)};
  if (!make_tmap(&tm_k, k16, 2, kdims, kstr, kbox, true, kSwizzle128) ||
      !make_tmap(&tm_v, v16, 2, kdims, kstr, kbox, true, kSwizzle128) ||
      !make_tmap(&tm_q, q16, 3, qdims, qstr, qbox, true, kSwizzle128) ||
      !make_tmap(&tm_g, g16, 3, qdims, qstr, qbox, true, kSwizzle128))
    return ATTN_ERR_UNSUPPORTED;
  const size_t kv_smem = sizeof(KvTcSmem<D>) + 1024, q_smem = sizeof(QTcSmem<D>) + 1024;
  auto kv_kern = bwd_dkdv_tc_kernel<D>;
  auto q_kern = bwd_dq_tc_kernel<D>;
  if (!set_smem_limit(reinterpret_cast<const void*>(kv_kern), kv_smem) ||
      !set_smem_limit(reinterpret_cast<const void*>(q_kern), q_smem))
    return ATTN_ERR_CUDA;
  BwdArgs aa = a;
  const float* d = delta;
  const float* l = l2;
  void* args[] = {&aa, &d, &l, &tm_k, &tm_v, &tm_q, &tm_g};
  const long long kb = (a.n_kv + kR - 1) / kR;
  const long long qb = ((long long)a.n_q * gs + kR - 1) / kR;
  // The two kernels are independent: dQ runs on a side stream forked after
  // the pre-passes and joined before the caller's stream moves on, so its
  // CTAs fill the SMs that the dK/dV grid's uneven causal tail leaves idle.
  return launch_forked(s, reinterpret_cast<const void*>(kv_kern), dim3((unsigned)kb, (unsigned)a.G), kv_smem,
                       reinterpret_cast<const void*>(q_kern), dim3((unsigned)qb, (unsigned)a.G), q_smem,
                       dim3(kThreads), args);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

bool backward_bf16_supported(const BwdArgs& a) {
  if (a.D != 64 && a.D != 128) return false;
  if (a.G > 65535) return false;
  const int gs = a.H / a.G;
  if (gs <= 0 || gs > kR || (gs & (gs - 1)) != 0) return false;
  const uintptr_t al = reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) |
                       reinterpret_cast<uintptr_t>(a.v) | reinterpret_cast<uintptr_t>(a.out) |
                       reinterpret_cast<uintptr_t>(a.dout) | reinterpret_cast<uintptr_t>(a.dq) |
                       reinterpret_cast<uintptr_t>(a.dk) | reinterpret_cast<uintptr_t>(a.dv);
  return al % 16 == 0;
}

// delta and the base-2 log-sum-exp per (row, head), then bf16 copies of q,
// dout, k and v, each part 256-byte aligned.
size_t backward_bf16_scratch_bytes(const BwdArgs& a) {
  const size_t pairs = (size_t)a.n_q * a.H, qe = pairs * a.D, ke = (size_t)a.n_kv * a.G * a.D;
  return 2 * align256(pairs * 4) + 2 * align256(qe * 2) + 2 * align256(ke * 2);
}

int launch_backward_bf16(const BwdArgs& a, cudaStream_t s) {
  const long long pairs = (long long)a.n_q * a.H;
  if (pairs == 0 || a.n_kv == 0) return ATTN_OK;
  if (!backward_bf16_supported(a)) return ATTN_ERR_UNSUPPORTED;
  const size_t qe = (size_t)pairs * a.D, ke = (size_t)a.n_kv * a.G * a.D;
  const size_t off_l2 = align256((size_t)pairs * 4), off_q = off_l2 + align256((size_t)pairs * 4);
  const size_t off_g = off_q + align256(qe * 2), off_k = off_g + align256(qe * 2), off_v = off_k + align256(ke * 2);
  void* scratch = nullptr;
  if (scratch_alloc(&scratch, backward_bf16_scratch_bytes(a), s) != cudaSuccess) return ATTN_ERR_CUDA;
  char* base = static_cast<char*>(scratch);
  float* delta = reinterpret_cast<float*>(base);
  float* l2 = reinterpret_cast<float*>(base + off_l2);
  uint16_t* q16 = reinterpret_cast<uint16_t*>(base + off_q);
  uint16_t* g16 = reinterpret_cast<uint16_t*>(base + off_g);
  uint16_t* k16 = reinterpret_cast<uint16_t*>(base + off_k);
  uint16_t* v16 = reinterpret_cast<uint16_t*>(base + off_v);
  int rc = ATTN_OK;
  if (launch_bwd_prep(a, delta, l2, s) != cudaSuccess || to_bf16(a.q, a.dout, q16, g16, (long long)qe, s) != cudaSuccess ||
      to_bf16(a.k, a.v, k16, v16, (long long)ke, s) != cudaSuccess)
    rc = ATTN_ERR_CUDA;
  if (rc == ATTN_OK)
    rc = a.D == 128 ? launch_d<128>(a, delta, l2, q16, g16, k16, v16, s) : launch_d<64>(a, delta, l2, q16, g16, k16, v16, s);
  if (scratch_free(scratch, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
  return rc;
}

}  // namespace attn
