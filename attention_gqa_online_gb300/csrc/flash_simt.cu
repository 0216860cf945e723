// flash_simt.cu -- fp32 CUDA-core flash attention (forward, prefill, and the
// generic decode path).
//
// One CTA owns 64 packed rows of one kv head g: row r of the block is the
// pair (query i, head g*gs + j) with i*gs + j = 64*block + r, so every K/V
// tile loaded into shared memory serves all gs query heads that read kv head
// g (the GQA map kv_head = head / (n_heads / n_kv_heads) of all three shader
// pages).  Keys are walked in tiles of 64 with a per-tile online softmax: the
// tile max is taken first, then one correction factor per row per tile
// (cera attention_prefill.wgsl, fn attention_prefill: tile max, correction
// exp(m - m'), p = exp(s - m'), running sum and accumulator rescale).  The
// exponentials are base 2 with scale*log2(e) folded into the scores, which is
// the same function.  Per-row windows implement causal / full / cross /
// prefill / decode masking, and a sliding window keeps the last `window` keys
// of each row's window; key tiles outside every row's window of the block
// are never loaded.
//
// Thread layout (256 threads): rg = tid / 16 owns rows 4rg..4rg+3; cl = tid %
// 16 owns score columns cl + 16j (j < 4) and output columns 4cl + 64j.  Row
// reductions stay inside a half-warp (xor shuffles 8, 4, 2, 1).
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace attn {

int launch_flash_simt_plain(const FlashArgs& a, cudaStream_t s);

namespace {

constexpr int BM = 64;   // packed rows per CTA
constexpr int BN = 64;   // keys per tile
constexpr int NT = 256;  // threads per CTA

template <int DMAX>
struct SimtSmem {
  static constexpr int QS = DMAX + 4;  // padded row stride of the Q and K tiles (floats)
  static constexpr int PS = BM + 4;    // padded row stride of the transposed P tile
  float q[BM * QS];
  float k[2][BN * QS];
  float v[2][BN * DMAX];
  float p[BN * PS];
  int row_n[BM];
  int row_lo[BM];
};

// Issues the async copies of one (rows x DMAX) tile into shared memory, with
// zero fill for rows >= valid_rows, columns >= D and rows whose src(r) is
// nullptr.  src(r) is the global address of row r's first element; `any` is
// a valid address used for the zero-fill copies.
template <int DMAX, int STRIDE, bool VEC, typename SrcFn>
__device__ __forceinline__ void load_tile(float* dst, int rows, int valid_rows, int D, SrcFn src, const float* any) {
  if constexpr (VEC) {
    constexpr int F = DMAX / 4;
    for (int idx = threadIdx.x; idx < rows * F; idx += NT) {
      const int r = idx / F, f = idx % F;
      const float* row = r < valid_rows && 4 * f < D ? src(r) : nullptr;
      cp_async16(dst + r * STRIDE + 4 * f, row ? row + 4 * f : any, row ? 16u : 0u);
    }
  } else {
    for (int idx = threadIdx.x; idx < rows * DMAX; idx += NT) {
      const int r = idx / DMAX, c = idx % DMAX;
      const float* row = r < valid_rows && c < D ? src(r) : nullptr;
      cp_async4(dst + r * STRIDE + c, row ? row + c : any, row ? 4u : 0u);
    }
  }
}

template <int DMAX, bool VEC, bool PAGED>
__global__ void __launch_bounds__(NT, 1) flash_simt_kernel(const FlashArgs a) {
  using Smem = SimtSmem<DMAX>;
  constexpr int QS = Smem::QS, PS = Smem::PS;
  constexpr int OC = DMAX / 64 > 0 ? DMAX / 64 : 1;  // float4 output groups per thread
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);

  // Programmatic dependent launch (see common.cuh): no global access before
  // the previous kernel in the stream has completed.
  allow_dependent_launch();
  grid_dependency_wait();
  const int tid = threadIdx.x;
  const int rg = tid >> 4, cl = tid & 15;
  const int r0 = 4 * rg;
  const int g = blockIdx.y;
  const int blk = gridDim.x - 1 - blockIdx.x;  // heaviest (latest) causal rows first
  const int gs = a.H / a.G;
  const int D = a.D;

  long long base_pos = a.base_pos;
  if (a.kv_pos_dev != nullptr) {
    const unsigned kp = *a.kv_pos_dev;
    if (tid == 0 && blk == 0 && (long long)kp >= (long long)a.cap) record_status(a.status, ATTN_ERR_INVALID_ARG);
    base_pos = kp;
  }

  // Window of every packed row of this block.
  if (tid < BM) {
    const long long packed = (long long)blk * BM + tid;
    const long long i = packed / gs;
    int n = 0;
    if (i < a.n_q) {
      if (a.causal) {
        long long w = base_pos + i + 1;
        n = (int)(w < a.cap ? w : a.cap);
      } else {
        n = a.n_all;
      }
    }
    sm.row_n[tid] = n;
    sm.row_lo[tid] = first_key(n, a.window);
  }
  __syncthreads();
  // Keys [t_begin, n_max) cover every row's window; t_begin is tile-aligned.
  int n_max = 0, lo_min = INT_MAX;
  for (int r = 0; r < BM; ++r) {
    n_max = max(n_max, sm.row_n[r]);
    if (sm.row_n[r] > 0) lo_min = min(lo_min, sm.row_lo[r]);
  }
  const int t_begin = n_max > 0 ? lo_min / BN * BN : 0;
  int my_n[4], my_lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    my_n[i] = sm.row_n[r0 + i];
    my_lo[i] = sm.row_lo[r0 + i];
  }

  // Q tile (rows past n_q are zero-filled and never stored).
  const long long row_base = (long long)blk * BM;
  const long long rows_left = (long long)a.n_q * gs - row_base;
  const int q_valid = (int)(rows_left < BM ? rows_left : BM);
  auto q_src = [&](int r) {
    const long long packed = row_base + r;
    const long long i = packed / gs;
    const int h = g * gs + (int)(packed % gs);
    return a.q + i * a.q_row_stride + (long long)h * D;
  };
  load_tile<DMAX, QS, VEC>(sm.q, BM, q_valid, D, q_src, a.q);

  const int n_tiles = (n_max - t_begin + BN - 1) / BN;
  // Row t of K or V (through the block table for a paged cache; nullptr for
  // a page outside the pool, which then reads as zeros).
  auto kv_src = [&](const float* base, int t0) {
    return [=](int r) -> const float* {
      long long row = t0 + r;
      if constexpr (PAGED) {
        row = paged_row(a.block_table, a.page_rows, a.num_pages, t0 + r, a.status);
        if (row < 0) return nullptr;
      }
      return base + row * a.kv_row_stride + (long long)g * D;
    };
  };
  if (n_tiles > 0) {
    load_tile<DMAX, QS, VEC>(sm.k[0], BN, min(BN, n_max - t_begin), D, kv_src(a.k, t_begin), a.q);
    load_tile<DMAX, DMAX, VEC>(sm.v[0], BN, min(BN, n_max - t_begin), D, kv_src(a.v, t_begin), a.q);
  }
  cp_async_commit();

  const float sl2 = a.scale * kLog2e;
  float m_run[4], l_run[4];
  float o[4][OC * 4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int c = 0; c < OC * 4; ++c) o[i][c] = 0.f;
  }

  // Turns the pairs (d, d + D/2) of `rows` rows of a shared-memory tile, row
  // r at position pos(r), by the RoPE table.
  auto rope_rows = [&](float* tile, int rows, auto pos) {
    const int half = D / 2;
    for (int idx = tid; idx < rows * half; idx += NT) {
      const int r = idx / half, d = idx % half;
      const float* cs = a.rope + pos(r) * D;
      const float c = cs[d], s = cs[half + d];
      const float x = tile[r * QS + d], y = tile[r * QS + half + d];
      tile[r * QS + d] = x * c - y * s;
      tile[r * QS + half + d] = y * c + x * s;
    }
  };

  for (int it = 0; it < n_tiles; ++it) {
    const int buf = it & 1;
    const int t0 = t_begin + it * BN;
    if (it + 1 < n_tiles) {
      const int t1 = t0 + BN;
      const int valid = min(BN, n_max - t1);
      load_tile<DMAX, QS, VEC>(sm.k[buf ^ 1], BN, valid, D, kv_src(a.k, t1), a.q);
      load_tile<DMAX, DMAX, VEC>(sm.v[buf ^ 1], BN, valid, D, kv_src(a.v, t1), a.q);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (a.rope != nullptr && it == 0) {
      // RoPE: Q once (query i at base_pos + i); K arrives turned (pre-pass).
      rope_rows(sm.q, q_valid, [&](int r) { return base_pos + (row_base + r) / gs; });
      __syncthreads();
    }

    // S = Q K^T for rows r0..r0+3, keys cl + 16j.
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
    // Each group of 8 products is summed on its own before it joins the
    // running dot product: 16 roundings of the large partial sum instead of
    // 128 keeps fp32 scores within a few ulp for widely spread inputs.  The
    // group runs as two chains (even and odd elements) of paired fmas, one
    // instruction for two products, on the register pairs the float4 loads
    // fill.
    const float* kt = sm.k[buf];
#pragma unroll 2
    for (int d = 0; d < DMAX; d += 8) {
      float4 qa[4][2], kb[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        qa[i][0] = *reinterpret_cast<const float4*>(&sm.q[(r0 + i) * QS + d]);
        qa[i][1] = *reinterpret_cast<const float4*>(&sm.q[(r0 + i) * QS + d + 4]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        kb[j][0] = *reinterpret_cast<const float4*>(&kt[(cl + 16 * j) * QS + d]);
        kb[j][1] = *reinterpret_cast<const float4*>(&kt[(cl + 16 * j) * QS + d + 4]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float e0 = 0.f, e1 = 0.f;
          fma2_acc(e0, e1, qa[i][0].x, qa[i][0].y, kb[j][0].x, kb[j][0].y);
          fma2_acc(e0, e1, qa[i][0].z, qa[i][0].w, kb[j][0].z, kb[j][0].w);
          fma2_acc(e0, e1, qa[i][1].x, qa[i][1].y, kb[j][1].x, kb[j][1].y);
          fma2_acc(e0, e1, qa[i][1].z, qa[i][1].w, kb[j][1].z, kb[j][1].w);
          s[i][j] += e0 + e1;
        }
    }

    // Mask, tile max, correction, exponentials, running sum.
    float p[4][4], corr_row[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int t = t0 + cl + 16 * j;
        s[i][j] = (t >= my_lo[i] && t < my_n[i]) ? s[i][j] * sl2 : -INFINITY;
        mx = fmaxf(mx, s[i][j]);
      }
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m_run[i], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = ex2(m_run[i] - m_use);
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        p[i][j] = ex2(s[i][j] - m_use);
        sum += p[i][j];
      }
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l_run[i] = l_run[i] * corr + sum;
      m_run[i] = m_new;
      corr_row[i] = corr;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<float4*>(&sm.p[(cl + 16 * j) * PS + r0]) = make_float4(p[0][j], p[1][j], p[2][j], p[3][j]);
    __syncthreads();

    // O = O * corr + P V, with P V of this tile summed on its own first (one
    // rounding of the long-running accumulator per tile, not per key).
    float t[4][OC * 4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < OC * 4; ++c) t[i][c] = 0.f;
    const float* vt = sm.v[buf];
#pragma unroll 4
    for (int kk = 0; kk < BN; ++kk) {
      const float4 pv = *reinterpret_cast<const float4*>(&sm.p[kk * PS + r0]);
      const float pr[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
      for (int jj = 0; jj < OC; ++jj) {
        const int col = (DMAX >= 64) ? (4 * cl + 64 * jj) : (4 * cl);
        float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (DMAX >= 64 || col < DMAX) vv = *reinterpret_cast<const float4*>(&vt[kk * DMAX + col]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // two output columns per paired fma, same order per column
          fma2_acc(t[i][4 * jj + 0], t[i][4 * jj + 1], pr[i], pr[i], vv.x, vv.y);
          fma2_acc(t[i][4 * jj + 2], t[i][4 * jj + 3], pr[i], pr[i], vv.z, vv.w);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < OC * 4; ++c) o[i][c] = fmaf(o[i][c], corr_row[i], t[i][c]);
    __syncthreads();
  }

  // Epilogue: normalise, store rows, store (max, log sum).
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + i;
    if (r >= q_valid) continue;
    const long long packed = row_base + r;
    const long long qi = packed / gs;
    const int h = g * gs + (int)(packed % gs);
    const float inv = (l_run[i] == 0.f) ? 0.f : 1.f / l_run[i];
    float* dst = a.out + qi * a.out_row_stride + (long long)h * D;
#pragma unroll
    for (int jj = 0; jj < OC; ++jj) {
      const int col = (DMAX >= 64) ? (4 * cl + 64 * jj) : (4 * cl);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (col + c < D) dst[col + c] = o[i][4 * jj + c] * inv;
    }
    if (a.lse != nullptr && cl == 0) {
      float* l2 = a.lse + (qi * a.H + h) * 2;
      const bool empty = (l_run[i] == 0.f);
      l2[0] = empty ? kEmptyLse : m_run[i] * kLn2;
      l2[1] = empty ? kEmptyLse : logf(l_run[i]);
    }
  }
}

template <int DMAX, bool VEC, bool PAGED>
int launch_one(const FlashArgs& a, cudaStream_t s) {
  const int gs = a.H / a.G;
  const long long rows = (long long)a.n_q * gs;
  const long long nb = (rows + BM - 1) / BM;
  if (nb == 0) return 0;
  if (nb > 0x7fffffffLL || a.G > 65535) return ATTN_ERR_UNSUPPORTED;
  const size_t smem = sizeof(SimtSmem<DMAX>);
  auto kern = flash_simt_kernel<DMAX, VEC, PAGED>;
  if (!set_smem_limit(reinterpret_cast<const void*>(kern), smem)) return ATTN_ERR_CUDA;
  FlashArgs aa = a;
  void* args[] = {&aa};
  return launch_pdl(reinterpret_cast<const void*>(kern), dim3((unsigned)nb, (unsigned)a.G), dim3(NT), smem, s, args) ==
                 cudaSuccess
             ? 0
             : ATTN_ERR_CUDA;
}

}  // namespace

// RoPE only: K turned (kv_rows x kv_row_stride floats).
size_t flash_simt_scratch_bytes(const FlashArgs& a) {
  const long long kv_rows = a.causal ? min((long long)a.cap, a.base_pos + a.n_q) : a.n_all;
  if (a.rope == nullptr || kv_rows <= 0 || a.n_q == 0) return 0;
  return scratch_round((size_t)kv_rows * a.kv_row_stride * sizeof(float));
}

int launch_flash_simt(const FlashArgs& a0, cudaStream_t s) {
  // RoPE: K is turned once into stream-ordered scratch (rows of G*D floats,
  // row t at position t) and the kernel turns Q.
  FlashArgs a = a0;
  void* scratch = nullptr;
  const long long kv_rows = a.causal ? min((long long)a.cap, a.base_pos + a.n_q) : a.n_all;
  if (a.rope != nullptr && kv_rows > 0) {
    if (scratch_alloc(&scratch, flash_simt_scratch_bytes(a), s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (launch_rope_k(a.k, static_cast<float*>(scratch), a.rope, kv_rows, a.G, a.D, s) != cudaSuccess) {
      scratch_free(scratch, s);
      return ATTN_ERR_CUDA;
    }
    a.k = static_cast<const float*>(scratch);
  }
  int rc = launch_flash_simt_plain(a, s);
  if (scratch != nullptr && scratch_free(scratch, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
  return rc;
}

int launch_flash_simt_plain(const FlashArgs& a, cudaStream_t s) {
  const bool vec = (a.D % 4 == 0) && (a.q_row_stride % 4 == 0) && (a.kv_row_stride % 4 == 0) &&
                   ((reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) |
                     reinterpret_cast<uintptr_t>(a.v)) % 16 == 0);
  // Paged caches get their own instances (the row mapping stays out of the
  // contiguous kernels' load loops).
  if (a.block_table != nullptr) {
    if (a.D <= 64) return vec ? launch_one<64, true, true>(a, s) : launch_one<64, false, true>(a, s);
    return vec ? launch_one<128, true, true>(a, s) : launch_one<128, false, true>(a, s);
  }
  if (a.D <= 64) return vec ? launch_one<64, true, false>(a, s) : launch_one<64, false, false>(a, s);
  return vec ? launch_one<128, true, false>(a, s) : launch_one<128, false, false>(a, s);
}

}  // namespace attn
