// flash_tc.cu -- tcgen05 tensor-core flash attention (forward and prefill).
//
// Operation: softmax(scale * Q K^T) V over per-row causal / full / cross /
// prefill windows, with the running max / sum of the pages' online softmax
// (cera attention_prefill.wgsl, fn attention_prefill: per-tile max,
// correction, exponentials, running sum; meganeura attention.wgsl, fn main:
// the final (max, log sum) store).  Both contractions run on the 5th-generation
// tensor cores with TF32 operands and fp32 accumulation in tensor memory.
//
// One CTA owns 128 packed rows of one kv head g: row r is (query i, head
// g*gs + j) with i*gs + j = 128*block + r, so each K/V tile feeds all gs
// query heads that share it.  Keys are walked in tiles of 128.
//
// Warp roles (256 threads):
//   warp 0      TMA producer: K tile (128 keys x D, 128-byte swizzle, K-major
//               operand) and V tile (same box, 32-byte-atom swizzle, MN-major
//               operand) into a ring of 64 KB shared-memory slots.
//   warp 1      tensor-memory allocation; one thread issues every MMA:
//                 S_b = Q K_j^T      (A = Q in TMEM, B = K tile)      M=128 N=128
//                 O  += P_j V_j      (A = P in TMEM over S_b, B = V)  M=128 N=D
//   warps 4-7   softmax: thread t owns row t (TMEM lane t).  Loads S, masks
//               the row's window, takes the tile max, writes P = 2^(S - m)
//               (rounded to TF32) back over S, keeps the row sum, rescales O
//               when the reference max moves, and finally writes O / l and
//               (max, log sum).
// Tensor memory (512 columns): Q [0, D), S0 [128, 256), S1 [256, 384),
// O [384, 384 + D).  Scores are in base-2 units: Q is pre-multiplied by
// scale * log2(e).  The reference max only moves when a row's tile max
// exceeds it by more than 8 (so P <= 256), which leaves the result exact and
// skips most O rescales; the true max is tracked separately for the LSE.
#include <cfloat>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace attn {
namespace {

constexpr int kRows = 128;       // packed rows per CTA (MMA M)
constexpr int kKeys = 128;       // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kThreads = 256;
constexpr int kRingBytes = 3 * 65536;  // K/V tile ring in shared memory
constexpr int kMaxRing = 6;
constexpr int kColQ = 0, kColS0 = 128, kColO = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct __align__(1024) TcSmem {
  unsigned char ring[kRingBytes];
  uint64_t kv_full[kMaxRing];
  uint64_t kv_empty[kMaxRing];
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t pv_done[2];
  uint64_t q_ready;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint32_t tf32_round(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    flash_tc_kernel(const FlashArgs a, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v) {
  constexpr int kChunks = D / 32;              // 32-float column chunks of a row
  constexpr int kChunkBytes = kKeys * 128;     // one TMA box: 128 keys x 128 bytes
  constexpr int kTileBytes = kChunks * kChunkBytes;
  constexpr int kRing = kRingBytes / kTileBytes;          // tiles in flight: 3 (D=128) or 6 (D=64)
  static_assert(kRing <= kMaxRing, "ring barriers");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y;
  const int blk = gridDim.x - 1 - blockIdx.x;  // heaviest causal blocks first
  const int gs = a.H / a.G;
  const int qpb = kRows / gs;                  // queries per block
  const long long i0 = (long long)blk * qpb;   // first query of the block
  const long long i1 = min((long long)a.n_q, i0 + qpb) - 1;  // last valid query
  auto window = [&](long long i) -> int {
    if (i < 0 || i >= a.n_q) return 0;
    if (!a.causal) return a.n_all;
    const long long w = a.base_pos + i + 1;
    return (int)(w < a.cap ? w : a.cap);
  };
  const int n_max = window(i1);
  const int n_min = window(i0);
  const int nt = (n_max + kKeys - 1) / kKeys;

  if (tid == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.p_ready[b], 4);
      mbar_init(&sm.pv_done[b], 1);
    }
    mbar_init(&sm.q_ready, 4);
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
    if (lane == 0 && nt > 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      // Tile idx: K_(idx/2) for even idx, V_(idx/2) for odd; ring slot idx % kRing.
      for (int idx = 0; idx < 2 * nt; ++idx) {
        const int s = idx % kRing, use = idx / kRing;
        unsigned char* dst = sm.ring + s * kTileBytes;
        if (use >= 1) mbar_wait_bounded(&sm.kv_empty[s], (unsigned)((use - 1) & 1), a.status, &sm.abort);
        mbar_arrive_expect_tx(&sm.kv_full[s], (unsigned)kTileBytes);
        const CUtensorMap* tm = (idx & 1) ? &tm_v : &tm_k;
        const int y = kKeys * (idx >> 1);
#pragma unroll
        for (int c = 0; c < kChunks; ++c) tma_load_2d(dst + c * kChunkBytes, tm, g * D + 32 * c, y, &sm.kv_full[s]);
      }
      // No copy may still be landing in shared memory when the CTA exits
      // (normally every fill was already consumed, so these return at once).
      for (int s = 0; s < kRing && s < 2 * nt; ++s) {
        const int last = s + ((2 * nt - 1 - s) / kRing) * kRing;
        mbar_wait_bounded(&sm.kv_full[s], (unsigned)((last / kRing) & 1), a.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idesc_qk = tc::idesc_f32acc(tc::kFmtTF32, false, kRows, kKeys);
      constexpr uint32_t idesc_pv = tc::idesc_f32acc(tc::kFmtTF32, true, kRows, D);
      const uint32_t ring0 = smem_u32(sm.ring);
      mbar_wait_bounded(&sm.q_ready, 0, a.status, &sm.abort);
      tc::fence_after_sync();
      auto tile_addr = [&](int idx) { return ring0 + (uint32_t)((idx % kRing) * kTileBytes); };
      auto full_wait = [&](int idx) {
        mbar_wait_bounded(&sm.kv_full[idx % kRing], (unsigned)((idx / kRing) & 1), a.status, &sm.abort);
      };
      auto release = [&](int idx) { tc::commit(&sm.kv_empty[idx % kRing]); };
      for (int j = 0; j <= nt; ++j) {
        if (j < nt) {
          const int b = j & 1;
          if (j >= 2) mbar_wait_bounded(&sm.pv_done[b], (unsigned)(((j - 2) >> 1) & 1), a.status, &sm.abort);
          full_wait(2 * j);
          tc::fence_after_sync();
          const uint32_t kb = tile_addr(2 * j);
#pragma unroll
          for (int kk = 0; kk < D / 8; ++kk) {
            const uint64_t bdesc = tc::sdesc_sw128(kb + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024);
            tc::mma_tf32_ts(tmem + kColS0 + 128 * b, tmem + kColQ + 8 * kk, bdesc, idesc_qk, kk > 0);
          }
          tc::commit(&sm.s_full[b]);
          release(2 * j);
        }
        if (j >= 1) {
          const int jj = j - 1, b = jj & 1;
          mbar_wait_bounded(&sm.p_ready[b], (unsigned)((jj >> 1) & 1), a.status, &sm.abort);
          full_wait(2 * jj + 1);
          tc::fence_after_sync();
          const uint32_t vb = tile_addr(2 * jj + 1);
#pragma unroll
          for (int kk = 0; kk < kKeys / 8; ++kk) {
            const uint64_t bdesc = tc::sdesc_sw128(vb + kk * 1024, kChunkBytes, 512, tc::kLayoutSw128Atom32);
            tc::mma_tf32_ts(tmem + kColO, tmem + kColS0 + 128 * b + 8 * kk, bdesc, idesc_pv, (jj > 0 || kk > 0));
          }
          tc::commit(&sm.pv_done[b]);
          release(2 * jj + 1);
        }
      }
      // Every MMA has finished before tensor memory is released.
      tc::commit(&sm.drain);
      mbar_wait_bounded(&sm.drain, 0, a.status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / epilogue
    const int r = tid - 128;                       // row == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp - 4)) << 16;
    const long long packed = (long long)blk * kRows + r;
    const long long qi = packed / gs;
    const int h = g * gs + (int)(packed % gs);
    const int n_r = window(qi);
    const bool row_ok = qi < a.n_q;
    const float sl2 = a.scale * kLog2e;

    // Q row -> TMEM (pre-scaled); rows past n_q are zero.
    {
      const float* qrow = a.q + qi * a.q_row_stride + (long long)h * D;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float4 x = row_ok ? *reinterpret_cast<const float4*>(qrow + 32 * c + e) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[e] = __float_as_uint(x.x * sl2);
          v[e + 1] = __float_as_uint(x.y * sl2);
          v[e + 2] = __float_as_uint(x.z * sl2);
          v[e + 3] = __float_as_uint(x.w * sl2);
        }
        tc::tmem_st32(tmem + lane_base + kColQ + 32 * c, v);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.q_ready);
    }

    float m_ref = -INFINITY, m_true = -INFINITY, l = 0.f;
    for (int j = 0; j < nt; ++j) {
      const int b = j & 1;
      const uint32_t s_col = tmem + lane_base + kColS0 + 128 * b;
      mbar_wait_bounded(&sm.s_full[b], (unsigned)((j >> 1) & 1), a.status, &sm.abort);
      tc::fence_after_sync();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(s_col + 32 * c, s[c]);
      tc::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::reg_fence(s[c]);

      const bool masked = (j + 1) * kKeys > n_min;
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float x = __uint_as_float(s[c][e]);
          if (masked && (j * kKeys + 32 * c + e) >= n_r) x = -INFINITY;
          s[c][e] = __float_as_uint(x);
          tmax = fmaxf(tmax, x);
        }
      m_true = fmaxf(m_true, tmax);
      float corr = 1.f;
      if (tmax > m_ref + kRescaleThreshold) {  // also true for the first finite tile max
        corr = ex2(m_ref - tmax);              // m_ref = -inf gives 0
        m_ref = tmax;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const uint32_t p = tf32_round(ex2(__uint_as_float(s[c][e]) - m_use));
          sum += __uint_as_float(p);
          s[c][e] = p;
        }
        tc::tmem_st32(s_col + 32 * c, s[c]);
      }
      l = l * corr + sum;
      tc::tmem_st_wait();

      // O was accumulated against the old reference: rescale it (after the
      // previous P V has landed) when any row of this warp moved its reference.
      if (j > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
        const int pb = (j - 1) & 1;
        mbar_wait_bounded(&sm.pv_done[pb], (unsigned)(((j - 1) >> 1) & 1), a.status, &sm.abort);
        tc::fence_after_sync();
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(tmem + lane_base + kColO + 32 * c, o);
          tc::tmem_ld_wait();
          tc::reg_fence(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
          tc::tmem_st32(tmem + lane_base + kColO + 32 * c, o);
        }
        tc::tmem_st_wait();
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_ready[b]);
    }

    // Epilogue: out = O / l, lse = (max, log sum).
    if (nt > 0) {
      const int lb = (nt - 1) & 1;
      mbar_wait_bounded(&sm.pv_done[lb], (unsigned)(((nt - 1) >> 1) & 1), a.status, &sm.abort);
      tc::fence_after_sync();
    }
    const float inv = (l == 0.f) ? 0.f : 1.f / l;
    float* orow = a.out + qi * a.out_row_stride + (long long)h * D;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      uint32_t o[32];
      if (nt > 0) {
        tc::tmem_ld32(tmem + lane_base + kColO + 32 * c, o);
        tc::tmem_ld_wait();
        tc::reg_fence(o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (row_ok) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(orow + 32 * c + e) =
              make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                          __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
      }
    }
    if (row_ok && a.lse != nullptr) {
      float* l2 = a.lse + (qi * a.H + h) * 2;
      const bool empty = (l == 0.f);
      l2[0] = empty ? kEmptyLse : m_true * kLn2;
      l2[1] = empty ? kEmptyLse : logf(l) + (m_ref - m_true) * kLn2;
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

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

template <int D>
int launch_d(const FlashArgs& a, cudaStream_t s) {
  const int gs = a.H / a.G;
  const long long rows = (long long)a.n_q * gs;
  const long long nb = (rows + kRows - 1) / kRows;
  if (nb == 0) return 0;
  // Rows of K/V any CTA may read: the largest window of the call.  Rows past
  // it are outside the tensor map and arrive as zeros.
  long long kv_rows = a.causal ? a.base_pos + a.n_q : a.n_all;
  if (kv_rows > a.cap) kv_rows = a.cap;
  if (kv_rows < 1) kv_rows = 1;
  CUtensorMap tm_k, tm_v;
  const uint64_t dims[2] = {(uint64_t)a.kv_row_stride, (uint64_t)kv_rows};
  const uint64_t strides[1] = {(uint64_t)a.kv_row_stride * 4};
  const uint32_t box[2] = {32, (uint32_t)kKeys};
  const float* kp = a.k != nullptr ? a.k : a.q;  // an empty key set never reads K/V
  const float* vp = a.v != nullptr ? a.v : a.q;
  if (!make_tmap(&tm_k, kp, 2, dims, strides, box, false, kSwizzle128) ||
      !make_tmap(&tm_v, vp, 2, dims, strides, box, false, kSwizzle128Atom32))
    return ATTN_ERR_UNSUPPORTED;
  const size_t smem = sizeof(TcSmem) + 1024;
  auto kern = flash_tc_kernel<D>;
  if (!set_smem_limit(reinterpret_cast<const void*>(kern), smem)) return ATTN_ERR_CUDA;
  kern<<<dim3((unsigned)nb, (unsigned)a.G), kThreads, smem, s>>>(a, tm_k, tm_v);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : ATTN_ERR_CUDA;
}

}  // namespace

bool flash_tc_supported(const FlashArgs& a, int prec) {
  if (prec != ATTN_TF32) return false;
  if (a.kv_pos_dev != nullptr) return false;
  if (a.D != 64 && a.D != 128) return false;
  const int gs = a.H / a.G;
  if (!is_pow2(gs) || gs > kRows) return false;
  const uintptr_t al = reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.out) |
                       reinterpret_cast<uintptr_t>(a.k) | reinterpret_cast<uintptr_t>(a.v);
  if (al % 16 != 0) return false;
  if (a.q_row_stride % 4 != 0 || a.out_row_stride % 4 != 0 || a.kv_row_stride % 4 != 0) return false;
  return true;
}

int launch_flash_tc(const FlashArgs& a, int prec, cudaStream_t s) {
  if (!flash_tc_supported(a, prec)) return ATTN_ERR_UNSUPPORTED;
  return a.D == 128 ? launch_d<128>(a, s) : launch_d<64>(a, s);
}

}  // namespace attn
