// flash_tc.cu -- tcgen05 tensor-core flash attention (forward and prefill).
//
// Operation: softmax(scale * Q K^T) V over per-row causal / full / cross /
// prefill windows, with the running max / sum of the pages' online softmax
// (cera attention_prefill.wgsl, fn attention_prefill: per-tile max,
// correction, exponentials, running sum; meganeura attention.wgsl, fn main:
// the final (max, log sum) store).  Both contractions run on the 5th-generation
// tensor cores with fp32 accumulation in tensor memory, with TF32 operands
// (K/V tiles straight from the fp32 inputs) or bf16 operands (K/V converted
// once per call by a small pre-pass; Q and P rounded on their way into TMEM).
//
// One CTA owns 128 packed rows of one kv head g: row r is (query i, head
// g*gs + j) with i*gs + j = 128*block + r, so each K/V tile feeds all gs
// query heads that share it.  Keys are walked in tiles of 128.
//
// Warp roles (384 threads):
//   warp 0      TMA producer: K tile (128 keys x D, 128-byte swizzle, K-major
//               operand) and V tile (MN-major operand; TF32 needs the
//               32-byte-atom swizzle, bf16 the plain 128-byte one) into a
//               192 KB shared-memory ring: 3 tiles deep for TF32, 6 for bf16.
//   warp 1      tensor-memory allocation; one thread issues every MMA:
//                 S_b = Q K_j^T      (A = Q in TMEM, B = K tile)      M=128 N=128
//                 O  += P_j V_j      (A = P in TMEM over S_b, B = V)  M=128 N=D
//               The issuer is greedy: it issues whichever of the next Q K^T
//               and the next P V has its inputs ready.
//   warps 4-11  softmax, two warpgroups: warp w of group c handles rows
//               32(w%4)..+31 (TMEM lanes) and score columns 64c..64c+63.  The
//               two halves of a row swap their tile max through shared
//               memory; each group writes its half of P = 2^(S - m) back into
//               the score buffer, keeps its half of the row sum, rescales its
//               half of O when the reference max moves, and finally writes its
//               half of O / l; group 0 writes (max, log sum).
// Tensor memory (512 columns): Q [0, 128), two 128-column score buffers
// [128, 384), O [384, 384 + D).  Scores are in base-2 units: Q is
// pre-multiplied by scale * log2(e).  The reference max only moves when a
// row's tile max exceeds it by more than 8 (so P <= 256), which leaves the
// result exact and skips most O rescales; the true max is tracked separately
// for the LSE.  Every wait is bounded; a CTA whose pipeline breaks drains its
// copies and MMAs before it releases tensor memory.
#include <cfloat>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace attn {
namespace {

constexpr int kRows = 128;        // packed rows per CTA (MMA M)
constexpr int kKeys = 128;        // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kSBuf = 2;          // score buffers in tensor memory
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;
constexpr int kRingBytes = 3 * 65536;  // K/V tile ring in shared memory
constexpr int kMaxRing = 12;
constexpr int kColQ = 0, kColS0 = 128, kColO = 384;  // S buffer b at kColS0 + kKeys * b
constexpr float kRescaleThreshold = 8.0f;             // log2 units

struct __align__(1024) TcSmem {
  unsigned char ring[kRingBytes];
  uint64_t kv_full[kMaxRing];
  uint64_t kv_empty[kMaxRing];
  uint64_t s_full[kSBuf];
  uint64_t p_ready[kSBuf];
  uint64_t pv_done[kSBuf];
  uint64_t q_ready;
  uint64_t drain;
  float red_max[2][2][kRows];  // [tile parity][group][row] partial tile maxima
  float red_l[2][kRows];       // [group][row] partial row sums (epilogue)
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint32_t tf32_round(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// Two floats as round-to-nearest bf16 in one word: lo in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// BF = false: TF32 operands (fp32 K/V tiles straight from the inputs).
// BF = true: bf16 operands (K/V already converted to bf16; Q and P rounded to
// bf16 on their way into tensor memory, two values per 32-bit column).
template <int D, bool BF>
__global__ void __launch_bounds__(kThreads, 1)
    flash_tc_kernel(const FlashArgs a, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v) {
  constexpr int kEpr = BF ? 64 : 32;           // elements per 128-byte row
  constexpr int kChunks = D / kEpr;            // 128-byte column chunks of a K/V row
  constexpr int kChunkBytes = kKeys * 128;     // one TMA box: 128 keys x 128 bytes
  constexpr int kTileBytes = kChunks * kChunkBytes;
  constexpr int kRing = kRingBytes / kTileBytes;  // tiles in flight
  static_assert(kRing <= kMaxRing, "ring barriers");
  constexpr int kKStep = BF ? 16 : 8;          // MMA K per instruction (32 bytes)
  // V operand form.  The bf16 path reads V^T (keys contiguous), written by the
  // pre-pass, as a K-major operand: an MN-major V measured about twice as slow
  // in P V as the same-size K-major Q K^T.
  constexpr bool kVT = BF;
  constexpr int kVtChunkBytes = D * 128;       // one V^T box: D rows x 128 bytes of keys
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u));

  // Programmatic dependent launch: the next kernel may start launching; this
  // one touches no global memory before the previous kernel has completed.
  allow_dependent_launch();
  grid_dependency_wait();
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
    for (int b = 0; b < kSBuf; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.p_ready[b], 8);
      mbar_init(&sm.pv_done[b], 1);
    }
    mbar_init(&sm.q_ready, 8);
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
        const int t0 = kKeys * (idx >> 1);
        if ((idx & 1) && kVT) {
          // V^T tile: kKeys / kEpr boxes of [D rows (d) x 128 bytes of keys].
#pragma unroll
          for (int c = 0; c < kKeys / kEpr; ++c)
            tma_load_2d(dst + c * kVtChunkBytes, &tm_v, t0 + kEpr * c, g * D, &sm.kv_full[s]);
        } else {
          const CUtensorMap* tm = (idx & 1) ? &tm_v : &tm_k;
#pragma unroll
          for (int c = 0; c < kChunks; ++c) tma_load_2d(dst + c * kChunkBytes, tm, g * D + kEpr * c, t0, &sm.kv_full[s]);
        }
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
      constexpr uint32_t kFmt = BF ? tc::kFmtBF16 : tc::kFmtTF32;
      constexpr uint32_t idesc_qk = tc::idesc_f32acc(kFmt, false, kRows, kKeys);
      constexpr uint32_t idesc_pv = tc::idesc_f32acc(kFmt, !kVT, kRows, D);
      // V (MN-major B): TF32 needs the 32-byte-atom layout with 4-row K groups;
      // bf16 uses the plain 128-byte swizzle with 8-row groups.
      constexpr uint32_t kVLayout = BF ? tc::kLayoutSw128 : tc::kLayoutSw128Atom32;
      constexpr uint32_t kVSbo = BF ? 1024 : 512;
      constexpr uint32_t kVStep = kKStep * 128;  // bytes of V rows per K step
      const uint32_t ring0 = smem_u32(sm.ring);
      mbar_wait_bounded(&sm.q_ready, 0, a.status, &sm.abort);
      tc::fence_after_sync();
      auto tile_addr = [&](int idx) { return ring0 + (uint32_t)((idx % kRing) * kTileBytes); };
      auto full_ready = [&](int idx) {
        return mbar_test_wait(&sm.kv_full[idx % kRing], (unsigned)((idx / kRing) & 1));
      };
      auto release = [&](int idx) { tc::commit(&sm.kv_empty[idx % kRing]); };
      int nq = 0, np = 0;  // next Q K^T and next P V to issue
      unsigned long long t_idle = 0;
      while (np < nt) {
        // Q K^T for tile nq writes S buffer nq % kSBuf, last read by P V of tile nq - kSBuf.
        const bool qk_ok =
            nq < nt && nq < np + kSBuf &&
            (nq < kSBuf || mbar_test_wait(&sm.pv_done[nq % kSBuf], (unsigned)(((nq - kSBuf) / kSBuf) & 1))) &&
            full_ready(2 * nq);
        const bool pv_ok = !qk_ok && nq > np &&
                           mbar_test_wait(&sm.p_ready[np % kSBuf], (unsigned)((np / kSBuf) & 1)) &&
                           full_ready(2 * np + 1);
        if (qk_ok) {
          const int b = nq % kSBuf;
          tc::fence_after_sync();
          const uint32_t kb = tile_addr(2 * nq);
#pragma unroll
          for (int kk = 0; kk < D / kKStep; ++kk) {
            const uint64_t bdesc = tc::sdesc_sw128(kb + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024);
            if constexpr (BF)
              tc::mma_f16_ts(tmem + kColS0 + kKeys * b, tmem + kColQ + 8 * kk, bdesc, idesc_qk, kk > 0);
            else
              tc::mma_tf32_ts(tmem + kColS0 + kKeys * b, tmem + kColQ + 8 * kk, bdesc, idesc_qk, kk > 0);
          }
          tc::commit(&sm.s_full[b]);
          release(2 * nq);
          ++nq;
          t_idle = 0;
        } else if (pv_ok) {
          const int b = np % kSBuf;
          tc::fence_after_sync();
          const uint32_t vb = tile_addr(2 * np + 1);
#pragma unroll
          for (int kk = 0; kk < kKeys / kKStep; ++kk) {
            const uint64_t bdesc =
                kVT ? tc::sdesc_sw128(vb + (kk >> 2) * kVtChunkBytes + (kk & 3) * 32, 16, 1024)
                    : tc::sdesc_sw128(vb + kk * kVStep, kChunkBytes, kVSbo, kVLayout);
            if constexpr (BF)
              tc::mma_f16_ts(tmem + kColO, tmem + kColS0 + kKeys * b + 8 * kk, bdesc, idesc_pv, (np > 0 || kk > 0));
            else
              tc::mma_tf32_ts(tmem + kColO, tmem + kColS0 + kKeys * b + 8 * kk, bdesc, idesc_pv, (np > 0 || kk > 0));
          }
          tc::commit(&sm.pv_done[b]);
          release(2 * np + 1);
          ++np;
          t_idle = 0;
        } else {
          const unsigned long long now = globaltimer_ns();
          if (t_idle == 0) t_idle = now;
          if (*reinterpret_cast<volatile int*>(&sm.abort) != 0) break;
          if (now - t_idle > kWaitLimitNs) {
            record_status(a.status, ATTN_ERR_TIMEOUT);
            *reinterpret_cast<volatile int*>(&sm.abort) = 1;
            break;
          }
        }
      }
      // Every MMA has finished before tensor memory is released.
      tc::commit(&sm.drain);
      mbar_wait_bounded(&sm.drain, 0, a.status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / epilogue
    constexpr int kHalfD = D / 2;              // O columns per group
    const int grp = (warp - 4) >> 2;           // column group 0 or 1
    const int r = 32 * (warp & 3) + lane;      // row == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const long long packed = (long long)blk * kRows + r;
    const long long qi = packed / gs;
    const int h = g * gs + (int)(packed % gs);
    const int n_r = window(qi);
    const bool row_ok = qi < a.n_q;
    const float sl2 = a.scale * kLog2e;

    // Q row -> TMEM (pre-scaled); rows past n_q are zero.  TF32: one value per
    // column; bf16: two per column (lower index in the low half).  Each group
    // stores half the row, unless half is under one 32-column store (bf16,
    // D = 64): then group 0 stores the whole row.
    {
      constexpr int kPer = BF ? 2 : 1;
      constexpr int kQAll = D / kPer;          // TMEM columns of a Q row
      constexpr bool kSplitQ = kQAll >= 64;
      constexpr int kQCols = kSplitQ ? kQAll / 2 : kQAll;
      const int q_grp = kSplitQ ? grp : 0;
      const int n_chunks = (kSplitQ || grp == 0) ? kQCols / 32 : 0;
      const float* qrow = a.q + qi * a.q_row_stride + (long long)h * D + q_grp * kQCols * kPer;
      for (int c = 0; c < n_chunks; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int e = 0; e < 32; e += 4 / kPer) {
          const float* src = qrow + kPer * (32 * c + e);
          const float4 x = row_ok ? *reinterpret_cast<const float4*>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
          if constexpr (BF) {
            v[e] = pack_bf16(x.x * sl2, x.y * sl2);
            v[e + 1] = pack_bf16(x.z * sl2, x.w * sl2);
          } else {
            v[e] = __float_as_uint(x.x * sl2);
            v[e + 1] = __float_as_uint(x.y * sl2);
            v[e + 2] = __float_as_uint(x.z * sl2);
            v[e + 3] = __float_as_uint(x.w * sl2);
          }
        }
        tc::tmem_st32(tmem + lane_base + kColQ + q_grp * kQCols + 32 * c, v);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.q_ready);
    }

    constexpr int kCols = kKeys / 2;           // score columns per group per tile
    constexpr int kCC = kCols / 32;            // 32-column TMEM loads per group per tile
    float m_ref = -INFINITY, m_true = -INFINITY, l = 0.f;
    for (int j = 0; j < nt; ++j) {
      const int b = j % kSBuf;
      const uint32_t s_col = tmem + lane_base + kColS0 + kKeys * b + kCols * grp;
      mbar_wait_bounded(&sm.s_full[b], (unsigned)((j / kSBuf) & 1), a.status, &sm.abort);
      tc::fence_after_sync();
      uint32_t s[kCC][32];
#pragma unroll
      for (int c = 0; c < kCC; ++c) tc::tmem_ld32(s_col + 32 * c, s[c]);
      tc::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < kCC; ++c) tc::reg_fence(s[c]);

      // Mask and this half's max (four independent chains).
      const bool masked = (j + 1) * kKeys > n_min;
      const int col0 = j * kKeys + kCols * grp;
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < kCC; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float x = __uint_as_float(s[c][e]);
          if (masked && (col0 + 32 * c + e) >= n_r) x = -INFINITY;
          s[c][e] = __float_as_uint(x);
          mx[e & 3] = fmaxf(mx[e & 3], x);
        }
      sm.red_max[j & 1][grp][r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      named_barrier(1, kSoftmaxThreads);
      const float tmax = fmaxf(sm.red_max[j & 1][0][r], sm.red_max[j & 1][1][r]);
      m_true = fmaxf(m_true, tmax);
      float corr = 1.f;
      if (tmax > m_ref + kRescaleThreshold) {  // also true for the first finite tile max
        corr = ex2(m_ref - tmax);              // m_ref = -inf gives 0
        m_ref = tmax;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      float sm4[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (BF) {
        // P as bf16 pairs into the first half of this buffer's columns: this
        // group's 64 values become 32 columns at offset 32 * grp.  Both groups
        // finished reading S before the max exchange above.
        uint32_t pk[32];
        static_assert(kCC * 16 == 32, "one 32-column P store per group");
#pragma unroll
        for (int c = 0; c < kCC; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 = ex2(__uint_as_float(s[c][e]) - m_use);
            const float p1 = ex2(__uint_as_float(s[c][e + 1]) - m_use);
            const uint32_t w = pack_bf16(p0, p1);
            sm4[e & 3] += __uint_as_float(w << 16);
            sm4[(e + 1) & 3] += __uint_as_float(w & 0xffff0000u);
            pk[16 * c + e / 2] = w;
          }
        tc::tmem_st32(tmem + lane_base + kColS0 + kKeys * b + 32 * grp, pk);
      } else {
#pragma unroll
        for (int c = 0; c < kCC; ++c) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const uint32_t p = tf32_round(ex2(__uint_as_float(s[c][e]) - m_use));
            sm4[e & 3] += __uint_as_float(p);
            s[c][e] = p;
          }
          tc::tmem_st32(s_col + 32 * c, s[c]);
        }
      }
      l = l * corr + ((sm4[0] + sm4[1]) + (sm4[2] + sm4[3]));
      tc::tmem_st_wait();

      // O was accumulated against the old reference: rescale this group's half
      // (after the previous P V has landed) when any row of the warp moved.
      if (j > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
        const int pb = (j - 1) % kSBuf;
        mbar_wait_bounded(&sm.pv_done[pb], (unsigned)(((j - 1) / kSBuf) & 1), a.status, &sm.abort);
        tc::fence_after_sync();
#pragma unroll
        for (int c = 0; c < kHalfD / 32; ++c) {
          uint32_t o[32];
          const uint32_t oc = tmem + lane_base + kColO + grp * kHalfD + 32 * c;
          tc::tmem_ld32(oc, o);
          tc::tmem_ld_wait();
          tc::reg_fence(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
          tc::tmem_st32(oc, o);
        }
        tc::tmem_st_wait();
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_ready[b]);
    }

    // Epilogue: out = O / l, lse = (max, log sum).
    sm.red_l[grp][r] = l;
    if (nt > 0) {
      const int lb = (nt - 1) % kSBuf;
      mbar_wait_bounded(&sm.pv_done[lb], (unsigned)(((nt - 1) / kSBuf) & 1), a.status, &sm.abort);
      tc::fence_after_sync();
    }
    named_barrier(1, kSoftmaxThreads);
    const float l_row = sm.red_l[0][r] + sm.red_l[1][r];
    const float inv = (l_row == 0.f) ? 0.f : 1.f / l_row;
    float* orow = a.out + qi * a.out_row_stride + (long long)h * D + grp * kHalfD;
#pragma unroll
    for (int c = 0; c < kHalfD / 32; ++c) {
      uint32_t o[32];
      if (nt > 0) {
        tc::tmem_ld32(tmem + lane_base + kColO + grp * kHalfD + 32 * c, o);
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
    if (grp == 0 && row_ok && a.lse != nullptr) {
      float* l2 = a.lse + (qi * a.H + h) * 2;
      const bool empty = (l_row == 0.f);
      l2[0] = empty ? kEmptyLse : m_true * kLn2;
      l2[1] = empty ? kEmptyLse : logf(l_row) + (m_ref - m_true) * kLn2;
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

// fp32 -> bf16, n4 groups of four values (the source is 16-byte aligned).
__global__ void __launch_bounds__(256) to_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst,
                                                      long long n4) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    const float4 x = src[i];
    dst[i] = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
  }
}

// V [rows][row_stride] fp32 -> V^T [cols][pad] bf16 (cols = G*D), zero for
// rows >= rows.  32 x 32 tiles through shared memory; block (32, 8).
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const float* __restrict__ v, uint16_t* __restrict__ vt,
                                                             long long rows, long long pad, long long row_stride,
                                                             int cols) {
  __shared__ float tile[32][33];
  const long long t0 = (long long)blockIdx.x * 32;
  const int c0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const long long t = t0 + i;
    const int c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (t < rows && c < cols) ? v[t * row_stride + c] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i;
    const long long t = t0 + threadIdx.x;
    if (c < cols && t < pad) {
      const uint32_t w = pack_bf16(tile[threadIdx.x][i], 0.f);
      vt[(long long)c * pad + t] = (uint16_t)(w & 0xffffu);
    }
  }
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

template <int D, bool BF>
int launch_d(const FlashArgs& a, cudaStream_t s) {
  const int gs = a.H / a.G;
  const long long rows = (long long)a.n_q * gs;
  const long long nb = (rows + kRows - 1) / kRows;
  if (nb == 0) return 0;
  // Rows of K/V any CTA may read: the largest window of the call.  Rows past
  // it are outside the tensor map and arrive as zeros.
  long long kv_rows = a.causal ? a.base_pos + a.n_q : a.n_all;
  if (kv_rows > a.cap) kv_rows = a.cap;
  const bool no_keys = kv_rows < 1 || a.k == nullptr || a.v == nullptr;
  if (kv_rows < 1) kv_rows = 1;
  CUtensorMap tm_k, tm_v;
  const uint64_t dims[2] = {(uint64_t)a.kv_row_stride, (uint64_t)kv_rows};
  const uint32_t box[2] = {(uint32_t)(BF ? 64 : 32), (uint32_t)kKeys};
  void* scratch = nullptr;
  long long kv_pad = 64;
  const void* kp = a.q;  // an empty key set never reads K/V: any aligned base will do
  const void* vp = a.q;
  if (!no_keys) {
    if constexpr (BF) {
      // K and V as bf16 in stream-ordered temporary memory, released on the
      // same stream once the attention kernel has run.
      // K keeps its layout; V is written transposed, V^T [G*D][kv_pad] with
      // keys contiguous and the pad columns zero.
      const long long elems = kv_rows * a.kv_row_stride;
      kv_pad = (kv_rows + 63) / 64 * 64;
      const long long vt_elems = (long long)a.G * D * kv_pad;
      if (cudaMallocAsync(&scratch, (size_t)(elems + vt_elems) * 2, s) != cudaSuccess) return ATTN_ERR_CUDA;
      uint16_t* k16 = static_cast<uint16_t*>(scratch);
      uint16_t* vt16 = k16 + elems;
      to_bf16_kernel<<<4 * 152, 256, 0, s>>>(reinterpret_cast<const float4*>(a.k), reinterpret_cast<uint2*>(k16),
                                             elems / 4);
      const dim3 tgrid((unsigned)(kv_pad / 32), (unsigned)((a.G * D + 31) / 32));
      transpose_bf16_kernel<<<tgrid, dim3(32, 8), 0, s>>>(a.v, vt16, kv_rows, kv_pad, a.kv_row_stride, a.G * D);
      kp = k16;
      vp = vt16;
    } else {
      kp = a.k;
      vp = a.v;
    }
  }
  const uint64_t strides[1] = {(uint64_t)a.kv_row_stride * (BF ? 2 : 4)};
  bool maps_ok = make_tmap(&tm_k, kp, 2, dims, strides, box, BF, kSwizzle128);
  if (BF) {
    // V^T: [G*D rows][kv_pad keys], boxes of 64 keys x D rows.
    const uint64_t vdims[2] = {(uint64_t)kv_pad, (uint64_t)a.G * D};
    const uint64_t vstrides[1] = {(uint64_t)kv_pad * 2};
    const uint32_t vbox[2] = {64, (uint32_t)D};
    maps_ok = maps_ok && make_tmap(&tm_v, vp, 2, vdims, vstrides, vbox, true, kSwizzle128);
  } else {
    maps_ok = maps_ok && make_tmap(&tm_v, vp, 2, dims, strides, box, false, kSwizzle128Atom32);
  }
  int rc = ATTN_OK;
  if (!maps_ok) {
    rc = ATTN_ERR_UNSUPPORTED;
  } else {
    const size_t smem = sizeof(TcSmem) + 1024;
    auto kern = flash_tc_kernel<D, BF>;
    if (!set_smem_limit(reinterpret_cast<const void*>(kern), smem)) {
      rc = ATTN_ERR_CUDA;
    } else {
      FlashArgs aa = a;
      void* args[] = {&aa, &tm_k, &tm_v};
      if (launch_pdl(reinterpret_cast<const void*>(kern), dim3((unsigned)nb, (unsigned)a.G), dim3(kThreads), smem, s,
                     args) != cudaSuccess)
        rc = ATTN_ERR_CUDA;
    }
  }
  if (scratch != nullptr && cudaFreeAsync(scratch, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
  return rc;
}

}  // namespace

bool flash_tc_supported(const FlashArgs& a, int prec) {
  if (prec != ATTN_TF32 && prec != ATTN_BF16) return false;
  if (a.kv_pos_dev != nullptr) return false;
  if (a.D != 64 && a.D != 128) return false;
  if (a.G > 65535) return false;
  const int gs = a.H / a.G;
  if (!is_pow2(gs) || gs > kRows) return false;
  const uintptr_t al = reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.out) |
                       reinterpret_cast<uintptr_t>(a.k) | reinterpret_cast<uintptr_t>(a.v);
  if (al % 16 != 0) return false;
  if (a.q_row_stride % 4 != 0 || a.out_row_stride % 4 != 0 || a.kv_row_stride % 4 != 0) return false;
  if (prec == ATTN_BF16 && a.kv_row_stride % 8 != 0) return false;  // bf16 rows in 16-byte units
  return true;
}

int launch_flash_tc(const FlashArgs& a, int prec, cudaStream_t s) {
  if (!flash_tc_supported(a, prec)) return ATTN_ERR_UNSUPPORTED;
  if (prec == ATTN_BF16) return a.D == 128 ? launch_d<128, true>(a, s) : launch_d<64, true>(a, s);
  return a.D == 128 ? launch_d<128, false>(a, s) : launch_d<64, false>(a, s);
}

}  // namespace attn
