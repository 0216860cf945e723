// flash_tc.cu -- tcgen05 tensor-core flash attention with TF32-class
// accuracy (forward and prefill).
//
// Operation: softmax(scale * Q K^T) V over per-row causal / full / cross /
// prefill windows (optionally cut to their last `window` keys), with the
// running max / sum of the pages' online softmax (cera attention_prefill.wgsl,
// fn attention_prefill: per-tile max, correction, exponentials, running sum;
// meganeura attention.wgsl, fn main: the final (max, log sum) store).  Both
// contractions run on the 5th-generation tensor cores with fp32 accumulation
// in tensor memory.  (The 16-bit-operand kernel is flash_bf16.cu.)
//
// Precision.  The scores enter the softmax through an exponential, so their
// operand rounding dominates the error: with scores of standard deviation 9
// (Q, K ~ N(0, 3^2), D = 128), TF32 Q and K (11 significant bits) move the
// output by up to about 3.5e-3 max|V|.  Q K^T is therefore computed with Q
// kept to 22 significant bits: each query row, scaled by a power of two that
// puts its largest magnitude in [2^14, 2^15), is split into fp16 hi + lo
// (hi = fp16(x), lo = fp16(x - hi)), and K is one fp16 operand under a power
// of two per 128-key tile of a kv head (the pre-pass); the two products
// Qhi K^T + Qlo K^T accumulate in fp32 -- the tensor time of one TF32 product
// -- and the two powers of two turn the raw score back in the softmax, as the
// multiplier of the fma that subtracts the running max.  K's own rounding
// (2^-11) leaves an error near 1.4e-3 max|V| on those inputs.  P V uses TF32
// operands: P (fp32 in tensor memory) and the V tiles straight from the fp32
// input.
//
// One CTA owns the packed rows of 128/gs queries of one kv head g (rpb =
// (128/gs)*gs of its 128 MMA rows; the rest idle when gs does not divide
// 128): row r is (query i, head g*gs + j) with i*gs + j = rpb*block + r, so
// each K/V tile feeds all gs query heads that share it.  Keys are walked in
// tiles of 128, from the tile holding the block's first kept key to the one
// holding its last.
//
// Warp roles (384 threads):
//   warp 0      TMA producer: K tile (128 keys x D fp16, 128-byte swizzle,
//               K-major operand, in the first half of a slot) and V tile (fp32, MN-major
//               operand, which for 32-bit elements needs the 128-byte swizzle
//               of 32-byte atoms) into a 192 KB shared-memory ring three tiles
//               deep, in the order the MMAs consume them.
//   warp 1      tensor-memory allocation; issues S_(j%2) = Q K_j^T
//               (A = Q hi / lo in TMEM, B = K tile, M=128 N=128) once
//               P V of tile j-2 has released that buffer.
//   warp 2      issues O += P_j V_j (A = P in TMEM over S_(j%2), B = V,
//               M=128 N=D) in tile order once both softmax groups wrote P_j.
//               The issuing warps run their loops warp-uniformly; one elected
//               lane issues.
//   warps 4-11  softmax, two warpgroups: warp w of group c handles rows
//               32(w%4)..+31 (TMEM lanes) and score columns 64c..64c+63.  The
//               two halves of a row swap their tile max through shared
//               memory; each group writes its half of P = 2^(S - m) back into
//               the score buffer, keeps its half of the row sum, rescales its
//               half of O when the reference max moves, and finally writes its
//               half of O / l; group 0 writes (max, log sum).
// Tensor memory (512 columns): Q hi [0, D/2) and Q lo [D/2, D) as packed
// fp16 pairs, two 128-column score buffers [128, 384), O [384, 384 + D).
// Scores are in base-2 units once scaled: Q is pre-multiplied by
// scale * log2(e) before it is split.  The reference max only moves when a row's tile max exceeds it
// by more than 8 (so P <= 256), which leaves the result exact and skips most
// O rescales; the true max is tracked separately for the LSE.  Every wait is
// bounded; a CTA whose pipeline breaks drains its copies and MMAs before it
// releases tensor memory.
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
constexpr int kColQ = 0, kColS0 = 128, kColO = 384;  // Q hi / lo in [0, 128); S buffer b at kColS0 + kKeys * b
constexpr float kRescaleThreshold = 8.0f;             // log2 units
constexpr int kPageBox = 32;     // fewest key rows per TMA box of a paged cache (page_rows % 32 == 0)
constexpr int kPageCache = 1024;  // block-table entries a CTA keeps in shared memory
constexpr int kFacCache = 512;    // K tile powers of two a CTA keeps in shared memory

// Key rows per TMA box of a paged cache with pages of page_rows rows.
__host__ __device__ inline int page_box(int page_rows) {
  return page_rows % kKeys == 0 ? kKeys : page_rows % 64 == 0 ? 64 : kPageBox;
}

struct __align__(1024) TcSmem {
  unsigned char ring[kRingBytes];
  uint64_t kv_full[kMaxRing];
  uint64_t kv_empty[kMaxRing];
  uint64_t s_full[kSBuf];
  uint64_t p_ready[kSBuf];
  uint64_t pv_done[kSBuf];
  uint64_t q_full;   // the fp32 Q block has landed in the staging slot
  uint64_t q_ready;  // Q is in tensor memory
  uint64_t drain[2];
  float red_max[2][2][kRows];  // [tile parity][group][row] partial tile maxima
  float red_l[2][kRows];       // [group][row] partial row sums (epilogue)
  uint32_t pages[kPageCache];  // block-table entries of the CTA's key range (paged caches)
  float kfac[kFacCache];       // powers of two of the CTA's K tiles jt0, jt0 + 1, ...
  uint32_t tmem_base;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    flash_tc_kernel(const FlashArgs a, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_o, const float* __restrict__ kfac, int early_q) {
  constexpr int kEpr = 32;                     // fp32 elements per 128-byte row
  constexpr int kChunks = D / kEpr;            // 128-byte column chunks of an fp32 V (or Q) row
  constexpr int kChunkBytes = kKeys * 128;     // one TMA box: 128 keys x 128 bytes
  constexpr int kTileBytes = kChunks * kChunkBytes;
  constexpr int kKChunks = D / 64;             // 128-byte column chunks of an fp16 K row
  constexpr int kKBytes = kKChunks * kChunkBytes;  // an fp16 K tile: the first half of a ring slot
  static_assert(2 * kKBytes == kTileBytes, "ring slots hold an fp32 V tile");
  constexpr int kColQl = D / 2;                // Q lo after the D/2 columns of Q hi pairs
  constexpr int kRing = kRingBytes / kTileBytes;  // tiles in flight
  static_assert(kRing <= kMaxRing, "ring barriers");
  constexpr int kKStep = 8;                    // MMA K per instruction (32 bytes)
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u));
  // The CTA's fp32 Q block lands by TMA in ring slot 2 (which holds no K/V
  // copy until Q is in tensor memory): D/32 chunks of 128 rows x 128 bytes,
  // 128-byte swizzle (16-byte unit u of row r at unit u ^ (r & 7)).
  static_assert(kTileBytes == kRows * D * 4, "Q staging fills one ring slot");
  unsigned char* const qstage = sm.ring + 2 * kTileBytes;

  // Programmatic dependent launch: the next kernel may start launching; this
  // one touches no global memory before the previous kernel has completed.
  allow_dependent_launch();
  // With the pre-pass launched just before (early_q), everything up to the
  // first K/V copy -- set-up and the Q block, which the pre-pass does not
  // write -- overlaps its tail: the pre-pass lets this grid start only once it
  // has itself waited for the kernels before it.  Each thread that reads what
  // the pre-pass wrote, or writes the outputs, waits for it first.
  if (!early_q) grid_dependency_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y;
  const int blk = gridDim.x - 1 - blockIdx.x;  // heaviest causal blocks first
  const int gs = a.H / a.G;
  const int qpb = kRows / gs;                  // queries per block
  const int rpb = qpb * gs;                    // packed rows used (rows rpb..127 idle when gs does not divide 128)
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
  const int lo_max = first_key(n_max, a.window);
  const int jt0 = first_key(n_min, a.window) / kKeys;  // first key tile of the block
  const int nt = (n_max + kKeys - 1) / kKeys - jt0;    // key tiles the block walks

  if (warp == 0) {
    // The Q block is copied first, so that it lands while the rest of the
    // set-up runs; the other barriers are initialised across the warp.
    if (lane == 0) {
      mbar_init(&sm.q_full, 1);
      fence_mbar_init();
      if (nt > 0) {
        prefetch_tmap(&tm_q);
        mbar_arrive_expect_tx(&sm.q_full, (unsigned)(rpb * D * 4));
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
          tma_load_3d(qstage + c * kChunkBytes, &tm_q, kEpr * c, g * gs, (int)i0, &sm.q_full);
      }
      sm.abort = 0;
    }
    for (int s = lane; s < kRing; s += 32) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int b = lane; b < kSBuf; b += 32) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.p_ready[b], 8);
      mbar_init(&sm.pv_done[b], 1);
    }
    if (lane < 2) mbar_init(&sm.drain[lane], 1);
    if (lane == 2) mbar_init(&sm.q_ready, 8);
    fence_mbar_init();
  }
  // Paged cache: the block-table entries of pages [page0, page0 + n_pages)
  // (the CTA's key range) are read once into shared memory.
  const int pr = a.page_rows;
  int page0 = 0, n_pages = 0;
  if (a.block_table != nullptr && nt > 0) {
    page0 = jt0 * kKeys / pr;
    n_pages = min(kPageCache, (n_max - 1) / pr - page0 + 1);
    for (int i = tid; i < n_pages; i += kThreads) sm.pages[i] = a.block_table[page0 + i];
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
      prefetch_tmap(&tm_o);
      if (early_q) grid_dependency_wait();  // the K copies are the pre-pass's output
      // Copies go out in the order the MMA issuer consumes the tiles: K_0,
      // K_1, V_0, K_2, V_1, ..., K_(nt-1), V_(nt-2), V_(nt-1).  Ring slot
      // p % kRing holds copy p; it is refilled once its consumer completes.
      for (int p = 0; p < 2 * nt; ++p) {
        const int s = p % kRing, use = p / kRing;
        unsigned char* dst = sm.ring + s * kTileBytes;
        if (p == 2) mbar_wait_bounded(&sm.q_ready, 0, a.status, &sm.abort);  // the staging slot is free again
        if (use >= 1) mbar_wait_bounded(&sm.kv_empty[s], (unsigned)((use - 1) & 1), a.status, &sm.abort);
        const bool is_v = (p == 2 * nt - 1) || (p > 0 && (p & 1) == 0);
        mbar_arrive_expect_tx(&sm.kv_full[s], (unsigned)(is_v ? kTileBytes : kKBytes));
        const int t0 = kKeys * (jt0 + (is_v ? (p == 2 * nt - 1 ? nt - 1 : p / 2 - 1) : (p + 1) / 2));
        if (!is_v) {
          // K: the pre-pass's fp16 copy (logical rows, also for a paged
          // cache), 64-element column chunks.
#pragma unroll
          for (int c = 0; c < kKChunks; ++c) tma_load_2d(dst + c * kChunkBytes, &tm_k, g * D + 64 * c, t0, &sm.kv_full[s]);
        } else if (a.block_table == nullptr) {
#pragma unroll
          for (int c = 0; c < kChunks; ++c) tma_load_2d(dst + c * kChunkBytes, &tm_v, g * D + kEpr * c, t0, &sm.kv_full[s]);
        } else {
          // Paged: boxes of page_box rows (128, 64 or 32: the largest that
          // divides page_rows), each inside one page.  Rows no query of the
          // CTA reads, and pages outside the pool, come from a row past the
          // pool's end (zeros).
          const int box = page_box(pr);
          for (int sub = 0; sub < kKeys / box; ++sub) {
            const int t = t0 + box * sub;
            int y = a.num_pages * pr;
            if (t < n_max) {
              const int pi = t / pr;
              const uint32_t page = pi - page0 < n_pages ? sm.pages[pi - page0] : a.block_table[pi];
              if (page < (uint32_t)a.num_pages)
                y = (int)page * pr + t % pr;
              else
                record_status(a.status, ATTN_ERR_INVALID_ARG);
            }
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
              tma_load_2d(dst + c * kChunkBytes + sub * box * 128, &tm_v, g * D + kEpr * c, y, &sm.kv_full[s]);
          }
        }
      }
      // No copy may still be landing in shared memory when the CTA exits
      // (normally every fill was already consumed, so these return at once).
      for (int s = 0; s < kRing && s < 2 * nt; ++s) {
        const int last = s + ((2 * nt - 1 - s) / kRing) * kRing;
        mbar_wait_bounded(&sm.kv_full[s], (unsigned)((last / kRing) & 1), a.status);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issue
    // Warp 1 issues Q K^T, warp 2 P V, each in tile order.  The whole warp
    // runs its loop (warp-uniform values); one elected lane issues each MMA
    // and commit.
    if (nt > 0) {
      constexpr uint32_t idesc_qk = tc::idesc_f32acc(tc::kFmtF16, false, kRows, kKeys);
      constexpr uint32_t idesc_pv = tc::idesc_f32acc(tc::kFmtTF32, true, kRows, D);
      // V (MN-major B): the 32-byte-atom layout, 4-row K groups 512 bytes apart.
      constexpr uint32_t kVStep = kKStep * 128;  // bytes of V rows per K step
      // One descriptor per operand form at the ring's base; an operand at byte
      // offset off is that descriptor plus off >> 4 (the start-address field;
      // shared-memory offsets stay far below its 14-bit range).
      const uint32_t ring0 = smem_u32(sm.ring);
      const uint64_t dk0 = tc::sdesc_sw128(ring0, 16, 1024);
      const uint64_t dv0 = tc::sdesc_sw128(ring0, kChunkBytes, 512, tc::kLayoutSw128Atom32);
      auto slot_off = [&](int p) { return (uint64_t)(((p % kRing) * kTileBytes) >> 4); };
      auto wait = [&](uint64_t* bar, int phase) {
        return __all_sync(0xffffffffu, mbar_wait_bounded(bar, (unsigned)(phase & 1), a.status, &sm.abort));
      };
      // Ring positions of K_j and V_j (the copy order above).
      auto k_pos = [&](int j) { return j == 0 ? 0 : 2 * j - 1; };
      auto v_pos = [&](int j) { return j == nt - 1 ? 2 * nt - 1 : 2 * j + 2; };
      // S_(j%2) = Q K_j^T; it overwrites the P that P V of tile j-2 reads.
      auto issue_qk = [&](int j) {
        const int p = k_pos(j), b = j % kSBuf;
        if (!wait(&sm.kv_full[p % kRing], p / kRing)) return false;
        if (j >= kSBuf && !wait(&sm.pv_done[b], (j - kSBuf) / kSBuf)) return false;
        tc::fence_after_sync();
        const uint64_t dk = dk0 + slot_off(p);
        const uint32_t ds = tmem + kColS0 + kKeys * b;
        // Four K steps (16 fp16, 32 bytes each) per 128-byte chunk of the K
        // tile; Q takes 8 TMEM columns (16 packed fp16) per step.  Per chunk:
        // Qhi K and Qlo K, both accumulating into S.
#pragma unroll
        for (int c4 = 0; c4 < kKChunks; ++c4) {
          const uint64_t c = (uint64_t)((c4 * kChunkBytes) >> 4);
          const uint32_t qh = tmem + kColQ + 32 * c4, ql = qh + kColQl;
          tc::mma4_f16_ts(ds, qh, qh + 8, qh + 16, qh + 24, dk + c, dk + c + 2, dk + c + 4, dk + c + 6, idesc_qk,
                          c4 > 0 ? 1u : 0u);
          tc::mma4_f16_ts(ds, ql, ql + 8, ql + 16, ql + 24, dk + c, dk + c + 2, dk + c + 4, dk + c + 6, idesc_qk, 1u);
        }
        tc::commit_elect(&sm.s_full[b]);
        tc::commit_elect(&sm.kv_empty[p % kRing]);
        return true;
      };
      // O += P_j V_j once both softmax groups have written P_j.
      auto issue_pv = [&](int j) {
        const int p = v_pos(j), b = j % kSBuf;
        if (!wait(&sm.kv_full[p % kRing], p / kRing)) return false;
        if (!wait(&sm.p_ready[b], j / kSBuf)) return false;
        tc::fence_after_sync();
        const uint64_t dv = dv0 + slot_off(p);
        const uint32_t dp = tmem + kColS0 + kKeys * b;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int c4 = 0; c4 < kKeys / kKStep / 4; ++c4) {
          // K steps 4 c4 .. 4 c4 + 3; P takes 8 TMEM columns per step.
          const uint32_t pa = dp + 32 * c4;
          constexpr uint64_t st = kVStep >> 4;  // V rows of one K step
          const uint64_t c = 4 * st * c4;
          tc::mma4_tf32_ts(tmem + kColO, pa, pa + 8, pa + 16, pa + 24, dv + c, dv + c + st, dv + c + 2 * st,
                           dv + c + 3 * st, idesc_pv, c4 > 0 ? 1u : acc0);
        }
        tc::commit_elect(&sm.pv_done[b]);
        tc::commit_elect(&sm.kv_empty[p % kRing]);
        return true;
      };
      // Every wait blocks in hardware (a loop of test-waits competes with
      // the tensor core for shared memory and notices completions late).
      if (warp == 1) {
        bool ok = wait(&sm.q_ready, 0);
        tc::fence_after_sync();
        for (int j = 0; ok && j < nt; ++j) ok = issue_qk(j);
      } else {
        bool ok = true;
        for (int j = 0; ok && j < nt; ++j) ok = issue_pv(j);
      }
      // Every MMA has finished before tensor memory is released.
      tc::commit_elect(&sm.drain[warp - 1]);
      mbar_wait_bounded(&sm.drain[warp - 1], 0, a.status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / epilogue
    constexpr int kHalfD = D / 2;              // O columns per group
    const int grp = (warp - 4) >> 2;           // column group 0 or 1
    const int r = 32 * (warp & 3) + lane;      // row == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const long long qi = i0 + r / gs;         // packed row blk * rpb + r
    const int h = g * gs + r % gs;
    const bool row_ok = r < rpb && qi < a.n_q;
    const int n_r = row_ok ? window(qi) : 0;
    const int lo_r = first_key(n_r, a.window);
    const float sl2 = a.scale * kLog2e;

    // Q row -> TMEM: pre-scaled by scale * log2(e) and by the row's power of
    // two (its largest magnitude into [2^14, 2^15)), then split into fp16 hi
    // and lo parts, two values per column; each group converts half the row,
    // read from the staging slot (rows past n_q arrived as zeros), and the two
    // halves agree on the power of two through shared memory.
    float f_row = 1.f;  // 2^(E_r - 14): turns this row's raw scores back
    if (nt > 0) {
      constexpr int kQCols = D / 2;
      mbar_wait_bounded(&sm.q_full, 0, a.status, &sm.abort);
      // RoPE: the group's half pairs with the other half of the row (query
      // qi at position base_pos + qi; rows past n_q are zeros and stay so).
      const float* cs = (a.rope != nullptr && row_ok) ? a.rope + (a.base_pos + qi) * D : nullptr;
      const float sgn = grp == 0 ? -1.f : 1.f;
      float v[kQCols / 32][32];
      float qmax = 0.f;
#pragma unroll
      for (int c = 0; c < kQCols / 32; ++c) {
        const unsigned char* src = qstage + (grp * (kQCols / 32) + c) * kChunkBytes + r * 128;
        // The chunk's eight loads are issued before any is used.
        float4 x[8];
        if (r < rpb) {
#pragma unroll
          for (int u = 0; u < 8; ++u) x[u] = *reinterpret_cast<const float4*>(src + 16 * (u ^ (r & 7)));
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (cs != nullptr) {  // rows with a table are rows below rpb
          const unsigned char* other = qstage + ((1 - grp) * (kQCols / 32) + c) * kChunkBytes + r * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 y = *reinterpret_cast<const float4*>(other + 16 * (u ^ (r & 7)));
            const float4 cv = *reinterpret_cast<const float4*>(cs + 32 * c + 4 * u);
            const float4 sv = *reinterpret_cast<const float4*>(cs + kQCols + 32 * c + 4 * u);
            x[u] = make_float4(fmaf(sgn * y.x, sv.x, x[u].x * cv.x), fmaf(sgn * y.y, sv.y, x[u].y * cv.y),
                               fmaf(sgn * y.z, sv.z, x[u].z * cv.z), fmaf(sgn * y.w, sv.w, x[u].w * cv.w));
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          v[c][4 * u] = x[u].x * sl2;
          v[c][4 * u + 1] = x[u].y * sl2;
          v[c][4 * u + 2] = x[u].z * sl2;
          v[c][4 * u + 3] = x[u].w * sl2;
          qmax = fmaxf(qmax, fmaxf(fmaxf(fabsf(v[c][4 * u]), fabsf(v[c][4 * u + 1])),
                                   fmaxf(fabsf(v[c][4 * u + 2]), fabsf(v[c][4 * u + 3]))));
        }
      }
      sm.red_l[grp][r] = qmax;
      named_barrier(1, kSoftmaxThreads);
      const int er = pow2_scale_exp(fmaxf(sm.red_l[0][r], sm.red_l[1][r]));
      const float up = pow2f(14 - er);
      f_row = pow2f(er - 14);
#pragma unroll
      for (int c = 0; c < kQCols / 32; ++c) {
        // Element pairs (2i, 2i+1) of the chunk: hi = fp16 of each, lo = fp16
        // of what hi leaves (exact in fp32).  Pair i goes to column i.
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float y0 = v[c][2 * i] * up, y1 = v[c][2 * i + 1] * up;
          const uint32_t h = tc::pack_f16(y0, y1);
          const float2 hf = tc::unpack_f16(h);
          hi[i] = h;
          lo[i] = tc::pack_f16(y0 - hf.x, y1 - hf.y);
        }
        const uint32_t qcol = tmem + lane_base + kColQ + (grp * kQCols + 32 * c) / 2;
        tc::tmem_st16(qcol, hi);
        tc::tmem_st16(qcol + kColQl, lo);
      }
      tc::tmem_st_wait();
    }
    {
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.q_ready);
    }
    if (early_q) grid_dependency_wait();  // the pre-pass's output; before the outputs are written
    // The K tiles' powers of two (the pre-pass's output), read once.
    for (int i = 32 * (warp - 4) + lane; i < min(nt, kFacCache); i += kSoftmaxThreads)
      sm.kfac[i] = kfac[(long long)(jt0 + i) * a.G + g];
    named_barrier(2, kSoftmaxThreads);
    auto tile_fac = [&](int j) {
      return j < kFacCache ? sm.kfac[j] : __ldg(kfac + (long long)(jt0 + j) * a.G + g);
    };
    float f_next = nt > 0 ? tile_fac(0) : 1.f;

    constexpr int kCols = kKeys / 2;           // score columns per group per tile
    constexpr int kCC = kCols / 32;            // 32-column TMEM loads per group per tile
    float m_ref = -INFINITY, m_true = -INFINITY, l = 0.f;
    for (int j = 0; j < nt; ++j) {
      const int b = j % kSBuf;
      const uint32_t s_col = tmem + lane_base + kColS0 + kKeys * b + kCols * grp;
      // Raw score -> base-2 units (at least FLT_MIN, so a masked -inf stays -inf).
      const float cf = fmaxf(f_row * f_next, FLT_MIN);
      mbar_wait_bounded(&sm.s_full[b], (unsigned)((j / kSBuf) & 1), a.status, &sm.abort);
      tc::fence_after_sync();
      uint32_t s[kCC][32];
#pragma unroll
      for (int c = 0; c < kCC; ++c) tc::tmem_ld32(s_col + 32 * c, s[c]);
      tc::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < kCC; ++c) tc::reg_fence(s[c]);

      // Mask (only a tile that crosses some row's window end or start) and
      // this half's max.
      const int key0 = (jt0 + j) * kKeys + kCols * grp;  // key of this half's first column
      if (key0 - kCols * grp + kKeys > n_min) {
        const int lim = n_r - key0;
#pragma unroll
        for (int c = 0; c < kCC; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * c + e >= lim) s[c][e] = __float_as_uint(-INFINITY);
      }
      if (key0 - kCols * grp < lo_max) {
        const int lim = lo_r - key0;
#pragma unroll
        for (int c = 0; c < kCC; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * c + e < lim) s[c][e] = __float_as_uint(-INFINITY);
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < kCols; i += 8)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mx[k] = max3(mx[k], __uint_as_float(s[i >> 5][(i & 31) + 2 * k]), __uint_as_float(s[i >> 5][(i & 31) + 2 * k + 1]));
      sm.red_max[j & 1][grp][r] = max3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
      named_barrier(1, kSoftmaxThreads);
      const float tmax = cf * fmaxf(sm.red_max[j & 1][0][r], sm.red_max[j & 1][1][r]);
      if (j + 1 < nt) f_next = tile_fac(j + 1);
      m_true = fmaxf(m_true, tmax);
      float corr = 1.f;
      if (tmax > m_ref + kRescaleThreshold) {  // also true for the first finite tile max
        corr = ex2(m_ref - tmax);              // m_ref = -inf gives 0
        m_ref = tmax;
      }
      const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
      // P = 2^(S - m) in place.  The tensor core reads its 32-bit operands as
      // TF32 (the low 13 mantissa bits dropped), so P is stored unrounded; the
      // row sum is taken over the unrounded values.
      float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < kCC; ++c) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float x0 = __uint_as_float(s[c][e]), x1 = __uint_as_float(s[c][e + 1]);
          fma2(x0, x1, cf, cf, neg_m, neg_m);
          const float p0 = ex2(x0), p1 = ex2(x1);
          const int k = (e >> 1) & 3;
          add2(sum[2 * k], sum[2 * k + 1], p0, p1);
          s[c][e] = __float_as_uint(p0);
          s[c][e + 1] = __float_as_uint(p1);
        }
        tc::tmem_st32(s_col + 32 * c, s[c]);
      }
      l = l * corr + (((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7])));
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
    // O / l leaves by TMA tensor stores.  Each group stages its D/2 columns in
    // the (now idle) K/V ring as 32-float chunks of 128 rows x 128 bytes, in
    // the order of a 3-D box {32 floats, gs heads, 128/gs queries} (row r =
    // query r / gs, head r % gs of the block) with the 128-byte swizzle
    // (16-byte unit u of row r at u ^ (r & 7)); one thread then stores every
    // chunk with one box each.  Rows past n_q fall outside the tensor and are
    // not written, nor are the idle rows past (128/gs)*gs.
    constexpr int kOChunks = kHalfD / 32;  // 32-float chunks per group
    unsigned char* const ostage = sm.ring;   // [group][chunk][128 rows][128 bytes]
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the ring was last written by TMA
#pragma unroll
    for (int c = 0; c < kOChunks; ++c) {
      uint32_t o[32];
      if (nt > 0) {
        tc::tmem_ld32(tmem + lane_base + kColO + grp * kHalfD + 32 * c, o);
        tc::tmem_ld_wait();
        tc::reg_fence(o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      unsigned char* dst = ostage + (grp * kOChunks + c) * (kRows * 128) + r * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<float4*>(dst + 16 * (u ^ (r & 7))) =
            make_float4(__uint_as_float(o[4 * u]) * inv, __uint_as_float(o[4 * u + 1]) * inv,
                        __uint_as_float(o[4 * u + 2]) * inv, __uint_as_float(o[4 * u + 3]) * inv);
    }
    // The tensor stores read the staging chunks through the async proxy.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    named_barrier(1, kSoftmaxThreads);
    if (warp == 4 && lane == 0) {
      for (int k = 0; k < 2 * kOChunks; ++k) tma_store_3d(&tm_o, ostage + k * (kRows * 128), 32 * k, g * gs, (int)i0);
      bulk_commit();
      bulk_wait_read_all();  // the staging memory stays live until the stores have read it
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

template <int D>
int launch_d(const FlashArgs& a, cudaStream_t s) {
  const int gs = a.H / a.G;
  const int qpb = kRows / gs;  // queries per 128-row block
  const long long nb = ((long long)a.n_q + qpb - 1) / qpb;
  if (nb == 0) return 0;
  // Logical K/V rows any CTA may read: the largest window of the call.  Rows
  // past it are outside the tensor maps and arrive as zeros.  A paged V is
  // read from its pool (the whole pool is mapped).
  long long kv_rows = a.causal ? a.base_pos + a.n_q : a.n_all;
  if (kv_rows > a.cap) kv_rows = a.cap;
  const bool paged = a.block_table != nullptr;
  const bool no_keys = kv_rows < 1 || a.k == nullptr || a.v == nullptr;
  if (kv_rows < 1) kv_rows = 1;
  const long long v_rows = (paged && !no_keys) ? (long long)a.num_pages * a.page_rows : kv_rows;
  // An empty key set never reads K/V: any aligned base will do.
  const void* khp = a.q;
  const void* vp = no_keys ? static_cast<const void*>(a.q) : a.v;
  void* scratch = nullptr;
  uint16_t* kh16 = nullptr;
  const float* kfac = nullptr;
  if (!no_keys) {
    // K as fp16 with one power of two per (tile, kv head) (turned by RoPE,
    // gathered from pages) in stream-ordered scratch memory (library pool),
    // released on the same stream once the attention kernel has run.  Only
    // tiles from the first one any CTA reads are written.
    const long long elems = kv_rows * a.kv_row_stride;
    const int n_first = a.causal ? (int)min((long long)a.cap, a.base_pos + 1) : a.n_all;  // window of query 0
    const size_t fac_off = scratch_round((size_t)elems * 2);
    if (scratch_alloc(&scratch, flash_tc_scratch_bytes(a), s) != cudaSuccess) return ATTN_ERR_CUDA;
    const int n_tiles = (int)((kv_rows + kKeys - 1) / kKeys);
    kh16 = static_cast<uint16_t*>(scratch);
    kfac = reinterpret_cast<float*>(static_cast<char*>(scratch) + fac_off);
    PrepArgs pa{};
    pa.k = a.k;
    pa.v = a.v;
    pa.out0 = kh16;
    pa.out1 = nullptr;  // V is read as it is
    pa.kfac = const_cast<float*>(kfac);
    pa.stride = a.kv_row_stride;
    pa.G = a.G;
    pa.D = D;
    pa.tile0 = first_key(n_first, a.window) / kKeys;
    pa.n_tiles = n_tiles;
    pa.rows_end = kv_rows;
    pa.rope = a.rope;
    pa.table = a.block_table;
    pa.page_rows = a.page_rows;
    pa.num_pages = a.num_pages;
    pa.status = a.status;
    if (launch_kv_prep(pa, s) != cudaSuccess) {
      scratch_free(scratch, s);
      return ATTN_ERR_CUDA;
    }
    khp = kh16;
  }
  CUtensorMap tm_k, tm_v, tm_q, tm_o;
  // Q: fp32 [n_q][H][D] (query rows q_row_stride floats apart); one CTA's
  // block is D/32 boxes of 32 floats x gs heads x 128/gs queries, rows past
  // n_q read as 0.
  const uint64_t qdims[3] = {(uint64_t)D, (uint64_t)a.H, (uint64_t)a.n_q};
  const uint64_t qstrides[2] = {(uint64_t)D * 4, (uint64_t)a.q_row_stride * 4};
  const uint32_t qbox[3] = {32, (uint32_t)gs, (uint32_t)qpb};
  // out: the same box over [n_q][H][D] (query rows out_row_stride floats apart).
  const uint64_t odims[3] = {(uint64_t)D, (uint64_t)a.H, (uint64_t)a.n_q};
  const uint64_t ostrides[2] = {(uint64_t)D * 4, (uint64_t)a.out_row_stride * 4};
  // K: [kv_rows][kv_row_stride] fp16, boxes of 64 elements x 128 keys.
  const uint64_t kdims[2] = {(uint64_t)a.kv_row_stride, (uint64_t)kv_rows};
  const uint64_t kstrides[1] = {(uint64_t)a.kv_row_stride * 2};
  const uint32_t kbox[2] = {64, (uint32_t)kKeys};
  // V: fp32 rows (a paged pool: boxes inside one page).
  const uint64_t vdims[2] = {(uint64_t)a.kv_row_stride, (uint64_t)v_rows};
  const uint64_t vstrides[1] = {(uint64_t)a.kv_row_stride * 4};
  const uint32_t vbox[2] = {32, (uint32_t)(paged ? page_box(a.page_rows) : kKeys)};
  int rc = ATTN_OK;
  if (!make_tmap(&tm_k, khp, 2, kdims, kstrides, kbox, true, kSwizzle128) ||
      !make_tmap(&tm_v, vp, 2, vdims, vstrides, vbox, false, kSwizzle128Atom32) ||
      !make_tmap(&tm_q, a.q, 3, qdims, qstrides, qbox, false, kSwizzle128) ||
      !make_tmap(&tm_o, a.out, 3, odims, ostrides, qbox, false, kSwizzle128)) {
    rc = ATTN_ERR_UNSUPPORTED;
  } else {
    const size_t smem = sizeof(TcSmem) + 1024;
    auto kern = flash_tc_kernel<D>;
    if (!set_smem_limit(reinterpret_cast<const void*>(kern), smem)) {
      rc = ATTN_ERR_CUDA;
    } else {
      FlashArgs aa = a;
      int early_q = scratch != nullptr ? 1 : 0;  // the pre-pass ran just before
      void* args[] = {&aa, &tm_k, &tm_v, &tm_q, &tm_o, &kfac, &early_q};
      if (launch_pdl(reinterpret_cast<const void*>(kern), dim3((unsigned)nb, (unsigned)a.G), dim3(kThreads), smem, s,
                     args) != cudaSuccess)
        rc = ATTN_ERR_CUDA;
    }
  }
  if (scratch != nullptr && scratch_free(scratch, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
  return rc;
}

}  // namespace

// Logical K/V rows a call reads (at least 1) and whether it has no keys.
static long long kv_rows_of(const FlashArgs& a, bool* no_keys) {
  long long kv_rows = a.causal ? a.base_pos + a.n_q : a.n_all;
  if (kv_rows > a.cap) kv_rows = a.cap;
  *no_keys = kv_rows < 1 || a.k == nullptr || a.v == nullptr;
  return kv_rows < 1 ? 1 : kv_rows;
}

// K as fp16 (kv_rows x kv_row_stride) and one float per (128-key tile, kv head).
size_t flash_tc_scratch_bytes(const FlashArgs& a) {
  bool no_keys = false;
  const long long kv_rows = kv_rows_of(a, &no_keys);
  if (no_keys || a.n_q == 0) return 0;
  return scratch_round(scratch_round((size_t)kv_rows * a.kv_row_stride * 2) +
                       (size_t)((kv_rows + kKeys - 1) / kKeys) * a.G * sizeof(float));
}

bool flash_tc_supported(const FlashArgs& a, int prec) {
  if (prec != ATTN_TF32 && prec != ATTN_BF16) return false;
  if (a.kv_pos_dev != nullptr) return false;
  if (a.D != 64 && a.D != 128) return false;
  if (a.G > 65535) return false;
  const int gs = a.H / a.G;
  if (gs < 1 || gs > kRows) return false;
  const uintptr_t al = reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.out) |
                       reinterpret_cast<uintptr_t>(a.k) | reinterpret_cast<uintptr_t>(a.v);
  if (al % 16 != 0) return false;
  if (a.q_row_stride % 4 != 0 || a.out_row_stride % 4 != 0 || a.kv_row_stride % 4 != 0) return false;
  if (a.kv_row_stride % 8 != 0) return false;  // the 16-bit K (and V) copies: rows in 16-byte units
  if (a.block_table != nullptr && (a.page_rows % kPageBox != 0 || (long long)a.num_pages * a.page_rows > 0x7fffffffLL))
    return false;
  return true;
}

int launch_flash_tc(const FlashArgs& a, int prec, cudaStream_t s) {
  if (!flash_tc_supported(a, prec)) return ATTN_ERR_UNSUPPORTED;
  if (prec == ATTN_BF16) return launch_flash_bf16(a, s);
  return a.D == 128 ? launch_d<128>(a, s) : launch_d<64>(a, s);
}

}  // namespace attn
