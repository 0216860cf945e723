// flash_bf16.cu -- tcgen05 flash attention with 16-bit operands (forward and
// prefill): Q K^T in fp16, P V in bf16, both accumulated in fp32.
//
// Operation: softmax(scale * Q K^T) V over per-row causal / full / cross /
// prefill windows (optionally cut to their last `window` keys) with the
// online softmax's running max and sum (cera attention_prefill.wgsl, fn
// attention_prefill: per-tile max, correction, exponentials, running sum;
// meganeura attention.wgsl, fn main: the final (max, log sum) store).
//
// Operand precision.  The scores decide the softmax weights exponentially,
// so their operands carry 11 significant bits (fp16) instead of bf16's 8:
// with scores of standard deviation 9 (Q, K ~ N(0, 3^2), D = 128) bf16 Q and
// K move the output by up to about 2.2e-2 max|V|, fp16 ones by about 3e-3.
// fp16 has a narrow exponent range, so every operand set carries a power of
// two: each query row r is stored as q * scale * log2(e) * 2^(14 - E_r) and
// each 128-key tile T of a kv head as k * 2^(14 - E_T), where E is the
// binary exponent of the set's largest magnitude (so its values lie below
// 2^15, inside fp16's range, whatever the fp32 inputs).  The product of the
// two powers of two, 2^(E_r + E_T - 28), turns a raw score back into base-2
// units in the softmax, at no extra instruction (it is the multiplier of the
// fma that subtracts the running max).  P (<= 256) and V keep bf16 operands:
// their rounding enters the output linearly, not through an exponential.
// A pre-pass writes K as fp16 (with the tile factors) and V as bf16, in
// their own layout; Q is converted inside the kernel.
//
// One CTA owns the packed rows of 128/gs queries of one kv head g (rpb =
// (128/gs)*gs of its 128 MMA rows; the rest idle when gs does not divide
// 128): row r is (query i, head g*gs + j) with i*gs + j = rpb*block + r, so
// each K/V tile feeds all gs query heads that share it.  Keys are walked in
// tiles of 128, from the tile holding the block's first kept key to the one
// holding its last.
//
// Two score buffers S_0, S_1 and two P buffers in tensor memory let Q K^T of
// tile j + 2 start as soon as the softmax has read S_(j%2) (P_j has its own
// columns), so the tensor core is not held up by P V.  The two softmax
// warpgroups take alternate key tiles (group 0 the even ones, group 1 the
// odd ones), each thread a whole 128-column row, so while one group waits
// for its scores the other computes exponentials.  The reference max that P
// is taken against is one chain through the tiles: the warp of tile j reads
// the reference its counterpart (same 32 rows, other group) left at tile
// j - 1, moves it to the tile max when that exceeds it by more than 24 (so P
// <= 2^24; a wide gap between the two only makes P large, which fp32
// accumulation and bf16's 8-bit exponent carry without loss), and hands it
// on through shared memory and a per-warp barrier.  When the reference
// moves, the warp rescales its rows of the single O accumulator once P V of
// tile j - 1 has landed.  Each group keeps the row sum of its own tiles;
// the two sums are combined at the end.
//
// Warp roles (352 threads):
//   warp 0      TMA producer: K tile (128 keys x D, 128-byte swizzle, K-major)
//               and V tile (the same boxes; read as the MN-major operand of
//               P V) into a shared-memory ring, in the order they are consumed.
//   warp 1      tensor-memory allocation; issues S_(j%2) = Q K_j^T
//               (A = Q in shared memory, B = K tile) once the softmax has
//               read the scores of tile j - 2 from that buffer.
//   warp 2      issues O += P_j V_j (A = P_(j%2) in TMEM, B = V tile) in
//               tile order once P_j is written.
//   warps 3-10  softmax, two groups of four warps (3-6 and 7-10): warp w
//               covers rows 32(w%4)..+31 (its TMEM lanes).
// The issuing warps run their loops warp-uniformly; one elected lane issues.
// Tensor memory (512 columns): S_b [128 b, 128 b + 128) and P_b [256 + 64 b,
// 256 + 64 b + 64) for b = 0, 1, O [384, 384 + D).  Scores are in base-2
// units once scaled (Q carries scale * log2(e)).  The true max is tracked
// apart for the LSE.  Every wait is bounded; a CTA whose pipeline breaks
// drains its copies and MMAs before it releases tensor memory.
#include <cfloat>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace attn {
namespace {

constexpr int kRows = 128;                 // packed rows per CTA (MMA M)
constexpr int kKeys = 128;                 // keys per tile
constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;
constexpr int kOperandBytes = 192 * 1024;  // Q tile + K/V ring
constexpr int kMaxRing = 12;
constexpr int kSBuf = 2;                   // score buffers (and P buffers)
constexpr int kColP = 256;                 // S_b at 128 b, P_b at 256 + 64 b, O at 384
constexpr int kColO = 384;
constexpr float kRescaleThreshold = 24.0f;  // log2 units: P <= 2^24
constexpr int kFacCache = 512;             // K tile powers of two a CTA keeps in shared memory

struct __align__(1024) Bf16Smem {
  unsigned char operands[kOperandBytes];  // [Q tile][ring slots]
  uint64_t kv_full[kMaxRing];
  uint64_t kv_empty[kMaxRing];
  uint64_t s_full[kSBuf];
  uint64_t s_free[kSBuf];  // the softmax has read S_b of the tile
  uint64_t mref_bar[4][2];  // [row quarter][tile parity]: the tile's reference max is in mref
  uint64_t p_ready[kSBuf];
  uint64_t pv_done[2];     // P V of tile j completes phase j/2 of pv_done[j & 1]
  uint64_t q_full;         // the fp32 Q block has landed in the staging area
  uint64_t q_ready;        // the bf16 Q tile is written
  uint64_t o_final;        // every P V has completed
  uint64_t drain[2];
  float mref[2][kRows];        // [tile parity][row] reference max handed from one tile's group to the next
  float red_m[2][kRows];       // [group][row] the group's last reference max
  float red_t[2][kRows];       // [group][row] the group's true max
  float red_l[2][kRows];       // [group][row] partial row maxima of Q, then partial row sums
  float kfac[kFacCache];       // powers of two of the CTA's K tiles jt0, jt0 + 1, ...
  uint32_t tmem_base;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    flash_bf16_kernel(const FlashArgs a, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_o, const float* __restrict__ kfac, int early_q,
                      int q_ahead) {
  constexpr int kChunks = D / 64;                // 128-byte (64-element) column chunks of a K row
  constexpr int kChunkBytes = kKeys * 128;       // one K box: 128 keys x 128 bytes
  constexpr int kTileBytes = kChunks * kChunkBytes;
  constexpr int kQBytes = kRows * D * 2;
  constexpr int kRing = (kOperandBytes - kQBytes) / kTileBytes;
  static_assert(kRing <= kMaxRing && kRing >= 4, "ring depth");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  Bf16Smem& sm = *reinterpret_cast<Bf16Smem*>(smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u));
  unsigned char* const qtile = sm.operands;
  unsigned char* const ring = sm.operands + kQBytes;
  // The CTA's fp32 Q block ([queries][gs heads][D], 128 rows of D floats)
  // lands by TMA in ring slots 3 and 4, which hold no K/V copy until the Q
  // tile has been converted.
  static_assert(2 * kTileBytes == kRows * D * 4, "Q staging fills two ring slots");
  const float* const qstage = reinterpret_cast<const float*>(ring + 3 * kTileBytes);

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
  const long long i0 = (long long)blk * qpb;
  auto window = [&](long long i) -> int {
    if (i < 0 || i >= a.n_q) return 0;
    if (!a.causal) return a.n_all;
    const long long w = a.base_pos + i + 1;
    return (int)(w < a.cap ? w : a.cap);
  };
  const int n_min = window(i0);
  const int n_max = window(min((long long)a.n_q, i0 + qpb) - 1);
  const int lo_max = first_key(n_max, a.window);
  const int jt0 = first_key(n_min, a.window) / kKeys;  // first key tile of the block
  const int nt = (n_max + kKeys - 1) / kKeys - jt0;    // key tiles the block walks
  // Ring positions (copy order): K_0, K_1, K_2, then V_j followed by K_(j+3).
  auto k_pos = [&](int j) { return j < 3 ? j : 2 * j - 2; };
  auto v_pos = [&](int j) { return min(2 * j + 3, j + nt); };

  if (warp == 0) {
    // The Q block is copied first, so that it lands while the rest of the
    // set-up runs; the other barriers are initialised across the warp.
    if (lane == 0) {
      mbar_init(&sm.q_full, 1);
      fence_mbar_init();
      if (nt > 0) {
        prefetch_tmap(&tm_q);
        mbar_arrive_expect_tx(&sm.q_full, (unsigned)(rpb * D * 4));
        tma_load_3d(ring + 3 * kTileBytes, &tm_q, 0, g * gs, (int)i0, &sm.q_full);
      }
      sm.abort = 0;
    }
    for (int s = lane; s < kRing; s += 32) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int b = lane; b < kSBuf; b += 32) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.s_free[b], 4);
      mbar_init(&sm.p_ready[b], 4);
    }
    for (int i = lane; i < 4 * kSBuf; i += 32) mbar_init(&sm.mref_bar[i / kSBuf][i % kSBuf], 32);
    if (lane < 2) {
      mbar_init(&sm.pv_done[lane], 1);
      mbar_init(&sm.drain[lane], 1);
    }
    if (lane == 2) {
      mbar_init(&sm.q_ready, 8);
      mbar_init(&sm.o_final, 1);
    }
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
      prefetch_tmap(&tm_o);
      if (early_q) grid_dependency_wait();  // the K/V copies are the pre-pass's output
      int p = 0;  // copies issued; copy p goes to ring slot p % kRing
      auto load = [&](bool is_v, int j) {
        const int s = p % kRing, use = p / kRing;
        if (p == 3) mbar_wait_bounded(&sm.q_ready, 0, a.status, &sm.abort);  // slots 3-4 free again
        unsigned char* dst = ring + s * kTileBytes;
        if (use >= 1) mbar_wait_bounded(&sm.kv_empty[s], (unsigned)((use - 1) & 1), a.status, &sm.abort);
        mbar_arrive_expect_tx(&sm.kv_full[s], (unsigned)kTileBytes);
        const int t0 = kKeys * (jt0 + j);
        const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) tma_load_2d(dst + c * kChunkBytes, tm, g * D + 64 * c, t0, &sm.kv_full[s]);
        ++p;
      };
      for (int t = 0; t < 3 && t < nt; ++t) load(false, t);
      // After the first K copies: the CTA q_ahead places later in launch order (about one wave of the
      // grid) finds its Q block in L2: its start then waits for L2, not HBM.
      const long long la = (long long)blockIdx.y * gridDim.x + blockIdx.x + q_ahead;
      if (q_ahead > 0 && la < (long long)gridDim.x * gridDim.y) {
        const int xa = (int)(la % gridDim.x), ya = (int)(la / gridDim.x);
        tma_prefetch_l2_3d(&tm_q, 0, ya * gs, (int)((long long)(gridDim.x - 1 - xa) * qpb));
      }
      for (int j = 0; j < nt; ++j) {
        load(true, j);
        if (j + 3 < nt) load(false, j + 3);
      }
      // No copy may still be landing in shared memory when the CTA exits.
      for (int s = 0; s < kRing && s < p; ++s) {
        const int last = s + ((p - 1 - s) / kRing) * kRing;
        mbar_wait_bounded(&sm.kv_full[s], (unsigned)((last / kRing) & 1), a.status);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issue
    // Warp-uniform loops; one elected lane issues each MMA and commit.
    if (nt > 0) {
      // Operands use the 128-byte swizzle with 1024-byte groups of 8 rows; an
      // operand at byte offset off from a base is the base's descriptor plus
      // off >> 4 (the start-address field).  K (and Q) are K-major; V is read
      // MN-major: each key row holds 64 elements of D per 128-byte chunk,
      // chunks kChunkBytes apart.
      const uint64_t dk0 = tc::sdesc_sw128(smem_u32(ring), 16, 1024);
      const uint64_t dv0 = tc::sdesc_sw128(smem_u32(ring), kChunkBytes, 1024);
      auto slot_off = [&](int p) { return (uint64_t)(((p % kRing) * kTileBytes) >> 4); };
      auto wait = [&](uint64_t* bar, int phase) {
        return __all_sync(0xffffffffu, mbar_wait_bounded(bar, (unsigned)(phase & 1), a.status, &sm.abort));
      };
      if (warp == 1) {
        // S_b = Q K_j^T, b = j % 3.  It overwrites the P that P V of tile
        // j-3 reads, so that product must have completed.
        constexpr uint32_t idesc_qk = tc::idesc_f32acc(tc::kFmtF16, false, kRows, kKeys);
        const uint64_t dq = tc::sdesc_sw128(smem_u32(qtile), 16, 1024);
        bool ok = wait(&sm.q_ready, 0);
        tc::fence_after_sync();
        for (int j = 0; ok && j < nt; ++j) {
          const int pk = k_pos(j), b = j % kSBuf;
          ok = wait(&sm.kv_full[pk % kRing], pk / kRing) && (j < kSBuf || wait(&sm.s_free[b], (j - kSBuf) / kSBuf));
          if (!ok) break;
          tc::fence_after_sync();
          const uint64_t dk = dk0 + slot_off(pk);
          const uint32_t ds = tmem + kKeys * b;
#pragma unroll
          for (int c4 = 0; c4 < kChunks; ++c4) {  // four 16-element K steps per 64-element chunk
            const uint64_t c = (uint64_t)((c4 * kChunkBytes) >> 4);
            tc::mma4_f16_ss(ds, dq + c, dq + c + 2, dq + c + 4, dq + c + 6, dk + c, dk + c + 2, dk + c + 4,
                            dk + c + 6, idesc_qk, c4 > 0 ? 1u : 0u);
          }
          tc::commit_elect(&sm.s_full[b]);
          tc::commit_elect(&sm.kv_empty[pk % kRing]);
        }
        tc::commit_elect(&sm.drain[0]);
        mbar_wait_bounded(&sm.drain[0], 0, a.status);
      } else {
        // O += P_j V_j in tile order.
        constexpr uint32_t idesc_pv = tc::idesc_f32acc(tc::kFmtBF16, true, kRows, D);
        bool ok = true;
        for (int j = 0; ok && j < nt; ++j) {
          const int pv = v_pos(j), b = j % kSBuf;
          ok = wait(&sm.p_ready[b], j / kSBuf) && wait(&sm.kv_full[pv % kRing], pv / kRing);
          if (!ok) break;
          tc::fence_after_sync();
          const uint64_t dv = dv0 + slot_off(pv);
          constexpr uint64_t st = (16 * 128) >> 4;  // one K step: 16 key rows of 128 bytes
#pragma unroll
          for (int c4 = 0; c4 < kKeys / 64; ++c4) {
            const uint64_t c = 4 * st * c4;
            const uint32_t pa = tmem + kColP + 64 * b + 32 * c4;  // P: 8 columns (16 keys) per K step
            tc::mma4_f16_ts(tmem + kColO, pa, pa + 8, pa + 16, pa + 24, dv + c, dv + c + st, dv + c + 2 * st,
                            dv + c + 3 * st, idesc_pv, (j > 0 || c4 > 0) ? 1u : 0u);
          }
          tc::commit_elect(&sm.pv_done[j & 1]);
          tc::commit_elect(&sm.kv_empty[pv % kRing]);
        }
        tc::commit_elect(&sm.o_final);
        tc::commit_elect(&sm.drain[1]);
        mbar_wait_bounded(&sm.drain[1], 0, a.status);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int grp = (warp - 3) >> 2;           // group 0 (warps 3-6) or 1 (warps 7-10)
    const int r = 32 * (warp & 3) + lane;      // row == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const long long qi = i0 + r / gs;         // packed row blk * rpb + r
    const int h = g * gs + r % gs;
    const bool row_ok = r < rpb && qi < a.n_q;
    const int n_r = row_ok ? window(qi) : 0;
    const int lo_r = first_key(n_r, a.window);
    const float sl2 = a.scale * kLog2e;

    // Q row, pre-scaled by scale * log2(e), as fp16 into the K-major operand
    // tile: 64-element chunk c holds 128 rows of 128 bytes, 16-byte unit u of
    // row r at unit u ^ (r & 7) (the 128-byte swizzle).  Group c converts
    // elements [c D/2, (c + 1) D/2) of its row; the two halves agree on the
    // row's power of two through shared memory.  Each thread starts at float4
    // r % (D/8) of its half, which spreads both the staging reads and the
    // tile writes over the banks.
    constexpr int kQF4 = D / 8;  // float4 groups per half row
    float f_row = 1.f;           // 2^(E_r - 14): turns this row's raw scores back
    if (nt > 0) {
      mbar_wait_bounded(&sm.q_full, 0, a.status, &sm.abort);
      const float* qrow = qstage + r * D;
      // RoPE: element e pairs with e +- D/2 (query qi at position base_pos + qi).
      const float* cs = (a.rope != nullptr && row_ok) ? a.rope + (a.base_pos + qi) * D : nullptr;
      // All of the half row's loads are issued before any is used.
      float4 xq[kQF4];
      if (r < rpb) {
#pragma unroll
        for (int i = 0; i < kQF4; ++i)
          xq[i] = *reinterpret_cast<const float4*>(qrow + grp * (D / 2) + 4 * ((i + r) % kQF4));
      } else {
#pragma unroll
        for (int i = 0; i < kQF4; ++i) xq[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (cs != nullptr) {
#pragma unroll
        for (int i = 0; i < kQF4; ++i) {
          const int e = grp * (D / 2) + 4 * ((i + r) % kQF4);  // first element of this float4
          const int dd = grp == 0 ? e : e - D / 2;               // pair index
          const float4 y = *reinterpret_cast<const float4*>(qrow + (grp == 0 ? e + D / 2 : dd));
          const float4 cv = *reinterpret_cast<const float4*>(cs + dd);
          const float4 sv = *reinterpret_cast<const float4*>(cs + D / 2 + dd);
          const float sg = grp == 0 ? -1.f : 1.f;
          const float4 x = xq[i];
          xq[i] = make_float4(fmaf(sg * y.x, sv.x, x.x * cv.x), fmaf(sg * y.y, sv.y, x.y * cv.y),
                              fmaf(sg * y.z, sv.z, x.z * cv.z), fmaf(sg * y.w, sv.w, x.w * cv.w));
        }
      }
      float qmax = 0.f;
#pragma unroll
      for (int i = 0; i < kQF4; ++i) {
        const float4 x = make_float4(xq[i].x * sl2, xq[i].y * sl2, xq[i].z * sl2, xq[i].w * sl2);
        xq[i] = x;
        qmax = fmaxf(qmax, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
      }
      sm.red_l[grp][r] = qmax;
      named_barrier(1, kSoftmaxThreads);
      const int er = pow2_scale_exp(fmaxf(sm.red_l[0][r], sm.red_l[1][r]));
      const float up = pow2f(14 - er);
      f_row = pow2f(er - 14);
#pragma unroll
      for (int i = 0; i < kQF4; ++i) {
        const int f = (i + r) % kQF4;
        const int e = grp * (D / 2) + 4 * f;
        const int u = (e & 63) >> 3;
        unsigned char* qdst = qtile + (e >> 6) * kChunkBytes + r * 128 + 16 * (u ^ (r & 7)) + 8 * ((e >> 2) & 1);
        const float4 x = xq[i];
        *reinterpret_cast<uint2*>(qdst) = make_uint2(tc::pack_f16(x.x * up, x.y * up), tc::pack_f16(x.z * up, x.w * up));
      }
    }
    // The tensor core reads the tile through the async proxy.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.q_ready);
    if (early_q) grid_dependency_wait();
    // The K tiles' powers of two (the pre-pass's output), read once.
    for (int i = 32 * (warp - 3) + lane; i < min(nt, kFacCache); i += kSoftmaxThreads)
      sm.kfac[i] = kfac[(long long)(jt0 + i) * a.G + g];
    named_barrier(2, kSoftmaxThreads);

    const uint32_t o_col = tmem + lane_base + kColO;
    // Group grp takes key tiles j = grp, grp + 2, ...: whole 128-column rows.
    // Each group keeps its own row sum and true max against the reference it
    // last used; the two are combined at the end.
    float m_ref = -INFINITY, m_true = -INFINITY, l = 0.f;
    auto tile_fac = [&](int j) {
      return j < kFacCache ? sm.kfac[j] : __ldg(kfac + (long long)(jt0 + j) * a.G + g);
    };
    for (int j = grp; j < nt; j += 2) {
      const int b = j % kSBuf;
      const uint32_t s_col = tmem + lane_base + kKeys * b;
      // Raw score -> base-2 units (at least FLT_MIN, so a masked -inf stays -inf).
      const float cf = fmaxf(f_row * tile_fac(j), FLT_MIN);
      mbar_wait_bounded(&sm.s_full[b], (unsigned)((j / kSBuf) & 1), a.status, &sm.abort);
      tc::fence_after_sync();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(s_col + 32 * c, s[c]);
      tc::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::reg_fence(s[c]);
      // S_b may take the scores of tile j + 2 now.
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_free[b]);

      const int key0 = (jt0 + j) * kKeys;  // key of the tile's first column
      if (key0 + kKeys > n_min) {          // the tile crosses some row's window end
        const int lim = n_r - key0;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * c + e >= lim) s[c][e] = __float_as_uint(-INFINITY);
      }
      if (key0 < lo_max) {  // ... or some row's window start
        const int lim = lo_r - key0;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * c + e < lim) s[c][e] = __float_as_uint(-INFINITY);
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < 128; i += 8)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mx[k] = max3(mx[k], __uint_as_float(s[i >> 5][(i & 31) + 2 * k]), __uint_as_float(s[i >> 5][(i & 31) + 2 * k + 1]));
      const float tmax = cf * max3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
      m_true = fmaxf(m_true, tmax);

      // The reference left by tile j-1, then this tile's, handed to tile j+1.
      // Rows are handed over warp to warp: the warps of both groups that
      // cover the same 32 rows share barrier mref_bar[warp & 3][parity].
      float m_prev = m_ref;
      if (j >= 1) {
        mbar_wait_bounded(&sm.mref_bar[warp & 3][(j - 1) & 1], (unsigned)(((j - 1) >> 1) & 1), a.status, &sm.abort);
        m_prev = sm.mref[(j - 1) & 1][r];
      }
      const float m_new = (tmax > m_prev + kRescaleThreshold) ? tmax : m_prev;  // also for the first finite tile max
      if (j + 1 < nt) {
        sm.mref[j & 1][r] = m_new;
        mbar_arrive(&sm.mref_bar[warp & 3][j & 1]);
      }
      const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;

      // P = 2^(S - m) as bf16 pairs: chunk c's 32 values are packed in
      // place into s[c], then stored at column 16 c of P_b once P V of tile
      // j - 2 (the last reader of P_b) has completed.  The row sum is taken
      // in fp32.
      float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float x0 = __uint_as_float(s[c][e]), x1 = __uint_as_float(s[c][e + 1]);
          fma2(x0, x1, cf, cf, neg_m, neg_m);
          const float p0 = ex2(x0), p1 = ex2(x1);
          const int k = (e >> 1) & 3;
          add2(sum[2 * k], sum[2 * k + 1], p0, p1);
          s[c][e >> 1] = tc::pack_bf16(p0, p1);
        }
      }
      if (j >= kSBuf) {
        mbar_wait_bounded(&sm.pv_done[j & 1], (unsigned)(((j - 2) >> 1) & 1), a.status, &sm.abort);
        tc::fence_after_sync();
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_st16(tmem + lane_base + kColP + 64 * b + 16 * c, s[c]);
      const float tsum = ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
      // This group's sum moves to the new reference (m_ref = -inf: l is 0, the factor 0).
      l = l * ((m_new != m_ref) ? ex2(m_ref - m_new) : 1.f) + tsum;
      m_ref = m_new;

      // O holds tiles 0..j-1 against m_prev once P V of tile j-1 has landed;
      // P V of tile j waits for p_ready.  Rescale the row's O when any row of
      // the warp moved its reference at this tile.
      if (j >= 1 && __any_sync(0xffffffffu, m_new != m_prev)) {
        const float corr = (m_new != m_prev) ? ex2(m_prev - m_new) : 1.f;  // m_prev = -inf gives 0
        mbar_wait_bounded(&sm.pv_done[(j - 1) & 1], (unsigned)(((j - 1) >> 1) & 1), a.status, &sm.abort);
        tc::fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(o_col + 32 * c, o);
          tc::tmem_ld_wait();
          tc::reg_fence(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
          tc::tmem_st32(o_col + 32 * c, o);
        }
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_ready[b]);
    }

    // Epilogue: out = O / l, lse = (max, log sum).  The row's reference is
    // the larger of the two groups' last ones (it only grows along the
    // chain); each group's sum is moved onto it.
    sm.red_l[grp][r] = l;
    sm.red_m[grp][r] = m_ref;
    sm.red_t[grp][r] = m_true;
    if (nt > 0) mbar_wait_bounded(&sm.o_final, 0, a.status, &sm.abort);
    tc::fence_before_sync();
    named_barrier(1, kSoftmaxThreads);
    tc::fence_after_sync();
    const float m_fin = fmaxf(sm.red_m[0][r], sm.red_m[1][r]);
    float l_row = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k)
      if (sm.red_l[k][r] > 0.f) l_row += sm.red_l[k][r] * ex2(sm.red_m[k][r] - m_fin);
    m_true = fmaxf(sm.red_t[0][r], sm.red_t[1][r]);
    m_ref = m_fin;
    const float inv = (l_row == 0.f) ? 0.f : 1.f / l_row;
    // O / l leaves by TMA tensor stores.  Each group stages its D/2 columns in
    // the (now idle) K/V ring as 32-float chunks of 128 rows x 128 bytes, in
    // the order of a 3-D box {32 floats, gs heads, 128/gs queries} (row r =
    // query r / gs, head r % gs of the block) with the 128-byte swizzle
    // (16-byte unit u of row r at u ^ (r & 7)); one thread then stores every
    // chunk with one box each.  Rows past n_q fall outside the tensor and are
    // not written, nor are the idle rows past (128/gs)*gs.
    constexpr int kHalfD = D / 2;          // O columns per group
    constexpr int kOChunks = kHalfD / 32;  // 32-float chunks per group
    unsigned char* const ostage = ring;   // [group][chunk][128 rows][128 bytes]
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the ring was last written by TMA
#pragma unroll
    for (int c = 0; c < kOChunks; ++c) {
      uint32_t o[32];
      if (nt > 0) {
        tc::tmem_ld32(o_col + grp * kHalfD + 32 * c, o);
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
  // Rows of K/V any CTA may read: the largest window of the call.  Rows past
  // it are outside the tensor maps and arrive as zeros.
  long long kv_rows = a.causal ? a.base_pos + a.n_q : a.n_all;
  if (kv_rows > a.cap) kv_rows = a.cap;
  const bool no_keys = kv_rows < 1 || a.k == nullptr || a.v == nullptr;
  if (kv_rows < 1) kv_rows = 1;
  void* scratch = nullptr;
  const void* kp = a.q;  // an empty key set never reads K/V: any aligned base will do
  const void* vp = a.q;
  const float* kfac = nullptr;
  if (!no_keys) {
    // K as fp16 with one power of two per (tile, kv head), V as bf16, in
    // stream-ordered scratch memory (library pool), released on the same
    // stream once the attention kernel has run.  Only tiles from the first
    // one any CTA reads are converted (under a sliding window the earlier
    // rows are never read).
    const long long elems = kv_rows * a.kv_row_stride;
    const int n_tiles = (int)((kv_rows + kKeys - 1) / kKeys);
    const int n_first = a.causal ? (int)min((long long)a.cap, a.base_pos + 1) : a.n_all;  // window of query 0
    const int tile0 = first_key(n_first, a.window) / kKeys;
    const size_t fac_off = scratch_round((size_t)elems * 4);
    if (scratch_alloc(&scratch, flash_bf16_scratch_bytes(a), s) != cudaSuccess) return ATTN_ERR_CUDA;
    uint16_t* k16 = static_cast<uint16_t*>(scratch);
    uint16_t* v16 = k16 + elems;
    float* fac = reinterpret_cast<float*>(static_cast<char*>(scratch) + fac_off);
    PrepArgs pa{};
    pa.k = a.k;
    pa.v = a.v;
    pa.out0 = k16;
    pa.out1 = v16;
    pa.kfac = fac;
    pa.stride = a.kv_row_stride;
    pa.G = a.G;
    pa.D = D;
    pa.tile0 = tile0;
    pa.n_tiles = n_tiles;
    pa.rows_end = kv_rows;
    pa.rope = a.rope;
    pa.table = a.block_table;
    pa.page_rows = a.page_rows;
    pa.num_pages = a.num_pages;
    pa.status = a.status;
    const cudaError_t e = launch_kv_prep(pa, s);
    if (e != cudaSuccess) {
      scratch_free(scratch, s);
      return ATTN_ERR_CUDA;
    }
    kp = k16;
    vp = v16;
    kfac = fac;
  }
  CUtensorMap tm_k, tm_v, tm_q, tm_o;
  // Q: fp32 [n_q][H][D] (query rows q_row_stride floats apart); the box is
  // one CTA's block, D x gs heads x 128/gs queries; rows past n_q read as 0.
  const uint64_t qdims[3] = {(uint64_t)D, (uint64_t)a.H, (uint64_t)a.n_q};
  const uint64_t qstrides[2] = {(uint64_t)D * 4, (uint64_t)a.q_row_stride * 4};
  const uint32_t qbox[3] = {(uint32_t)D, (uint32_t)gs, (uint32_t)qpb};
  // out: [n_q][H][D] (query rows out_row_stride floats apart), stored in
  // boxes of 32 floats x gs heads x 128/gs queries.
  const uint64_t odims[3] = {(uint64_t)D, (uint64_t)a.H, (uint64_t)a.n_q};
  const uint64_t ostrides[2] = {(uint64_t)D * 4, (uint64_t)a.out_row_stride * 4};
  const uint32_t obox[3] = {32, (uint32_t)gs, (uint32_t)qpb};
  // K and V: [kv_rows][kv_row_stride] 16-bit, boxes of 64 elements x 128 keys.
  const uint64_t dims[2] = {(uint64_t)a.kv_row_stride, (uint64_t)kv_rows};
  const uint64_t strides[1] = {(uint64_t)a.kv_row_stride * 2};
  const uint32_t box[2] = {64, (uint32_t)kKeys};
  const bool maps_ok = make_tmap(&tm_k, kp, 2, dims, strides, box, true, kSwizzle128) &&
                       make_tmap(&tm_v, vp, 2, dims, strides, box, true, kSwizzle128) &&
                       make_tmap(&tm_q, a.q, 3, qdims, qstrides, qbox, false, kSwizzleNone) &&
                       make_tmap(&tm_o, a.out, 3, odims, ostrides, obox, false, kSwizzle128);
  int rc = ATTN_OK;
  if (!maps_ok) {
    rc = ATTN_ERR_UNSUPPORTED;
  } else {
    const size_t smem = sizeof(Bf16Smem) + 1024;
    auto kern = flash_bf16_kernel<D>;
    if (!set_smem_limit(reinterpret_cast<const void*>(kern), smem)) {
      rc = ATTN_ERR_CUDA;
    } else {
      FlashArgs aa = a;
      int early_q = kfac != nullptr ? 1 : 0;  // the pre-pass ran just before
      int q_ahead = device_sm_count();         // one CTA per SM: about one wave ahead
      void* args[] = {&aa, &tm_k, &tm_v, &tm_q, &tm_o, &kfac, &early_q, &q_ahead};
      if (launch_pdl(reinterpret_cast<const void*>(kern), dim3((unsigned)nb, (unsigned)a.G), dim3(kThreads), smem, s,
                     args) != cudaSuccess)
        rc = ATTN_ERR_CUDA;
    }
  }
  if (scratch != nullptr && scratch_free(scratch, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
  return rc;
}

}  // namespace

// K as fp16 and V as bf16 (kv_rows x kv_row_stride each) and one float per
// (128-key tile, kv head).
size_t flash_bf16_scratch_bytes(const FlashArgs& a) {
  long long kv_rows = a.causal ? a.base_pos + a.n_q : a.n_all;
  if (kv_rows > a.cap) kv_rows = a.cap;
  if (kv_rows < 1 || a.k == nullptr || a.v == nullptr || a.n_q == 0) return 0;
  return scratch_round(scratch_round((size_t)kv_rows * a.kv_row_stride * 4) +
                       (size_t)((kv_rows + kKeys - 1) / kKeys) * a.G * sizeof(float));
}

// Callers check flash_tc_supported(a, ATTN_BF16) first.
int launch_flash_bf16(const FlashArgs& a, cudaStream_t s) {
  return a.D == 128 ? launch_d<128>(a, s) : launch_d<64>(a, s);
}

}  // namespace attn
