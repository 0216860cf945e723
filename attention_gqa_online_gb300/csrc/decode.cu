// decode.cu -- split-KV single-token decode over a KV cache.
//
// Operation: meganeura cached_attention.wgsl, fn main -- one query token,
// H heads, attends to cache positions 0..kv_pos (kv_pos read from device
// memory), or to the last `window` of them under a sliding window.  Decode is bound by streaming the K/V cache from HBM, so the
// design is about bytes, not flops:
//
//   * Grid (S, G'): CTA (j, g) takes one contiguous range of cache positions
//     of a kv head and serves a group of GS query heads that read it (G' = G
//     and GS = gs = H/G up to 4 heads at D = 128, 8 at D = 64; larger groups
//     are split into G' = G * gs/GS head groups whose CTAs read the same K/V
//     rows at about the same time, the second read mostly from L2), so every
//     K/V byte leaves HBM once per call (the shader reads each row once per
//     query head).  S * G is about two CTAs per SM; the range length comes
//     from kv_pos on the device, so the launch does not depend on it.
//   * K and V rows of a stage (32 positions) are staged in shared memory with
//     bulk asynchronous copies (TMA, one 256/512-byte row per copy) that
//     complete on an mbarrier; three stages are in flight per CTA.
//   * Each warp runs its own online softmax (tile max, one correction per
//     stage, running sum and accumulator; the same recurrence as the pages)
//     over its 8 positions of every stage; the 4 warps merge at the end.
//   * Each CTA writes its partial (m, l, unnormalised o) to the workspace; the
//     last CTA of kv head g to finish (atomic ticket) merges the S partials
//     with the log-sum-exp rule: M = max m_j, L = sum l_j 2^(m_j - M),
//     out = sum o_j 2^(m_j - M) / L, and resets the ticket for the next call.
//   * Launched with programmatic dependent launch: a decode step's launch and
//     set-up overlap the previous step's merge tail; nothing touches global
//     memory before the previous kernel has completed.
//
// Scores are kept in the base-2 domain (scale * log2(e) folded into q).
#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

constexpr int kT = 32;                    // positions per stage
constexpr int kStages = 3;                // stages in flight
constexpr int kCWarps = 4;                // consumer warps
constexpr int kThreads = 32 * (kCWarps + 1);  // + one producer warp
constexpr int kCtasPerSm = 2;
constexpr int kMinChunk = 64;             // fewest positions a split is given
constexpr int kMaxSplits = 1024;          // most splits per kv head
constexpr int kMergeBatch = 16;           // splits merged per batch of loads
constexpr int kPrefetchStages = 4;        // stages per CTA pulled into L2 before the launch wait
constexpr int kPpw = kT / kCWarps;        // positions per consumer warp per stage
constexpr int kNg = kPpw / 4;             // groups of four positions per warp
static_assert(kPpw % 4 == 0, "each consumer warp takes whole groups of four positions");

template <int D, int GS>
struct __align__(128) DecodeSmem {
  float k[kStages][kT * D];
  float v[kStages][kT * D];
  float red_m[kCWarps][GS];
  float red_l[kCWarps][GS];
  float red_o[kCWarps][GS][D];
  float wts[kCWarps][kNg * 4 + 1][GS];  // per warp: P of its positions for every head, then the corrections
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t merge_bar[GS];  // per head of the round: its partials have landed
  int is_last;
  int abort;
};

struct WsLayout {
  unsigned* tickets;  // [G]
  float* ml;          // [H][S][2]
  float* o;           // [H][S][D]
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// (m, l) pairs of one head are kEvenS(S) pairs apart, so every head's pairs
// start on a 16-byte boundary (the final merge bulk-copies them).
__host__ __device__ inline int even_splits(int S) { return (S + 1) & ~1; }

__host__ __device__ inline WsLayout ws_layout(void* ws, int H, int G, int D, int S) {
  char* p = static_cast<char*>(ws);
  WsLayout l;
  l.tickets = reinterpret_cast<unsigned*>(p);
  p += align256(sizeof(unsigned) * G);
  l.ml = reinterpret_cast<float*>(p);
  p += align256(sizeof(float) * 2 * (size_t)H * even_splits(S));
  l.o = reinterpret_cast<float*>(p);
  return l;
}

// Positions [p_begin, p_end) of split j of kv head g, out of S splits, for a
// cache position kv_pos; s_eff = splits that get any position.  Positions
// [lo, end) are attended.  Splits cover [lo rounded down to a stage, end) and
// start on absolute stage boundaries, so no stage is read by two CTAs and no
// stage crosses a page of a paged cache; positions below lo are masked.
struct SplitRange {
  int p_begin, p_end, s_eff, lo;
};
__device__ __forceinline__ SplitRange split_range(unsigned kp, int max_seq, int window, int S, int j) {
  const long long n_ll = (long long)kp + 1 < (long long)max_seq ? (long long)kp + 1 : (long long)max_seq;
  const int lo = first_key((int)n_ll, window);
  const int base = lo / kT * kT;
  const int n = (int)n_ll - base;
  const int s0 = min(S, (n + kMinChunk - 1) / kMinChunk);
  const int chunk = ((n + s0 - 1) / s0 + kT - 1) / kT * kT;
  SplitRange r;
  r.s_eff = (n + chunk - 1) / chunk;
  r.p_begin = base + min(n, j * chunk);
  r.p_end = base + min(n, j * chunk + chunk);
  r.lo = lo;
  return r;
}

// Cache row of position t: t itself, or its pool row through the block table
// (a page outside the pool gives a row past the pool: zeros, and the status
// word records ATTN_ERR_INVALID_ARG unless `hint`).
__device__ __forceinline__ int cache_row(const DecodeArgs& a, int t, bool hint) {
  if (a.block_table == nullptr) return t;
  const uint32_t page = a.block_table[t / a.page_rows];
  if (page < (uint32_t)a.num_pages) return (int)page * a.page_rows + t % a.page_rows;
  if (!hint) record_status(a.status, ATTN_ERR_INVALID_ARG);
  return a.num_pages * a.page_rows;
}

// Warp roles: warps 0..3 consume, warp 4 issues the bulk copies.  Consumer
// warp w owns positions 4w..4w+3 of every stage; within it lane = 8p + c
// takes position p and dims {4c + 32u : u < D/32} (float4 each), so each
// 8-lane phase of a 16-byte shared load reads one contiguous row.
template <int D, int GS>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    decode_split_kernel(const DecodeArgs a, const int S, const float sl2, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v) {
  using Smem = DecodeSmem<D, GS>;
  constexpr int U = D / 32;   // float4 groups per lane in the score phase
  constexpr int VP = D / 32;  // output dims per lane in the PV phase
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Grid (S * kv_div, G): the kv_div head groups of one split are adjacent
  // CTAs, so they stream the same K/V rows at about the same time.
  const int j = blockIdx.x / a.kv_div;                  // split
  const int kvh = blockIdx.y;                           // kv head
  const int g = kvh * a.kv_div + blockIdx.x % a.kv_div;  // head group (query heads g*GS ..)

  // Launched with programmatic serialization: let the next decode start
  // launching now.  While the previous kernel in the stream drains, the
  // producer thread pulls this CTA's first stages into L2, steered by a read
  // of kv_pos that may predate the previous kernel's writes: these are only
  // hints (a wrong range costs bandwidth, never a result), and nothing read
  // before the wait below is used afterwards.
  allow_dependent_launch();
  if (tid == 32 * kCWarps) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    const unsigned kp_hint = *static_cast<const volatile uint32_t*>(a.kv_pos_dev);
    const SplitRange h = split_range(kp_hint, a.max_seq, a.window, S, j);
    // Twice as deep when one CTA serves all the query heads of its kv head;
    // with several head groups, whose CTAs hint the same rows, only the first
    // two stages.
    const int n_pf = a.kv_div == 1 ? 2 * kPrefetchStages : 2;
    for (int st = 0; st < n_pf && j < h.s_eff && h.p_begin + st * kT < h.p_end; ++st) {
      const int row = cache_row(a, h.p_begin + st * kT, true);
      tma_prefetch_l2_2d(&tm_k, kvh * D, row);
      tma_prefetch_l2_2d(&tm_v, kvh * D, row);
    }
  }
  grid_dependency_wait();
  const unsigned kp = *a.kv_pos_dev;
  if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0 && (long long)kp >= (long long)a.max_seq)
    record_status(a.status, ATTN_ERR_INVALID_ARG);
  const SplitRange range = split_range(kp, a.max_seq, a.window, S, j);
  const int s_eff = range.s_eff;
  if (j >= s_eff) return;
  const int p_begin = range.p_begin;
  const int p_end = range.p_end;
  const int lo = range.lo;
  const int len = p_end - p_begin;
  const int n_st = (len + kT - 1) / kT;

  // Append: the split that ends at kv_pos first writes the new token's K and
  // V row of its kv head into cache row kv_pos (only the CTAs of that split
  // read the row; head groups of one kv head write the same values), then
  // makes the writes visible to its own bulk copies.
  if (a.k_new != nullptr && j == s_eff - 1 && (long long)kp < (long long)a.max_seq) {
    const long long row = cache_row(a, (int)kp, false);
    if (row < (long long)a.num_pages * a.page_rows || a.block_table == nullptr) {
      const long long off = row * a.G * D + (long long)kvh * D;
      for (int d = 4 * tid; d < D; d += 4 * kThreads) {
        *reinterpret_cast<float4*>(const_cast<float*>(a.k_cache) + off + d) =
            *reinterpret_cast<const float4*>(a.k_new + (long long)kvh * D + d);
        *reinterpret_cast<float4*>(const_cast<float*>(a.v_cache) + off + d) =
            *reinterpret_cast<const float4*>(a.v_new + (long long)kvh * D + d);
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kCWarps);
    }
    for (int h = 0; h < GS; ++h) mbar_init(&sm.merge_bar[h], 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  float acc[GS][VP];
#pragma unroll
  for (int h = 0; h < GS; ++h)
#pragma unroll
    for (int e = 0; e < VP; ++e) acc[h][e] = 0.f;

  if (warp == kCWarps) {
    // ---------------- producer: one [kT x D] tile of K and of V per stage
    if (lane == 0) {
      for (int st = 0; st < n_st; ++st) {
        const int slot = st % kStages;
        if (st >= kStages) mbar_wait_bounded(&sm.empty[slot], ((st / kStages) - 1) & 1, a.status, &sm.abort);
        const int row = cache_row(a, p_begin + st * kT, false);
        mbar_arrive_expect_tx(&sm.full[slot], (unsigned)(kT * D * 4 * 2));
        tma_load_2d(&sm.k[slot][0], &tm_k, kvh * D, row, &sm.full[slot]);
        tma_load_2d(&sm.v[slot][0], &tm_v, kvh * D, row, &sm.full[slot]);
      }
      // No copy may still be landing when the CTA exits (normally all were
      // consumed already, so these return at once).
      for (int s = 0; s < kStages && s < n_st; ++s) {
        const int last = s + ((n_st - 1 - s) / kStages) * kStages;
        mbar_wait_bounded(&sm.full[s], (unsigned)((last / kStages) & 1), a.status);
      }
    }
    __syncwarp();
  } else {
    // ---------------- consumers
    const int qp = lane >> 3, qc = lane & 7;
    float4 qr[GS][U];
#pragma unroll
    for (int h = 0; h < GS; ++h)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float4 x = *reinterpret_cast<const float4*>(a.q + (size_t)(g * GS + h) * D + 4 * qc + 32 * u);
        qr[h][u] = make_float4(x.x * sl2, x.y * sl2, x.z * sl2, x.w * sl2);
      }
    // The eight lanes of a position reduce their GS partial dot products by
    // recursive halving: at each level a lane keeps half of its heads and
    // adds its partner's values for them, so after three levels it holds the
    // full score of one head, h_own (lanes 8p + c, 8p + c' with equal h_own
    // hold the same value).  The online softmax state of h_own lives in the
    // lane; the weights and corrections every lane needs for P V go through
    // the warp's slot of sm.wts.
    int h_own = 0;
    {
      int n = GS;
#pragma unroll
      for (int o = 4; o >= 1; o >>= 1)
        if (n > 1) {
          n >>= 1;
          if (qc & o) h_own += n;
        }
    }
    float m_own = -INFINITY, l_own = 0.f;
    // One writer per (position, head): the lowest lane c of each head.
    const bool writer = ((qc & ((8 / (GS < 8 ? GS : 8)) - 1)) == 0);
    float(*wts)[GS] = sm.wts[warp];
    for (int st = 0; st < n_st; ++st) {
      const int slot = st % kStages;
      mbar_wait_bounded(&sm.full[slot], (st / kStages) & 1, a.status, &sm.abort);
      const int valid = min(kT, p_end - (p_begin + st * kT));
      const int first = lo - (p_begin + st * kT);  // positions below this one are outside the window
      const float* ks = sm.k[slot];
      const float* vs = sm.v[slot];

      // Scores of this warp's kNg groups of four positions, head h_own.
      float sc[kNg];
#pragma unroll
      for (int grp = 0; grp < kNg; ++grp) {
        const int pos = kPpw * warp + 4 * grp + qp;
        float part[GS];
#pragma unroll
        for (int h = 0; h < GS; ++h) part[h] = 0.f;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float4 kv = *reinterpret_cast<const float4*>(&ks[pos * D + 4 * qc + 32 * u]);
          if constexpr (GS % 2 == 0) {
            // Two heads per paired fma: the same per-head order of products.
#pragma unroll
            for (int h = 0; h < GS; h += 2) {
              fma2_acc(part[h], part[h + 1], qr[h][u].x, qr[h + 1][u].x, kv.x, kv.x);
              fma2_acc(part[h], part[h + 1], qr[h][u].y, qr[h + 1][u].y, kv.y, kv.y);
              fma2_acc(part[h], part[h + 1], qr[h][u].z, qr[h + 1][u].z, kv.z, kv.z);
              fma2_acc(part[h], part[h + 1], qr[h][u].w, qr[h + 1][u].w, kv.w, kv.w);
            }
          } else {
#pragma unroll
            for (int h = 0; h < GS; ++h) {
              part[h] = fmaf(qr[h][u].x, kv.x, part[h]);
              part[h] = fmaf(qr[h][u].y, kv.y, part[h]);
              part[h] = fmaf(qr[h][u].z, kv.z, part[h]);
              part[h] = fmaf(qr[h][u].w, kv.w, part[h]);
            }
          }
        }
        int n = GS;
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) {
          if (n > 1) {
            const int half = n >> 1;
            const bool upper = (qc & o) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
              const float keep = upper ? part[half + i] : part[i];
              const float send = upper ? part[i] : part[half + i];
              part[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
            n = half;
          } else {
            part[0] += __shfl_xor_sync(0xffffffffu, part[0], o);
          }
        }
        sc[grp] = (pos < valid && pos >= first) ? part[0] : -INFINITY;
      }

      // Online softmax of head h_own over the warp's kPpw positions.
      float mx = sc[0];
#pragma unroll
      for (int grp = 1; grp < kNg; ++grp) mx = fmaxf(mx, sc[grp]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m_own, mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = ex2(m_own - m_use);
      float sum = 0.f;
#pragma unroll
      for (int grp = 0; grp < kNg; ++grp) {
        const float w = ex2(sc[grp] - m_use);
        sum += w;
        if (writer) wts[4 * grp + qp][h_own] = w;
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 8);
      sum += __shfl_xor_sync(0xffffffffu, sum, 16);
      l_own = l_own * corr + sum;
      m_own = m_new;
      if (writer && qp == 0) wts[kNg * 4][h_own] = corr;
      __syncwarp();

      // acc = acc * corr + w * V over the warp's positions; lane owns dims VP*lane ..
      auto row = [&](int i, float* out) {
        if constexpr (GS % 4 == 0) {
#pragma unroll
          for (int h = 0; h < GS; h += 4) {
            const float4 x = *reinterpret_cast<const float4*>(&wts[i][h]);
            out[h] = x.x; out[h + 1] = x.y; out[h + 2] = x.z; out[h + 3] = x.w;
          }
        } else if constexpr (GS == 2) {
          const float2 x = *reinterpret_cast<const float2*>(&wts[i][0]);
          out[0] = x.x; out[1] = x.y;
        } else {
          out[0] = wts[i][0];
        }
      };
      {
        float cb[GS];
        row(kNg * 4, cb);
#pragma unroll
        for (int h = 0; h < GS; ++h)
#pragma unroll
          for (int e = 0; e < VP; ++e) acc[h][e] *= cb[h];
      }
      // One position's weights times its V row; two output dims per paired fma.
      auto pv = [&](int i) {
        const int ppos = kPpw * warp + i;
        float wb[GS];
        row(i, wb);
        if constexpr (VP == 4) {
          const float4 vv = *reinterpret_cast<const float4*>(&vs[ppos * D + 4 * lane]);
#pragma unroll
          for (int h = 0; h < GS; ++h) {
            fma2_acc(acc[h][0], acc[h][1], wb[h], wb[h], vv.x, vv.y);
            fma2_acc(acc[h][2], acc[h][3], wb[h], wb[h], vv.z, vv.w);
          }
        } else {
          const float2 vv = *reinterpret_cast<const float2*>(&vs[ppos * D + 2 * lane]);
#pragma unroll
          for (int h = 0; h < GS; ++h) fma2_acc(acc[h][0], acc[h][1], wb[h], wb[h], vv.x, vv.y);
        }
      };
      if (valid == kT && first <= 0) {
        // Every position of the stage is kept (all but a split's last stage
        // and a window's first): no per-position test, so the loads of
        // several positions can be in flight together.
#pragma unroll
        for (int i = 0; i < kNg * 4; ++i) pv(i);
      } else {
        // Skipped positions may hold any bits (a cache row past kv_pos), so
        // they are left out rather than weighted by zero.
#pragma unroll
        for (int i = 0; i < kNg * 4; ++i) {
          const int ppos = kPpw * warp + i;
          if (ppos < valid && ppos >= first) pv(i);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }

    if (writer && qp == 0) {
      sm.red_m[warp][h_own] = m_own;
      sm.red_l[warp][h_own] = l_own;
    }
#pragma unroll
    for (int h = 0; h < GS; ++h)
#pragma unroll
      for (int e = 0; e < VP; ++e) sm.red_o[warp][h][VP * lane + e] = acc[h][e];
  }
  __syncthreads();

  // Merge the consumer warps' states into this split's partial.
  auto cta_state = [&](int h, int d, float& M, float& L, float& O) {
    M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < kCWarps; ++w2) M = fmaxf(M, sm.red_m[w2][h]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    L = 0.f;
    O = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kCWarps; ++w2) {
      const float f = ex2(sm.red_m[w2][h] - Mu);
      L += sm.red_l[w2][h] * f;
      O += sm.red_o[w2][h][d] * f;
    }
  };
  if (s_eff == 1) {
    // The only split: its state is the result (merging one partial would
    // reproduce it), so no partial, no ticket.
    for (int idx = tid; idx < GS * D; idx += kThreads) {
      const int h = idx / D, d = idx % D;
      float M, L, O;
      cta_state(h, d, M, L, O);
      const float inv = (L == 0.f) ? 0.f : 1.f / L;
      a.out[(size_t)(g * GS + h) * D + d] = O * inv;
    }
    return;
  }
  const WsLayout ws = ws_layout(a.workspace, a.H, a.G * a.kv_div, D, S);
  for (int idx = tid; idx < GS * D; idx += kThreads) {
    const int h = idx / D, d = idx % D;
    float M, L, O;
    cta_state(h, d, M, L, O);
    const size_t hs = (size_t)(g * GS + h) * S + j;
    ws.o[hs * D + d] = O;
    if (d == 0) {
      const size_t ms = ((size_t)(g * GS + h) * even_splits(S) + j) * 2;
      ws.ml[ms] = M;
      ws.ml[ms + 1] = L;
    }
  }

  // The last split of this kv head to finish merges all of them.  One
  // thread takes the ticket with an acquire-release atomic: the release
  // orders the CTA's partial (written by all its threads, ordered before it
  // by the barrier) before the ticket, and in the last CTA the acquire (with
  // the barrier after it) orders the other splits' partials before the
  // merge's reads.
  __syncthreads();
  if (tid == 0) {
    unsigned prev;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(prev) : "l"(&ws.tickets[g]) : "memory");
    sm.is_last = (prev == (unsigned)(s_eff - 1));
  }
  __syncthreads();
  if (!sm.is_last) return;

  // Fast path: the splits' partials of as many heads as fit in the (now
  // idle) stage buffers come in with one round of bulk copies, then the merge
  // runs from shared memory; rounds repeat until every head is merged.  Each
  // head's copies complete on its own barrier, so the threads of a head
  // merge as soon as its partials have landed.
  const int S2 = even_splits(S);
  const unsigned ml_head_bytes = ((unsigned)s_eff * 8u + 15u) & ~15u;
  const size_t head_bytes = (size_t)s_eff * D * 4 + ml_head_bytes;
  const int hr = (int)min((size_t)GS, (sizeof(sm.k) + sizeof(sm.v)) / head_bytes);  // heads per round
  if (hr > 0) {
    for (int h0 = 0, round = 0; h0 < GS; h0 += hr, ++round) {
      const int nh = min(hr, GS - h0);
      float* so = &sm.k[0][0];                  // [nh][s_eff][D]
      float* sml = so + (size_t)nh * s_eff * D;  // [nh][ml_head_bytes / 4]
      if (tid == 0) {
        asm volatile("fence.proxy.async;" ::: "memory");
        for (int h = 0; h < nh; ++h) {
          mbar_arrive_expect_tx(&sm.merge_bar[h], (unsigned)head_bytes);
          bulk_g2s(so + (size_t)h * s_eff * D, ws.o + (size_t)(g * GS + h0 + h) * S * D, (unsigned)(s_eff * D * 4),
                   &sm.merge_bar[h]);
          bulk_g2s(sml + (size_t)h * (ml_head_bytes / 4), ws.ml + (size_t)(g * GS + h0 + h) * S2 * 2, ml_head_bytes,
                   &sm.merge_bar[h]);
        }
      }
      for (int idx = tid; idx < nh * (D / 4); idx += kThreads) {
        const int h = idx / (D / 4), c = idx % (D / 4);
        mbar_wait_bounded(&sm.merge_bar[h], (unsigned)(round & 1), a.status);
        const float* mlh = sml + (size_t)h * (ml_head_bytes / 4);
        float M = -INFINITY;
        for (int s = 0; s < s_eff; ++s) M = fmaxf(M, mlh[2 * s]);
        const float Mu = (M == -INFINITY) ? 0.f : M;
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int s = 0; s < s_eff; ++s) {
          const float f = ex2(mlh[2 * s] - Mu);
          const float4 x = *reinterpret_cast<const float4*>(so + ((size_t)h * s_eff + s) * D + 4 * c);
          L = fmaf(mlh[2 * s + 1], f, L);
          fma2_acc(O.x, O.y, x.x, x.y, f, f);
          fma2_acc(O.z, O.w, x.z, x.w, f, f);
        }
        const float inv = (L == 0.f) ? 0.f : 1.f / L;
        *reinterpret_cast<float4*>(a.out + (size_t)(g * GS + h0 + h) * D + 4 * c) =
            make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
      }
      __syncthreads();  // the buffers are refilled by the next round
    }
    if (tid == 0) ws.tickets[g] = 0u;
    return;
  }

  // One pass over the splits with the same online rule (running max,
  // correction, sum), 16 splits' loads in flight at a time; one float4 of
  // one head per thread.
  for (int idx = tid; idx < GS * (D / 4); idx += kThreads) {
    const int h = idx / (D / 4), c = idx % (D / 4);
    const size_t hb = (size_t)(g * GS + h) * S;
    const float* op = ws.o + hb * D + 4 * c;
    const float2* mlp = reinterpret_cast<const float2*>(ws.ml + (size_t)(g * GS + h) * S2 * 2);
    float M = -INFINITY, L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < s_eff; s0 += kMergeBatch) {
      float2 ml[kMergeBatch];
      float4 ov[kMergeBatch];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        if (s0 + u < s_eff) {
          ml[u] = __ldcg(mlp + s0 + u);
          ov[u] = __ldcg(reinterpret_cast<const float4*>(op + (size_t)(s0 + u) * D));
        } else {
          ml[u] = make_float2(-INFINITY, 0.f);
          ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float m_new = M;
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) m_new = fmaxf(m_new, ml[u].x);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = ex2(M - m_use);
      L *= corr;
      O.x *= corr;
      O.y *= corr;
      O.z *= corr;
      O.w *= corr;
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const float f = ex2(ml[u].x - m_use);
        L = fmaf(ml[u].y, f, L);
        O.x = fmaf(ov[u].x, f, O.x);
        O.y = fmaf(ov[u].y, f, O.y);
        O.z = fmaf(ov[u].z, f, O.z);
        O.w = fmaf(ov[u].w, f, O.w);
      }
      M = m_new;
    }
    const float inv = (L == 0.f) ? 0.f : 1.f / L;
    *reinterpret_cast<float4*>(a.out + (size_t)(g * GS + h) * D + 4 * c) =
        make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
  }
  if (tid == 0) ws.tickets[g] = 0u;
}

template <int D, int GS>
int launch_t(const DecodeArgs& a, int S, cudaStream_t s) {
  const size_t smem = sizeof(DecodeSmem<D, GS>);
  auto kern = decode_split_kernel<D, GS>;
  if (!set_smem_limit(reinterpret_cast<const void*>(kern), smem)) return ATTN_ERR_CUDA;
  // K and V caches as 2-D tensors [max_seq rows][G*D floats]; one request
  // copies kT rows of one kv head's D columns.
  CUtensorMap tm_k, tm_v;
  // (A paged cache: the whole pool.)
  const uint64_t rows = a.block_table != nullptr ? (uint64_t)a.num_pages * a.page_rows : (uint64_t)a.max_seq;
  const uint64_t dims[2] = {(uint64_t)a.G * D, rows};
  const uint64_t strides[1] = {(uint64_t)a.G * D * 4};
  const uint32_t box[2] = {(uint32_t)D, (uint32_t)kT};
  if (!make_tmap(&tm_k, a.k_cache, 2, dims, strides, box, false, kSwizzleNone) ||
      !make_tmap(&tm_v, a.v_cache, 2, dims, strides, box, false, kSwizzleNone))
    return ATTN_ERR_UNSUPPORTED;
  const float sl2 = (1.0f / sqrtf((float)D)) * kLog2e;
  DecodeArgs aa = a;
  int SS = S;
  float sl = sl2;
  void* args[] = {&aa, &SS, &sl, &tm_k, &tm_v};
  return launch_pdl(reinterpret_cast<const void*>(kern), dim3(S * a.kv_div, a.G), dim3(kThreads), smem, s, args) == cudaSuccess
             ? 0
             : ATTN_ERR_CUDA;
}

__global__ void __launch_bounds__(256) cache_append_kernel(const float* __restrict__ k_new,
                                                           const float* __restrict__ v_new, float* k_cache,
                                                           float* v_cache, const uint32_t* kv_pos_dev, int kv_dim,
                                                           int max_seq, unsigned* status) {
  allow_dependent_launch();
  grid_dependency_wait();
  const unsigned kp = *kv_pos_dev;
  if ((long long)kp >= (long long)max_seq) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_status(status, ATTN_ERR_INVALID_ARG);
    return;
  }
  for (int d = blockIdx.x * 256 + threadIdx.x; d < kv_dim; d += gridDim.x * 256) {
    k_cache[(long long)kp * kv_dim + d] = k_new[d];
    v_cache[(long long)kp * kv_dim + d] = v_new[d];
  }
}

}  // namespace

cudaError_t launch_cache_append(const float* k_new, const float* v_new, float* k_cache, float* v_cache,
                                const uint32_t* kv_pos_dev, int kv_dim, int max_seq, unsigned* status, cudaStream_t s) {
  void* args[] = {&k_new, &v_new, &k_cache, &v_cache, &kv_pos_dev, &kv_dim, &max_seq, &status};
  return launch_pdl(reinterpret_cast<const void*>(cache_append_kernel), dim3((unsigned)((kv_dim + 255) / 256)),
                    dim3(256), 0, s, args);
}

// Query heads per CTA: the group size gs up to 4 (D = 128) or 8 (D = 64);
// larger power-of-two groups split into gs / GS head groups.
int heads_per_cta(int gs, int D) { return min(gs, D == 128 ? 4 : 8); }

bool decode_split_supported(int H, int G, int D) {
  if (G <= 0 || H % G != 0) return false;
  const int gs = H / G;
  if (D != 64 && D != 128) return false;
  return gs >= 1 && gs <= 32 && (gs & (gs - 1)) == 0;
}

int decode_groups(int H, int G, int D) { return G * ((H / G) / heads_per_cta(H / G, D)); }

int decode_splits(int G, int max_seq, int sm_count) {
  const int target = (kCtasPerSm * sm_count + G - 1) / G;
  const int by_len = (max_seq + kMinChunk - 1) / kMinChunk;
  return max(1, min(min(target, by_len), kMaxSplits));
}

size_t decode_workspace_bytes(int H, int G, int D, int max_seq, int sm_count) {
  if (!decode_split_supported(H, G, D) || max_seq <= 0) return 0;
  const int groups = decode_groups(H, G, D);
  const int S = decode_splits(groups, max_seq, sm_count);
  return align256(sizeof(unsigned) * groups) + align256(sizeof(float) * 2 * (size_t)H * even_splits(S)) +
         sizeof(float) * (size_t)H * S * D;
}

size_t decode_ticket_bytes(int G) { return align256(sizeof(unsigned) * G); }

int launch_decode_split(const DecodeArgs& a0, int S, cudaStream_t s) {
  DecodeArgs a = a0;
  const int gs = a.H / a.G, hp = heads_per_cta(gs, a.D);
  a.kv_div = gs / hp;
  if (a.D == 128) {
    if (hp == 1) return launch_t<128, 1>(a, S, s);
    if (hp == 2) return launch_t<128, 2>(a, S, s);
    if (hp == 4) return launch_t<128, 4>(a, S, s);
  } else if (a.D == 64) {
    if (hp == 1) return launch_t<64, 1>(a, S, s);
    if (hp == 2) return launch_t<64, 2>(a, S, s);
    if (hp == 4) return launch_t<64, 4>(a, S, s);
    if (hp == 8) return launch_t<64, 8>(a, S, s);
  }
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
