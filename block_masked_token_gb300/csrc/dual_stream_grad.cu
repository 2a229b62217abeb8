// Gradient of the dual-stream attention under the MARS mask M (papernotes.org notes of
// "MARS: Enabling Autoregressive Models Multi-Token Generation", Key design 1, eq. M; the
// training step of the overall framework runs the backward of this forward).
//
// With P = softmax(scale * S + M), S = Q K^T, and D_i = rowsum(dO_i * O_i):
//   dV = P^T dO,   dP = dO V^T,   dS = P * (dP - D),   dK = scale dS^T Q,   dQ = scale dS K.
// Two tcgen05 kernels, neither storing a score block:
//   - dual_grad_kernel (here): a work item is (batch, query head, 128-key tile of the
//     clean stream), or (batch, kv head, 128-key tile of the masked stream) for all query
//     heads of the kv group (see GItem); one persistent CTA per SM runs items heaviest
//     first. The item visits every 128-row query tile that sees one of its keys under M,
//     and per (key tile, query tile) pair runs four MMAs with TMEM accumulators:
//       S^T = K Q^T, dP^T = V dO^T            (keys on TMEM lanes, queries on columns)
//       dV += P^T dO, dK += dS^T Q            (A = P^T / dS^T from TMEM, bf16 over the
//                                              fp32 columns they were formed from)
//     each in two halves of 64 queries with barriers of their own, so that one half's
//     S^T (or dP^T) of the next pair goes as soon as that half's dV (or dK) has read it.
//     P^T = exp2(scale log2(e) S^T - lse) and dS^T are formed by two threads per key row
//     (64 query columns each: with lse known, no row-wide exchange is needed). One thread
//     issues S^T and dP^T (shared-memory operands), another dV and dK (A from TMEM), on
//     different sub-partitions: one thread alternating the two forms issues them about a
//     quarter slower. S^T of the next pair is issued as soon as dV has read P^T, so it
//     runs under this pair's dK.
//     dK and dV stay in TMEM over the item's pairs and are then added to dK and dV (fp32
//     vector atomics; the G query heads of a kv group add into the same rows).
//   - the dQ kernel (with the forward, whose work items and masks it shares): per query
//     tile, dQ accumulates dS K over the visible key tiles in TMEM and is written once.
// The row statistics (lse: log2 of each query row's softmax denominator) come from a
// statistics-only run of the forward kernel; P and dS are rounded to bf16 as MMA operands.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace mars {

namespace {

using namespace sm100;

constexpr int GT = 128;                // keys per key tile, query rows per query tile
constexpr int MATH_WARPS = 8;          // two per TMEM lane quadrant, 64 query columns each
// warp 0 loads, warp 1 owns TMEM and issues S^T and dP^T, warps 2..9 math, warp 10 issues
// dV and dK
constexpr int GRAD_THREADS = 96 + 32 * MATH_WARPS;
constexpr int GRAD_TS_WARP = 2 + MATH_WARPS;
constexpr int MATH_THREADS = 32 * MATH_WARPS;
constexpr int NSTAGE = 2;              // Q / dO ring depth

// dO (fp32) -> bf16 copy, and D[b][h][stream][t] = sum_d dO[b, i, h, d] * O[b, i, h, d]
// (i = stream * L + t; rows padded to lp per stream). One warp per (b, i, h) row.
__global__ void __launch_bounds__(256) grad_prep_kernel(const float* __restrict__ o,
                                                        const float* __restrict__ d_o,
                                                        __nv_bfloat16* __restrict__ do_bf,
                                                        float* __restrict__ drow,
                                                        long long nrows, int n, int hq, int d,
                                                        int lp) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= nrows) return;
  const float* a = o + row * d;
  const float* g = d_o + row * d;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) {
    const float x = g[c];
    acc += x * a[c];
    do_bf[row * d + c] = __float2bfloat16_rn(x);
  }
  acc = warp_sum(acc);
  const long long h = row % hq, bi = row / hq, i = bi % n, b = bi / n;
  const long long L = n / 2, stream = i / L, t = i % L;
  if (lane == 0) drow[((b * hq + h) * 2 + stream) * lp + t] = acc;
}

template <int D>
struct GSmem {
  static constexpr int T_BYTES = GT * D * 2;                 // one [128][D] bf16 tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = T_BYTES;
  static constexpr int OFF_RING = 2 * T_BYTES;
  // a stage: Q [128][D], dO [128][D], lse and D of its 128 query rows; 1024-byte aligned
  static constexpr int DO_BYTES = T_BYTES;
  static constexpr int ST_Q = 0, ST_DO = T_BYTES, ST_LSE = T_BYTES + DO_BYTES,
                       ST_D = ST_LSE + GT * 4;
  static constexpr int STAGE = (ST_D + GT * 4 + 1023) / 1024 * 1024;
  static constexpr int TOTAL = OFF_RING + NSTAGE * STAGE + 1024;   // + alignment slack
  // TMEM columns
  static constexpr int TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D, TM_COLS = 512;
};

struct GBar {
  uint64_t kv_full, kv_empty;
  uint64_t full[NSTAGE], empty[NSTAGE];
  // per 64-query half of a pair: its S^T and dP^T MMAs, P^T and dS^T, its dV and dK MMAs
  uint64_t s_full[2], dp_full[2], p_full[2], ds_full[2], dv_done[2], dk_done[2];
  uint64_t acc_full, acc_free, drain, drain_ts;
  uint32_t tmem_base;
  int abort;
};

struct GArgs {
  int batch, L, B, hq, hkv, G, nt;
  float scale, scale_log2;
  const float* lse;        // [batch][hq][2][Lp], Lp = 128 nt (pad rows zero)
  const float* drow;       // same layout
  float* dk;               // [batch][2L][hkv][D]
  float* dv;
  int32_t* status;
};

// Work item: keys [128 jt, 128 jt + 128) of stream ks (0 clean, 1 masked) of (b, kvh),
// against query heads kvh*G + g, g in [g0, g0 + ng). A clean key tile is one item per query
// head. A masked key tile is seen only by the query tiles of its own block (one or two when
// B <= 128); there one item takes all G heads of the kv group, so that its K and V are
// loaded, and its dK and dV drained, once for the group instead of once per head. Ids run
// over the clean key tiles from the first (seen by most query tiles) to the last, then over
// the masked key tiles.
struct GItem {
  int b, kvh, g0, ng, ks, jt;
  int nc, mlo;             // per head: clean query tiles [jt, nt), masked [mlo, nt)
  int np1, npg;            // pairs per head, pairs of the item (ng * np1)
};

__host__ __device__ inline bool grad_group_masked(int B) { return B <= GT; }

__host__ __device__ inline long long grad_item_count(int batch, int hkv, int G, int nt, int B) {
  const long long per = (long long)batch * hkv * G;
  return per * nt + (grad_group_masked(B) ? (long long)batch * hkv : per) * nt;
}

MARS_DEV GItem grad_item(const GArgs& a, int id) {
  GItem it;
  const int per = a.batch * a.hkv * a.G;
  int kt, bk;
  if (id < a.nt * per) {
    kt = id / per;
    bk = id % per;
    it.g0 = bk % a.G;
    it.ng = 1;
    bk /= a.G;
  } else if (grad_group_masked(a.B)) {
    const int r = id - a.nt * per, pm = a.batch * a.hkv;
    kt = a.nt + r / pm;
    bk = r % pm;
    it.g0 = 0;
    it.ng = a.G;
  } else {
    const int r = id - a.nt * per;
    kt = a.nt + r / per;
    bk = r % per;
    it.g0 = bk % a.G;
    it.ng = 1;
    bk /= a.G;
  }
  it.b = bk % a.batch;
  it.kvh = bk / a.batch;
  if (kt < a.nt) {
    it.ks = 0;
    it.jt = kt;
    it.nc = a.nt - kt;
    // masked row t sees clean key k iff its block start (t/B)*B > k: t >= (k/B + 1) B
    const int tmin = (GT * kt / a.B + 1) * a.B;
    it.mlo = tmin <= a.L - 1 ? tmin / GT : a.nt;
    it.np1 = it.nc + (a.nt - it.mlo);
  } else {
    it.ks = 1;
    it.jt = kt - a.nt;
    // masked key u is seen by masked rows t in [u, end of u's block)
    const int umax = min(GT * it.jt + GT - 1, a.L - 1);
    const int tmax = min(a.L, (umax / a.B + 1) * a.B) - 1;
    it.nc = 0;
    it.mlo = it.jt;
    it.np1 = tmax / GT - it.jt + 1;
  }
  it.npg = it.ng * it.np1;
  return it;
}

// Pair p of an item: query head kvh*G + g, query stream qs, query tile qi.
struct GPair {
  int g, qs, qi;
};

MARS_DEV GPair grad_pair(const GItem& it, int p) {
  GPair q;
  q.g = it.g0 + p / it.np1;
  const int r = p % it.np1;
  if (r < it.nc) {
    q.qs = 0;
    q.qi = it.jt + r;
  } else {
    q.qs = 1;
    q.qi = it.mlo + (r - it.nc);
  }
  return q;
}

// Query columns [lo, hi] of a pair's tile that key kk (index within its stream) is visible
// to; empty (lo > hi) for a key past L.
MARS_DEV void visible_cols(const GArgs& a, const GItem& it, const GPair& pr, int kk, int& lo,
                           int& hi) {
  const int q0 = GT * pr.qi;
  lo = 1;
  hi = 0;
  if (kk >= a.L) return;
  int tlo, thi;                              // visible query rows of stream qs
  if (it.ks == 0 && pr.qs == 0) {            // clean key, clean rows: t >= kk
    tlo = kk;
    thi = a.L - 1;
  } else if (it.ks == 0) {                   // clean key, masked rows: block start > kk
    tlo = (kk / a.B + 1) * a.B;
    thi = a.L - 1;
  } else {                                   // masked key, masked rows of its block, t >= kk
    tlo = kk;
    thi = min(a.L, (kk / a.B + 1) * a.B) - 1;
  }
  lo = max(tlo - q0, 0);
  hi = min(thi - q0, GT - 1);
}

MARS_DEV uint32_t bits(int lo, int hi) {     // bits [lo, hi) of a 32-bit word, clamped
  lo = max(0, min(32, lo));
  hi = max(0, min(32, hi));
  if (hi <= lo) return 0u;
  return (hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u)) & ~((1u << lo) - 1u);
}

MARS_DEV uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

MARS_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// TMEM column of K-step k (16 queries) of P^T or dS^T in its buffer: queries [0, 64) are
// packed over columns [0, 32) and queries [64, 128) over [64, 96), the first half of each
// half's own fp32 columns.
MARS_DEV uint32_t p_col(int k) { return (uint32_t)(8 * k + (k >= 4 ? 32 : 0)); }

// Instruction descriptor with A and B majorness (bit 15: A MN-major, bit 16: B MN-major).
MARS_DEV uint32_t idesc_ab(int M, int N, bool a_mn, bool b_mn) {
  return idesc_bf16_f32(M, N, b_mn) | ((a_mn ? 1u : 0u) << 15);
}

template <int D>
__global__ void __launch_bounds__(GRAD_THREADS, 1)
dual_grad_kernel(const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, GArgs a) {
  using S = GSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ GBar bar;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* ab = &bar.abort;

  if (threadIdx.x == 0) {
    bar.abort = 0;
    mbar_init(&bar.kv_full, 1);
    mbar_init(&bar.kv_empty, 1);
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&bar.full[i], 1);
      mbar_init(&bar.empty[i], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&bar.s_full[h], 1);
      mbar_init(&bar.dp_full[h], 1);
      mbar_init(&bar.p_full[h], MATH_THREADS / 2);
      mbar_init(&bar.ds_full[h], MATH_THREADS / 2);
      mbar_init(&bar.dv_done[h], 1);
      mbar_init(&bar.dk_done[h], 1);
    }
    mbar_init(&bar.acc_full, 1);
    mbar_init(&bar.acc_free, MATH_THREADS);
    mbar_init(&bar.drain, 1);
    mbar_init(&bar.drain_ts, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bar.tmem_base, S::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = __shfl_sync(0xffffffffu, bar.tmem_base, 0);

  const int total = (int)grad_item_count(a.batch, a.hkv, a.G, a.nt, a.B);
  const int G = gridDim.x, c = blockIdx.x;
  auto item_id = [&](int r) { return r * G + ((r & 1) ? G - 1 - c : c); };
  const int rounds = (total + G - 1) / G;
  const int n2 = 2 * a.L;

  if (warp == 0) {
    // ---------------------------------------------------------------- loads
    int gp = 0, ii = 0, nkv = 0;
    bool ok = true;
    for (int r = 0; r < rounds && ok; ++r) {
      const int id = item_id(r);
      if (id >= total) continue;
      const GItem it = grad_item(a, id);
      if (lane == 0) {
        if (ii > 0) ok = mbar_wait(&bar.kv_empty, (ii - 1) & 1, ab, a.status);
        if (ok) {
          mbar_arrive_expect_tx(&bar.kv_full, 2 * S::T_BYTES);
          const int z = it.b * n2 + it.ks * a.L + GT * it.jt;
          for (int x = 0; x < D / 64; ++x) {
            tma_load_3d(smem + S::OFF_K + x * (GT * 128), &tm_k, &bar.kv_full, x * 64, it.kvh, z);
            tma_load_3d(smem + S::OFF_V + x * (GT * 128), &tm_v, &bar.kv_full, x * 64, it.kvh, z);
          }
          ++nkv;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      const int np = it.npg;
      for (int p = 0; p < np && ok; ++p, ++gp) {
        const GPair pr = grad_pair(it, p);
        const int st = gp % NSTAGE;
        uint8_t* stage = smem + S::OFF_RING + st * S::STAGE;
        if (lane == 0) ok = mbar_wait(&bar.empty[st], ((gp / NSTAGE) & 1) ^ 1, ab, a.status);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        const int h = it.kvh * a.G + pr.g;
        if (lane == 0) {
          // lse and D of the tile's 128 rows (one padded row block each), then Q and dO
          const size_t rb = (((size_t)it.b * a.hq + h) * 2 + pr.qs) * (size_t)(GT * a.nt) +
                            (size_t)GT * pr.qi;
          mbar_arrive_expect_tx(&bar.full[st], 2 * S::T_BYTES + 2 * GT * 4);
          bulk_load(stage + S::ST_LSE, a.lse + rb, GT * 4, &bar.full[st]);
          bulk_load(stage + S::ST_D, a.drow + rb, GT * 4, &bar.full[st]);
          const int z = it.b * n2 + pr.qs * a.L + GT * pr.qi;
          for (int x = 0; x < D / 64; ++x) {
            tma_load_3d(stage + S::ST_Q + x * (GT * 128), &tm_q, &bar.full[st], x * 64, h, z);
            tma_load_3d(stage + S::ST_DO + x * (GT * 128), &tm_do, &bar.full[st], x * 64, h, z);
          }
        }
      }
      ++ii;
    }
    // wait (bounded) for the copies still in flight
    if (lane == 0) {
      if (nkv > 0) mbar_wait(&bar.kv_full, (nkv - 1) & 1, nullptr, a.status);
      for (int k = 1; k <= NSTAGE && gp - k >= 0; ++k)
        mbar_wait(&bar.full[(gp - k) % NSTAGE], ((gp - k) / NSTAGE) & 1, nullptr, a.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- S^T and dP^T MMAs
    if (lane == 0) {
      // S^T, dP^T: K-major A and B, one N = 64 group per 64-query half of the pair
      const uint32_t id_qk = idesc_ab(GT, GT / 2, false, false);
      const uint64_t kd = sdesc_sw128(smem_u32(smem + S::OFF_K), 16, 1024);
      const uint64_t vd = sdesc_sw128(smem_u32(smem + S::OFF_V), 16, 1024);
      auto stage_of = [&](int g2) { return smem_u32(smem + S::OFF_RING + (g2 % NSTAGE) * S::STAGE); };
      auto issue_st = [&](int g2) -> bool {            // S^T = K Q^T of pair g2, by halves
        if (!mbar_wait(&bar.full[g2 % NSTAGE], (g2 / NSTAGE) & 1, ab, a.status)) return false;
        const uint64_t qd = sdesc_sw128(stage_of(g2) + S::ST_Q, 16, 1024);
        for (int h = 0; h < 2; ++h) {
          // half h's S^T buffer holds its P^T of the previous pair until that dV has read it
          if (g2 > 0 && !mbar_wait(&bar.dv_done[h], (g2 - 1) & 1, ab, a.status)) return false;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * (GT * 128) + (k & 3) * 32;
            mma_bf16_ss(tmem + S::TM_S + (GT / 2) * h, sdesc_advance(kd, off),
                        sdesc_advance(qd, off + h * (GT / 2) * 128), id_qk, k != 0);
          }
          mma_commit(&bar.s_full[h]);
        }
        return true;
      };
      auto issue_dp = [&](int g2) -> bool {            // dP^T = V dO^T of pair g2, by halves
        const uint64_t dod = sdesc_sw128(stage_of(g2) + S::ST_DO, 16, 1024);
        for (int h = 0; h < 2; ++h) {
          // half h's dP^T buffer holds its dS^T of the previous pair until that dK has read it
          if (g2 > 0 && !mbar_wait(&bar.dk_done[h], (g2 - 1) & 1, ab, a.status)) return false;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * (GT * 128) + (k & 3) * 32;
            mma_bf16_ss(tmem + S::TM_DP + (GT / 2) * h, sdesc_advance(vd, off),
                        sdesc_advance(dod, off + h * (GT / 2) * 128), id_qk, k != 0);
          }
          mma_commit(&bar.dp_full[h]);
        }
        return true;
      };
      int gp = 0, ii = 0;
      bool ok = true;
      for (int r = 0; r < rounds && ok; ++r) {
        const int id = item_id(r);
        if (id >= total) continue;
        const int np = grad_item(a, id).npg;
        if (!(ok = mbar_wait(&bar.kv_full, ii & 1, ab, a.status))) break;
        for (int p = 0; p < np && ok; ++p, ++gp) ok = issue_st(gp) && issue_dp(gp);
        if (!ok) break;
        mma_commit(&bar.kv_empty);                       // K and V are read by these MMAs only
        ++ii;
      }
      mma_commit(&bar.drain);
      mbar_wait(&bar.drain, 0, nullptr, a.status);
    }
  } else if (warp == GRAD_TS_WARP) {
    // -------------------------------------------------------- dV and dK MMAs
    if (lane == 0) {
      const uint32_t id_acc = idesc_ab(GT, D, false, true);    // dV, dK: TMEM A, MN-major B
      int gp = 0, ii = 0;
      bool ok = true;
      for (int r = 0; r < rounds && ok; ++r) {
        const int id = item_id(r);
        if (id >= total) continue;
        const int np = grad_item(a, id).npg;
        for (int p = 0; p < np; ++p, ++gp) {
          const int st = gp % NSTAGE;
          const uint32_t sb = smem_u32(smem + S::OFF_RING + st * S::STAGE);
          const uint64_t dod = sdesc_sw128(sb + S::ST_DO, GT * 128, 1024);
          const uint64_t qd = sdesc_sw128(sb + S::ST_Q, GT * 128, 1024);
          // the stage's Q and dO have landed (it is released below, so this phase is current)
          if (!(ok = mbar_wait(&bar.full[st], (gp / NSTAGE) & 1, ab, a.status))) break;
          // dV of the item starts from zero: the previous item's dV and dK must be read
          if (p == 0 && ii > 0 && !(ok = mbar_wait(&bar.acc_free, (ii - 1) & 1, ab, a.status)))
            break;
          for (int h = 0; h < 2 && ok; ++h) {              // dV += P^T dO, half h's queries
            if (!(ok = mbar_wait(&bar.p_full[h], gp & 1, ab, a.status))) break;
            tc_fence_after();
#pragma unroll
            for (int kq = 0; kq < GT / 32; ++kq) {
              const int k = (GT / 32) * h + kq;
              mma_bf16_ts(tmem + S::TM_DV, tmem + S::TM_S + p_col(k),
                          sdesc_advance(dod, k * 2048), id_acc, (p | k) != 0);
            }
            mma_commit(&bar.dv_done[h]);
          }
          for (int h = 0; h < 2 && ok; ++h) {              // dK += dS^T Q, half h's queries
            if (!(ok = mbar_wait(&bar.ds_full[h], gp & 1, ab, a.status))) break;
            tc_fence_after();
#pragma unroll
            for (int kq = 0; kq < GT / 32; ++kq) {
              const int k = (GT / 32) * h + kq;
              mma_bf16_ts(tmem + S::TM_DK, tmem + S::TM_DP + p_col(k),
                          sdesc_advance(qd, k * 2048), id_acc, (p | k) != 0);
            }
            mma_commit(&bar.dk_done[h]);
          }
          if (!ok) break;
          // S^T and dP^T of this pair completed before the math warps formed dS^T, and the
          // math warps have read the stage's lse and D rows: the stage is free after dK
          mma_commit(&bar.empty[st]);
        }
        if (!ok) break;
        mma_commit(&bar.acc_full);
        ++ii;
      }
      mma_commit(&bar.drain_ts);
      mbar_wait(&bar.drain_ts, 0, nullptr, a.status);
    }
  } else {
    // ------------------------------------------------- math (warps 2..9, two per quadrant)
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;                  // query columns [64 half, 64 half + 64)
    const int row = quad * 32 + lane;                  // TMEM lane: key row, then query row
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    constexpr int HC = GT / 2;                         // columns per thread
    constexpr int HD = D / 2;                          // accumulator columns per thread
    auto warp_wait = [&](uint64_t* b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, ab, a.status));
    };
    int gp = 0, ii = 0;
    bool ok = true;
    for (int r = 0; r < rounds && ok; ++r) {
      const int id = item_id(r);
      if (id >= total) continue;
      const GItem it = grad_item(a, id);
      const int kk = GT * it.jt + row;                 // this thread's key (within stream ks)
      const int np = it.npg;
      for (int p = 0; p < np && ok; ++p, ++gp) {
        const GPair pr = grad_pair(it, p);
        const int st = gp % NSTAGE;
        uint8_t* stage = smem + S::OFF_RING + st * S::STAGE;
        const float* ls = reinterpret_cast<const float*>(stage + S::ST_LSE) + HC * half;
        const float* dsv = reinterpret_cast<const float*>(stage + S::ST_D) + HC * half;
        int lo, hi;
        visible_cols(a, it, pr, kk, lo, hi);
        lo -= HC * half;
        hi -= HC * half;
        // P^T: exp2(scale log2e S - lse) on the visible query columns, 0 elsewhere
        if (!(ok = warp_wait(&bar.s_full[half], gp & 1))) break;
        tc_fence_after();
        uint32_t v[HC];
#pragma unroll
        for (int q = 0; q < HC / 32; ++q)
          tmem_ld32(tmem + S::TM_S + HC * half + q * 32 + lane_off,
                    *reinterpret_cast<uint32_t(*)[32]>(v + q * 32));
        tmem_ld_wait();
        // masked columns become -inf (exp2 gives 0) only where this row's range does not
        // cover the whole half; the scale-and-shift runs as packed f32x2 FMAs
        if (!(lo <= 0 && hi >= HC - 1)) {
#pragma unroll
          for (int q = 0; q < HC / 32; ++q) {
            const uint32_t mk = bits(lo - 32 * q, hi + 1 - 32 * q);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (!((mk >> e) & 1u)) v[32 * q + e] = 0xff800000u;
          }
        }
        uint32_t pp[HC / 2];
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
#pragma unroll
        for (int e = 0; e < HC; e += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(ls + e);
          const float2 t01 = __ffma2_rn(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                        sc2, make_float2(-l4.x, -l4.y));
          const float2 t23 = __ffma2_rn(make_float2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])),
                                        sc2, make_float2(-l4.z, -l4.w));
          pp[e / 2] = pack2(ex2(t01.x), ex2(t01.y));
          pp[e / 2 + 1] = pack2(ex2(t23.x), ex2(t23.y));
        }
        // over this half's own S^T columns (the other half may still be reading its own)
        tmem_st32(tmem + S::TM_S + HC * half + lane_off, *reinterpret_cast<uint32_t(*)[32]>(pp));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&bar.p_full[half]);
        // dS^T = P^T * (dP^T - D), over this half's own dP^T columns (the dK MMA's A)
        if (!(ok = warp_wait(&bar.dp_full[half], gp & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < HC / 32; ++q)
          tmem_ld32(tmem + S::TM_DP + HC * half + q * 32 + lane_off,
                    *reinterpret_cast<uint32_t(*)[32]>(v + q * 32));
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < HC; e += 4) {                // dS over P, packed f32x2
          const float4 d4 = *reinterpret_cast<const float4*>(dsv + e);
          const float2 p01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pp[e / 2]));
          const float2 p23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pp[e / 2 + 1]));
          const float2 s01 = __fmul2_rn(p01, __fadd2_rn(make_float2(__uint_as_float(v[e]),
                                                                    __uint_as_float(v[e + 1])),
                                                        make_float2(-d4.x, -d4.y)));
          const float2 s23 = __fmul2_rn(p23, __fadd2_rn(make_float2(__uint_as_float(v[e + 2]),
                                                                    __uint_as_float(v[e + 3])),
                                                        make_float2(-d4.z, -d4.w)));
          pp[e / 2] = pack2(s01.x, s01.y);
          pp[e / 2 + 1] = pack2(s23.x, s23.y);
        }
        tmem_st32(tmem + S::TM_DP + HC * half + lane_off, *reinterpret_cast<uint32_t(*)[32]>(pp));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&bar.ds_full[half]);
      }
      if (!ok) break;
      // the item's dV and dK rows (this thread's half of the columns), added to dV and dK
      if (!(ok = warp_wait(&bar.acc_full, ii & 1))) break;
      tc_fence_after();
      uint32_t dvr[HD], dkr[HD];
#pragma unroll
      for (int q = 0; q < HD / 32; ++q) {
        tmem_ld32(tmem + S::TM_DV + HD * half + q * 32 + lane_off,
                  *reinterpret_cast<uint32_t(*)[32]>(dvr + q * 32));
        tmem_ld32(tmem + S::TM_DK + HD * half + q * 32 + lane_off,
                  *reinterpret_cast<uint32_t(*)[32]>(dkr + q * 32));
      }
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive_warp(&bar.acc_free);
      if (kk < a.L) {
        const size_t o =
            (((size_t)it.b * n2 + (size_t)it.ks * a.L + kk) * a.hkv + it.kvh) * D + HD * half;
#pragma unroll
        for (int e = 0; e < HD; e += 4) {
          atomicAdd(reinterpret_cast<float4*>(a.dv + o + e),
                    make_float4(__uint_as_float(dvr[e]), __uint_as_float(dvr[e + 1]),
                                __uint_as_float(dvr[e + 2]), __uint_as_float(dvr[e + 3])));
          atomicAdd(reinterpret_cast<float4*>(a.dk + o + e),
                    make_float4(__uint_as_float(dkr[e]) * a.scale,
                                __uint_as_float(dkr[e + 1]) * a.scale,
                                __uint_as_float(dkr[e + 2]) * a.scale,
                                __uint_as_float(dkr[e + 3]) * a.scale));
        }
      }
      ++ii;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S::TM_COLS);
  }
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct GradBuffers {
  __nv_bfloat16* do_bf;     // dO in bf16, [b, 2L, hq, d]
  float* drow;              // D, [b][hq][2][Lp], Lp = L rounded up to 128
  float* lse;               // same layout
  size_t bytes;
};

GradBuffers carve(void* base, int batch, int L, int hq, int d) {
  const size_t n = 2 * (size_t)L;
  const size_t np = 2 * (size_t)((L + GT - 1) / GT * GT);     // both streams, padded rows
  GradBuffers g{};
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* at = p ? p + off : nullptr;
    off += align256(bytes);
    return at;
  };
  g.do_bf = reinterpret_cast<__nv_bfloat16*>(take((size_t)batch * n * hq * d * sizeof(uint16_t)));
  g.drow = reinterpret_cast<float*>(take((size_t)batch * np * hq * sizeof(float)));
  g.lse = reinterpret_cast<float*>(take((size_t)batch * np * hq * sizeof(float)));
  g.bytes = off;
  return g;
}

template <int D>
cudaError_t launch_grad_tc(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const GradBuffers& w, int batch, int L, int B, int hq, int hkv,
                           float scale, float* dk, float* dv, int32_t* status,
                           cudaStream_t stream) {
  using S = GSmem<D>;
  static_assert(S::TOTAL + sizeof(GBar) <= 227 * 1024, "gradient layout fits shared memory");
  CUtensorMap tq, tdo, tk, tv;
  const uint64_t rows = (uint64_t)batch * 2 * L;
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)hq, rows};
    const uint64_t str[2] = {(uint64_t)D * 2, (uint64_t)hq * D * 2};
    const uint32_t box[3] = {64, 1, GT};
    if (!encode_tmap_bf16(&tq, q, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_tmap_bf16(&tdo, w.do_bf, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)hkv, rows};
    const uint64_t str[2] = {(uint64_t)D * 2, (uint64_t)hkv * D * 2};
    const uint32_t box[3] = {64, 1, GT};
    if (!encode_tmap_bf16(&tk, k, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_tmap_bf16(&tv, v, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  GArgs a{batch, L, B, hq, hkv, hq / hkv, (L + GT - 1) / GT, scale, scale * 1.4426950408889634f,
          w.lse, w.drow, dk, dv, status};
  static std::atomic<int> attr[64];
  const cudaError_t ea = set_smem_limit_once(dual_grad_kernel<D>, S::TOTAL, attr);
  if (ea != cudaSuccess) return ea;
  const long long items = grad_item_count(batch, hkv, hq / hkv, a.nt, B);
  const long long ctas = std::min<long long>(items, num_sms());
  dual_grad_kernel<D><<<(unsigned)ctas, GRAD_THREADS, S::TOTAL, stream>>>(tq, tdo, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

size_t dual_grad_workspace_bytes(int batch, int L, int B, int hq, int hkv, int d) {
  (void)B;
  (void)hkv;
  return carve(nullptr, batch, L, hq, d).bytes;
}

cudaError_t launch_dual_stream_grad(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    const float* o, const float* d_o, int batch, int L, int B,
                                    int hq, int hkv, int d, float scale, float* dq, float* dk,
                                    float* dv, void* workspace, int32_t* status,
                                    cudaStream_t stream, const float* lse_in) {
  const long long n = 2LL * L;
  GradBuffers w = carve(workspace, batch, L, hq, d);
  const int lp = (L + GT - 1) / GT * GT;
  cudaError_t e = cudaMemsetAsync(dk, 0, (size_t)batch * n * hkv * d * sizeof(float), stream);
  // D rows past L (the pads of a partial last tile) must read as finite zeros; the
  // forward writes the lse pads itself
  if (e == cudaSuccess)
    e = cudaMemsetAsync(w.drow, 0, (size_t)batch * hq * 2 * lp * sizeof(float), stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(dv, 0, (size_t)batch * n * hkv * d * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  if (lse_in) {
    w.lse = const_cast<float*>(lse_in);              // the forward's, read only
  } else if ((e = launch_dual_stream(q, k, v, nullptr, batch, L, B, hq, hkv, d, scale, status,
                                     stream, w.lse)) != cudaSuccess) {
    return e;                                        // row statistics: forward without O
  }
  const long long nrows = (long long)batch * n * hq;
  grad_prep_kernel<<<(unsigned)((nrows + 7) / 8), 256, 0, stream>>>(o, d_o, w.do_bf, w.drow,
                                                                    nrows, (int)n, hq, d, lp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = d == 64 ? launch_grad_tc<64>(q, k, v, w, batch, L, B, hq, hkv, scale, dk, dv, status,
                                   stream)
              : launch_grad_tc<128>(q, k, v, w, batch, L, B, hq, hkv, scale, dk, dv, status,
                                    stream);
  count_launches(2);
  if (e != cudaSuccess) return e;
  return launch_dual_stream_dq(q, k, v, reinterpret_cast<const uint16_t*>(w.do_bf), w.lse,
                               w.drow, dq, batch, L, B, hq, hkv, d, scale, status, stream);
}

}  // namespace mars
