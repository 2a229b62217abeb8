// Dual-stream (training-form) attention under the MARS mask M (papernotes.org notes of
// "MARS: Enabling Autoregressive Models Multi-Token Generation", Key design 1, eq. M,
// beta(t) = ceil(t/B); overall framework: clean stream x and masked stream x~ in one
// forward over z = [x; x~]).
//
// In 0-indexed stream-local terms a query row sees one or two contiguous key ranges:
//   clean row t (global t):    keys [0, t]
//   masked row t (global L+t): clean keys [0, B*(t/B)) and masked keys [L + B*(t/B), L + t]
// A work item is 128 consecutive rows of one stream for one (batch, query head); it visits
// only the 128-key tiles that intersect those ranges: for a clean tile the causal tiles
// 0..t/128, for a masked tile the clean tiles below its block start plus the tile(s)
// holding its own blocks. Fully masked tiles are never loaded; tiles every row sees in
// full skip the per-key test. One persistent CTA per SM runs many items back to back. The
// tile engine (flash_tc.cuh) runs QK^T and PV on tcgen05 with S and O in TMEM.
//
// The same items drive the dQ half of the attention gradient (dual_dq_kernel below); a
// statistics-only run of the forward (no O store) gives the gradient its row log-sum-exp.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "flash_tc.cuh"
#include "internal.h"

namespace mars {

namespace {

using flash::BKV;
using flash::BQ;

// A CTA runs many work items, so O is staged in an area of its own (two 32-column boxes per
// round) while the K/V rings already stream the next item.
template <int D>
struct DualPolicy {
  static constexpr bool kHandOff = true;
  static constexpr bool kRowStats = true;
  static constexpr int kStageBoxes = D / 32 < 2 ? D / 32 : 2;
  const CUtensorMap* tm_o;   // O as [2*batch][L][hq][D] fp32, box [1][128][1][32]
  float* lse;                // optional: [batch][hq][2][Lp] row log-sum-exp (log2 units),
                             // Lp = L rounded up to 128 (pad rows written as 0)
  int lp;
  int store_o;               // 0: O is not written (a statistics-only run)
  int L, B, hq;
  int b, h, stream, r0;
  int n_clean, n_total, mstart, full_limit;
  int kvh, zb;

  MARS_DEV bool row_valid(int row) const { return r0 + row < L; }
  MARS_DEV flash::RowVis row_vis(int row) const {
    const int t = r0 + row;
    if (stream == 0) return {t + 1, INT_MAX, -1};
    const int bs = (t / B) * B;
    return {bs, L + bs, L + t};
  }
  struct Tile {
    int kg0;     // global key index of column 0
    int kend;    // keys >= kend belong to another tile
    bool full;
  };
  MARS_DEV int tile_key0(int j) const {
    return j < n_clean ? j * BKV : mstart + (j - n_clean) * BKV;
  }
  // clean-segment tiles admit clean keys only (a tile starting at 0 can reach past L)
  MARS_DEV Tile tile(int j) const {
    return {tile_key0(j), j < n_clean ? L : INT_MAX, j < n_clean && (j + 1) * BKV <= full_limit};
  }
  // columns c with kg0 + c < kend and (kg0 + c < end1 or lo2 <= kg0 + c <= hi2)
  MARS_DEV flash::ColRange cols(const flash::RowVis& v, const Tile& t) const {
    const int lim = t.kend == INT_MAX ? BKV : min(BKV, t.kend - t.kg0);   // first col not owned
    flash::ColRange c;
    c.e1 = min(v.end1 - t.kg0, lim);
    c.s2 = v.lo2 == INT_MAX ? BKV : v.lo2 - t.kg0;
    c.e2 = min(v.hi2 - t.kg0, lim - 1);
    c.pmask = 0xffu;
    return c;
  }
  float* inv_slot;           // 1/l of the item's 128 rows for the epilogue warps
  int item;                  // index of this item among the CTA's items
  MARS_DEV void hand_off(int row, float inv) const { inv_slot[row] = inv; }
  MARS_DEV uint8_t* stage(uint8_t* smem) const {
    return smem + flash::Smem<D, kStageBoxes>::OFF_STAGE;
  }
  // log2 of the row's softmax denominator in units of scale*log2(e)*score: m + log2(l);
  // the pad rows of a partial last tile get 0
  MARS_DEV void row_stats(int row, float m, float l) const {
    if (lse)
      lse[(((size_t)b * hq + h) * 2 + stream) * lp + r0 + row] =
          row_valid(row) ? m + log2f(l) : 0.f;
  }
  // rows past L (a partial last query tile) fall outside the map's L extent and are not
  // written
  MARS_DEV void store_boxes(const uint8_t* stage, int b0, int n) const {
    if (!store_o) return;
    for (int c = 0; c < n; ++c)
      sm100::tma_store_4d(tm_o, stage + c * (BQ * 128), (b0 + c) * 32, h, r0, b * 2 + stream);
  }
};

struct DualArgs {
  int batch, L, B, hq, hkv, G, nqt;
  float scale_log2;
  int32_t* status;
  float* lse;
  int store_o;
};

// Work item id -> (batch, head, stream, query tile) and the key tiles it visits. Ids run
// over query tiles from the last (heaviest: most visible keys) to the first.
template <int D>
MARS_DEV DualPolicy<D> make_item(const DualArgs& a, int id, const CUtensorMap* tm_o) {
  DualPolicy<D> pol;
  const int b = id % a.batch;
  id /= a.batch;
  const int h = id % a.hq;
  id /= a.hq;
  const int stream = id & 1;
  const int qt = a.nqt - 1 - (id >> 1);
  pol.tm_o = tm_o;
  pol.lse = a.lse;
  pol.lp = a.nqt * BQ;
  pol.store_o = a.store_o;
  pol.L = a.L;
  pol.B = a.B;
  pol.hq = a.hq;
  pol.b = b;
  pol.h = h;
  pol.stream = stream;
  pol.r0 = qt * BQ;
  const int t_last = min(pol.r0 + BQ - 1, a.L - 1);
  if (stream == 0) {
    pol.n_clean = t_last / BKV + 1;
    pol.n_total = pol.n_clean;
    pol.mstart = 0;
    pol.full_limit = pol.r0 + 1;
  } else {
    const int clean_end = (t_last / a.B) * a.B;            // keys [0, clean_end)
    const int bs0 = (pol.r0 / a.B) * a.B;
    pol.n_clean = (clean_end + BKV - 1) / BKV;
    pol.mstart = a.L + bs0;
    pol.n_total = pol.n_clean + (t_last - bs0 + BKV) / BKV;
    pol.full_limit = bs0;
  }
  pol.kvh = h / a.G;
  pol.zb = b * 2 * a.L;
  return pol;
}

// K or V tile j of an item: one 3D box of 128 rows per 64-column half
template <int D, class Pol>
struct KVIssue {
  const Pol* pol;
  const CUtensorMap* tm;
  MARS_DEV void operator()(int j, uint8_t* dst, uint64_t* b) const {
    if ((threadIdx.x & 31) == 0) {
      const int z = pol->zb + pol->tile_key0(j);
      for (int x = 0; x < D / 64; ++x)
        sm100::tma_load_3d(dst + x * (BKV * 128), tm, b, x * 64, pol->kvh, z);
    }
  }
};

template <int D, class Pol>
MARS_DEV void load_q(uint8_t* smem, const CUtensorMap* tm_q, flash::Barriers& bar, const Pol& pol,
                     int L) {
  using S = flash::Smem<D>;
  sm100::mbar_arrive_expect_tx(&bar.q_full, S::Q_BYTES);
  for (int x = 0; x < D / 64; ++x)
    sm100::tma_load_3d(smem + S::OFF_Q + x * (BQ * 128), tm_q, &bar.q_full, x * 64, pol.h,
                       pol.zb + pol.stream * L + pol.r0);
}

// Shared set-up: barriers and TMEM; returns the warp-uniform TMEM base.
MARS_DEV uint32_t cta_setup(flash::Barriers& bar, int warp) {
  using namespace sm100;
  if (threadIdx.x == 0) flash::init_barriers(bar);
  if (warp == 1) {
    tmem_alloc(&bar.tmem_base, flash::Smem<64>::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // read once per warp and broadcast: a warp-uniform TMEM base
  return __shfl_sync(0xffffffffu, bar.tmem_base, 0);
}

MARS_DEV void cta_teardown(uint32_t tmem, int warp) {
  using namespace sm100;
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, flash::Smem<64>::TMEM_COLS);
  }
}

// One CTA per SM runs work items r*G + c (even rounds r) and r*G + G-1-c (odd rounds),
// G = gridDim.x, c = blockIdx.x, so heavy and light items even out. The rings, S buffers
// and barrier phases run on across items; the next item's Q is loaded as soon as the
// current item's last QK^T has completed. Three warpgroups: warps 0..3 K loader, QK^T
// issuer (TMEM owner), V loader, PV issuer; 4..7 softmax; 8..11 epilogue. The softmax
// warps hand each item's 1/l to the epilogue warps and go straight on to the next item,
// while those read O out of TMEM and write it back with TMA stores; the next item's
// first PV waits until O has been read.
constexpr int DUAL_THREADS = 384;
constexpr int DUAL_WG0_REGS = 88, DUAL_SOFTMAX_REGS = 232, DUAL_EPI_REGS = 160;
static_assert(128 * (DUAL_WG0_REGS + DUAL_SOFTMAX_REGS + DUAL_EPI_REGS) <=
                  DUAL_THREADS * (65536 / DUAL_THREADS / 8 * 8),
              "the register split fits the launch's register pool");

struct DualEpi {
  float inv[2][BQ];        // 1/l per row, by item parity
};

template <int D>
__global__ void __launch_bounds__(DUAL_THREADS, 1)
dual_stream_persistent_kernel(const __grid_constant__ CUtensorMap tm_q,
                              const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v,
                              const __grid_constant__ CUtensorMap tm_o, DualArgs a) {
  using namespace sm100;
  using Pol = DualPolicy<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ flash::Barriers bar;
  __shared__ DualEpi epi;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tmem = cta_setup(bar, warp);
  volatile int* ab = &bar.abort;
  const int total = a.nqt * 2 * a.hq * a.batch;
  const int G = gridDim.x, c = blockIdx.x;
  auto item_id = [&](int r) { return r * G + ((r & 1) ? G - 1 - c : c); };
  const int rounds = (total + G - 1) / G;
  const int wg = warp >> 2;

  if (wg == 0) {
    regs_lower<DUAL_WG0_REGS>();
    if (warp == 0 || warp == 2) {
      const bool is_v = warp == 2;
      int last_k[flash::K_STAGES], last_v[flash::V_STAGES];
      for (int i = 0; i < flash::K_STAGES; ++i) last_k[i] = -1;
      for (int i = 0; i < flash::V_STAGES; ++i) last_v[i] = -1;
      int j0 = 0;
      for (int r = 0; r < rounds; ++r) {
        const int id = item_id(r);
        if (id >= total) continue;
        const Pol pol = make_item<D>(a, id, &tm_o);
        const bool ok = is_v ? flash::load_ring_item<D, flash::V_STAGES>(
                                   bar, smem, pol.n_total, j0, last_v, false, a.status, true,
                                   KVIssue<D, Pol>{&pol, &tm_v})
                             : flash::load_ring_item<D, flash::K_STAGES>(
                                   bar, smem, pol.n_total, j0, last_k, false, a.status, false,
                                   KVIssue<D, Pol>{&pol, &tm_k});
        if (!ok) break;
        j0 += pol.n_total;
      }
      // wait (bounded) for every copy still in flight
      const Pol none{};
      if (is_v)
        flash::load_ring_item<D, flash::V_STAGES>(bar, smem, 0, j0, last_v, true, a.status, true,
                                                  KVIssue<D, Pol>{&none, &tm_v});
      else
        flash::load_ring_item<D, flash::K_STAGES>(bar, smem, 0, j0, last_k, true, a.status, false,
                                                  KVIssue<D, Pol>{&none, &tm_k});
    } else if (lane == 0) {
      const bool pv = warp == 3;
      int j0 = 0, i = 0, nq = 0;
      for (int r = 0; r < rounds; ++r) {
        const int id = item_id(r);
        if (id >= total) continue;
        const Pol pol = make_item<D>(a, id, &tm_o);
        if (pv) {
          if (!flash::pv_issuer<D>(bar, smem, pol.n_total, tmem, a.status, j0,
                                   i > 0 ? (i - 1) & 1 : -1))
            break;
        } else {
          // Q is replaced once the previous item's QK^T MMAs have completed
          if (i > 0 && !mbar_wait(&bar.q_empty, (i - 1) & 1, ab, a.status)) break;
          load_q<D>(smem, &tm_q, bar, pol, a.L);
          ++nq;
          if (!flash::s_issuer<D>(bar, smem, pol.n_total, tmem, a.status, j0, i & 1)) break;
          mma_commit(&bar.q_empty);
        }
        j0 += pol.n_total;
        ++i;
      }
      // wait (bounded) for this thread's own MMAs, so none is in flight at teardown
      uint64_t* drain = pv ? &bar.drain_pv : &bar.drain;
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr, a.status);
      // and for the last Q copy (in flight still if the item was abandoned)
      if (!pv && nq > 0) mbar_wait(&bar.q_full, (nq - 1) & 1, nullptr, a.status);
    }
  } else if (wg == 1) {
    regs_raise<DUAL_SOFTMAX_REGS>();
    int j0 = 0, i = 0;
    for (int r = 0; r < rounds; ++r) {
      const int id = item_id(r);
      if (id >= total) continue;
      Pol pol = make_item<D>(a, id, &tm_o);
      pol.inv_slot = epi.inv[i & 1];
      pol.item = i;
      if (!flash::softmax_loop<D>(bar, smem, pol, pol.n_total, tmem, a.scale_log2, a.status, j0))
        break;
      j0 += pol.n_total;
      ++i;
    }
  } else {
    regs_lower<DUAL_EPI_REGS>();
    const int store_thread = 8 * 32;
    const int row = (warp & 3) * 32 + lane;
    volatile int* abv = ab;
    int i = 0, er = 0;
    for (int r = 0; r < rounds; ++r) {
      const int id = item_id(r);
      if (id >= total) continue;
      const Pol pol = make_item<D>(a, id, &tm_o);
      // 1/l of this thread's row, handed over by the softmax warps
      if (!__all_sync(0xffffffffu, mbar_wait(&bar.epi_ready, i & 1, abv, a.status))) break;
      const float inv = epi.inv[i & 1][row];
      mbar_arrive_warp(&bar.epi_taken);
      if (!flash::staged_epilogue<D>(bar, smem, pol, tmem, i & 1, inv, er, store_thread,
                                     a.status))
        break;
      ++i;
    }
    if ((int)threadIdx.x == store_thread) bulk_wait_read_all();   // stores have read staging
  }
  cta_teardown(tmem, warp);
}

// ------------------------------------------------------------------ dQ of the gradient

// dQ = scale * sum over visible key tiles j of dS_j K_j, dS = P * (dP - D), P =
// exp2(scale log2(e) S - lse), S = Q K_j^T, dP = dO V_j^T: the row-parallel half of the
// attention gradient. Work items, their key tiles and the masks are the forward's; per key
// tile three MMAs (S, dP, dQ += dS K) with dQ accumulated in TMEM and written once per row.
// TMEM: S at column 0, dP at 128, dQ at 256, dS (bf16 pairs, 64 columns) at 384. S and dP
// are each free once the math warps have loaded them, so the next tile's S and dP never
// wait for a dQ MMA, and the math warps form P as soon as S has landed, loading dP only
// for dS: the next tile's S runs under this tile's exponentials. Warps: 0 K loader,
// 1 TMEM owner and S/dP issuer (it also loads each item's Q and dO), 2..9 math (two per
// TMEM lane quadrant, 64 key columns each), 10 V loader, 11 dQ issuer. The shared-memory
// operand MMAs (S, dP) and the TMEM-operand ones (dQ) come from two threads on different
// sub-partitions: one thread alternating the two forms issues them about a quarter slower.
constexpr int DQ_MATH_WARPS = 8;
constexpr int DQ_THREADS = 32 * (4 + DQ_MATH_WARPS);
constexpr int DQ_V_WARP = 2 + DQ_MATH_WARPS;
constexpr int DQ_ISSUE_WARP = 3 + DQ_MATH_WARPS;

struct DQBar {
  uint64_t s_full, dp_full, s_free, dp_free, ds_full, dq_done, acc_free;
};

struct DQArgs {
  DualArgs f;              // shape, scale_log2, status
  float scale;
  const float* lse;        // [batch][hq][2][Lp], Lp = L rounded up to 128
  const float* drow;       // same layout
  float* dq;               // [batch][2L][hq][D]
};

template <int D>
__global__ void __launch_bounds__(DQ_THREADS, 1)
dual_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, DQArgs da) {
  using namespace sm100;
  using Pol = DualPolicy<D>;
  using S = flash::Smem<D, Pol::kStageBoxes>;     // Q, K ring, V ring; dO over the staging
  static_assert(D * BQ * 2 <= Pol::kStageBoxes * BQ * 128, "dO tile fits the staging area");
  constexpr int TM_S = 0, TM_DP = BKV, TM_DQ = 2 * BKV, TM_DS = 3 * BKV;
  static_assert(TM_DQ + D <= TM_DS && TM_DS + BKV / 2 <= 512, "TMEM columns");
  const DualArgs& a = da.f;
  extern __shared__ uint8_t smem_raw[];
  __shared__ flash::Barriers bar;
  __shared__ DQBar qb;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&qb.s_full, 1);
    mbar_init(&qb.dp_full, 1);
    mbar_init(&qb.dq_done, 1);
    mbar_init(&qb.s_free, 32 * DQ_MATH_WARPS);
    mbar_init(&qb.dp_free, 32 * DQ_MATH_WARPS);
    mbar_init(&qb.ds_full, 32 * DQ_MATH_WARPS);
    mbar_init(&qb.acc_free, 32 * DQ_MATH_WARPS);
  }
  const uint32_t tmem = cta_setup(bar, warp);     // also initialises bar (thread 0)
  volatile int* ab = &bar.abort;
  const int total = a.nqt * 2 * a.hq * a.batch;
  const int G = gridDim.x, c = blockIdx.x;
  auto item_id = [&](int r) { return r * G + ((r & 1) ? G - 1 - c : c); };
  const int rounds = (total + G - 1) / G;

  if (warp == 0 || warp == DQ_V_WARP) {
    const bool is_v = warp != 0;
    int last_k[flash::K_STAGES], last_v[flash::V_STAGES];
    for (int i = 0; i < flash::K_STAGES; ++i) last_k[i] = -1;
    for (int i = 0; i < flash::V_STAGES; ++i) last_v[i] = -1;
    int j0 = 0;
    for (int r = 0; r < rounds; ++r) {
      const int id = item_id(r);
      if (id >= total) continue;
      const Pol pol = make_item<D>(a, id, nullptr);
      const bool ok = is_v ? flash::load_ring_item<D, flash::V_STAGES>(
                                 bar, smem, pol.n_total, j0, last_v, false, a.status, true,
                                 KVIssue<D, Pol>{&pol, &tm_v})
                           : flash::load_ring_item<D, flash::K_STAGES>(
                                 bar, smem, pol.n_total, j0, last_k, false, a.status, false,
                                 KVIssue<D, Pol>{&pol, &tm_k});
      if (!ok) break;
      j0 += pol.n_total;
    }
    const Pol none{};
    if (is_v)
      flash::load_ring_item<D, flash::V_STAGES>(bar, smem, 0, j0, last_v, true, a.status, true,
                                                KVIssue<D, Pol>{&none, &tm_v});
    else
      flash::load_ring_item<D, flash::K_STAGES>(bar, smem, 0, j0, last_k, true, a.status, false,
                                                KVIssue<D, Pol>{&none, &tm_k});
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(BQ, BKV, false);   // S, dP: K-major A and B
      const uint64_t qd = sdesc_sw128(smem_u32(smem + S::OFF_Q), 16, 1024);
      const uint64_t dd = sdesc_sw128(smem_u32(smem + S::OFF_STAGE), 16, 1024);
      int jg0 = 0, i = 0, nq = 0;
      bool ok = true;
      auto issue_s = [&](int jg) -> bool {                // S_jg = Q K^T
        const int st = jg % flash::K_STAGES;
        if (!mbar_wait(&bar.k_full[st], (jg / flash::K_STAGES) & 1, ab, a.status)) return false;
        // S of the previous tile has been loaded by the math warps
        if (jg >= 1 && !mbar_wait(&qb.s_free, (jg - 1) & 1, ab, a.status)) return false;
        tc_fence_after();
        const uint64_t kd = sdesc_sw128(smem_u32(smem + S::OFF_K + st * S::KV_BYTES), 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * (BQ * 128) + (k & 3) * 32;
          mma_bf16_ss(tmem + TM_S, sdesc_advance(qd, off), sdesc_advance(kd, off), id_s, k != 0);
        }
        mma_commit(&qb.s_full);
        return true;
      };
      auto issue_dp = [&](int jg) -> bool {               // dP_jg = dO V^T (after issue_s(jg))
        const int st = jg % flash::V_STAGES;
        if (!mbar_wait(&bar.v_full[st], (jg / flash::V_STAGES) & 1, ab, a.status)) return false;
        // dP of the previous tile has been loaded by the math warps
        if (jg >= 1 && !mbar_wait(&qb.dp_free, (jg - 1) & 1, ab, a.status)) return false;
        tc_fence_after();
        const uint64_t vd = sdesc_sw128(smem_u32(smem + S::OFF_V + st * S::KV_BYTES), 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * (BQ * 128) + (k & 3) * 32;
          mma_bf16_ss(tmem + TM_DP, sdesc_advance(dd, off), sdesc_advance(vd, off), id_s, k != 0);
        }
        mma_commit(&qb.dp_full);
        mma_commit(&bar.v_empty[st]);
        return true;
      };
      for (int r = 0; r < rounds && ok; ++r) {
        const int id = item_id(r);
        if (id >= total) continue;
        const Pol pol = make_item<D>(a, id, nullptr);
        // Q and dO are replaced once the previous item's S and dP MMAs have completed
        if (i > 0 && !(ok = mbar_wait(&bar.q_empty, (i - 1) & 1, ab, a.status))) break;
        mbar_arrive_expect_tx(&bar.q_full, 2 * S::Q_BYTES);
        for (int x = 0; x < D / 64; ++x) {
          const int z = pol.zb + pol.stream * a.L + pol.r0;
          tma_load_3d(smem + S::OFF_Q + x * (BQ * 128), &tm_q, &bar.q_full, x * 64, pol.h, z);
          tma_load_3d(smem + S::OFF_STAGE + x * (BQ * 128), &tm_do, &bar.q_full, x * 64, pol.h, z);
        }
        ++nq;
        if (!(ok = mbar_wait(&bar.q_full, i & 1, ab, a.status))) break;
        const int n = pol.n_total;
        for (int jl = 0; jl < n && ok; ++jl) ok = issue_s(jg0 + jl) && issue_dp(jg0 + jl);
        if (!ok) break;
        mma_commit(&bar.q_empty);
        jg0 += n;
        ++i;
      }
      mma_commit(&bar.drain);
      mbar_wait(&bar.drain, 0, nullptr, a.status);
      if (nq > 0) mbar_wait(&bar.q_full, (nq - 1) & 1, nullptr, a.status);
    }
  } else if (warp == DQ_ISSUE_WARP) {
    if (lane == 0) {
      const uint32_t id_q = idesc_bf16_f32(BQ, D, true);      // dQ: TMEM A, MN-major B
      int jg0 = 0, i = 0;
      bool ok = true;
      for (int r = 0; r < rounds && ok; ++r) {
        const int id = item_id(r);
        if (id >= total) continue;
        const int n = make_item<D>(a, id, nullptr).n_total;
        for (int jl = 0; jl < n; ++jl) {
          const int jg = jg0 + jl, st = jg % flash::K_STAGES;
          // the accumulator of the previous item has been read out
          if (jl == 0 && i > 0 && !(ok = mbar_wait(&qb.acc_free, (i - 1) & 1, ab, a.status)))
            break;
          // K_jg has landed (its stage is released below, so this phase is still current)
          if (!(ok = mbar_wait(&bar.k_full[st], (jg / flash::K_STAGES) & 1, ab, a.status))) break;
          if (!(ok = mbar_wait(&qb.ds_full, jg & 1, ab, a.status))) break;
          tc_fence_after();
          const uint64_t kd = sdesc_sw128(smem_u32(smem + S::OFF_K + st * S::KV_BYTES),
                                          BKV * 128, 1024);
#pragma unroll
          for (int k = 0; k < BKV / 16; ++k)             // dQ += dS K (K tile MN-major)
            mma_bf16_ts(tmem + TM_DQ, tmem + TM_DS + 8 * k, sdesc_advance(kd, k * 2048), id_q,
                        (jl | k) != 0);
          mma_commit(&qb.dq_done);
          // S_jg, which also read this stage, completed before the math warps wrote dS_jg
          mma_commit(&bar.k_empty[st]);
        }
        if (!ok) break;
        mma_commit(&bar.o_final);
        jg0 += n;
        ++i;
      }
      mma_commit(&bar.drain_pv);
      mbar_wait(&bar.drain_pv, 0, nullptr, a.status);
    }
  } else {
    // math: thread = query row (TMEM lane), 64 key columns per warp
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    auto warp_wait = [&](uint64_t* b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, ab, a.status));
    };
    int jg0 = 0, i = 0;
    bool ok = true;
    for (int r = 0; r < rounds && ok; ++r) {
      const int id = item_id(r);
      if (id >= total) continue;
      const Pol pol = make_item<D>(a, id, nullptr);
      const bool rv = pol.row_valid(row);
      const flash::RowVis vis = pol.row_vis(row);
      const size_t srow = (((size_t)pol.b * a.hq + pol.h) * 2 + pol.stream) * (a.nqt * BQ) +
                          pol.r0 + row;
      const float lse = rv ? da.lse[srow] : 0.f;
      const float dd = rv ? da.drow[srow] : 0.f;
      const int n = pol.n_total;
      for (int jl = 0; jl < n && ok; ++jl) {
        const int jg = jg0 + jl;
        const typename Pol::Tile tile = pol.tile(jl);
        const flash::ColRange cr = rv ? pol.cols(vis, tile) : flash::ColRange{0, 0, -1, 0u};
        if (!(ok = warp_wait(&qb.s_full, jg & 1))) break;
        tc_fence_after();
        uint32_t sv[64];
#pragma unroll
        for (int q = 0; q < 2; ++q)
          tmem_ld32(tmem + TM_S + 64 * half + 32 * q + lane_off,
                    *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * q));
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive_warp(&qb.s_free);
        // masked keys become -inf (exp2 gives 0) where the tile is not fully visible
        if (!rv || !tile.full) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint32_t mk = rv ? flash::chunk_mask(cr, 2 * half + q) : 0u;
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (!((mk >> e) & 1u)) sv[32 * q + e] = 0xff800000u;
          }
        }
        // P = exp2(scale log2e S - lse) rounded to bf16 (as the key-tile kernel's P), then,
        // once dP has landed, dS = P * (dP - D), in packed f32x2 operations
        uint32_t ds[32];
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
        const float2 nl2 = make_float2(-lse, -lse), nd2 = make_float2(-dd, -dd);
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const float2 t = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                      sc2, nl2);
          ds[e / 2] = flash::pack_bf16x2(flash::ex2_approx(t.x), flash::ex2_approx(t.y));
        }
        if (!(ok = warp_wait(&qb.dp_full, jg & 1))) break;
        tc_fence_after();
        uint32_t pv[64];
#pragma unroll
        for (int q = 0; q < 2; ++q)
          tmem_ld32(tmem + TM_DP + 64 * half + 32 * q + lane_off,
                    *reinterpret_cast<uint32_t(*)[32]>(pv + 32 * q));
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive_warp(&qb.dp_free);
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const float2 pf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ds[e / 2]));
          const float2 x = __fmul2_rn(pf, __fadd2_rn(make_float2(__uint_as_float(pv[e]),
                                                                 __uint_as_float(pv[e + 1])), nd2));
          ds[e / 2] = flash::pack_bf16x2(x.x, x.y);
        }
        // dS has one buffer: the previous tile's dQ MMA must have read it
        if (jg > 0 && !(ok = warp_wait(&qb.dq_done, (jg - 1) & 1))) break;
        tc_fence_after();
        tmem_st32(tmem + TM_DS + 32 * half + lane_off, ds);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&qb.ds_full);
      }
      if (!ok) break;
      // dQ row, this warp's half of the columns
      if (!(ok = warp_wait(&bar.o_final, i & 1))) break;
      tc_fence_after();
      constexpr int HD = D / 2;
      uint32_t o[HD];
#pragma unroll
      for (int q = 0; q < HD / 32; ++q)
        tmem_ld32(tmem + TM_DQ + HD * half + 32 * q + lane_off,
                  *reinterpret_cast<uint32_t(*)[32]>(o + 32 * q));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive_warp(&qb.acc_free);
      if (rv) {
        float* dst = da.dq + ((((size_t)pol.b * 2 * a.L + (size_t)pol.stream * a.L + pol.r0 + row) *
                                   a.hq + pol.h) * D) + HD * half;
#pragma unroll
        for (int e = 0; e < HD; e += 4)
          *reinterpret_cast<float4*>(dst + e) =
              make_float4(__uint_as_float(o[e]) * da.scale, __uint_as_float(o[e + 1]) * da.scale,
                          __uint_as_float(o[e + 2]) * da.scale, __uint_as_float(o[e + 3]) * da.scale);
      }
      jg0 += n;
      ++i;
    }
  }
  cta_teardown(tmem, warp);
}

template <int D>
cudaError_t launch_dq_tc(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const uint16_t* do_bf, const float* lse, const float* drow, float* dq,
                         int batch, int L, int B, int hq, int hkv, float scale, int32_t* status,
                         cudaStream_t stream) {
  using SP = flash::Smem<D, DualPolicy<D>::kStageBoxes>;
  static_assert(SP::TOTAL + sizeof(flash::Barriers) + sizeof(DQBar) <= 227 * 1024,
                "dQ layout fits shared memory");
  CUtensorMap tq, tdo, tk, tv;
  const uint64_t rows = (uint64_t)batch * 2 * L;
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)hq, rows};
    const uint64_t str[2] = {(uint64_t)D * 2, (uint64_t)hq * D * 2};
    const uint32_t box[3] = {64, 1, BQ};
    if (!encode_tmap_bf16(&tq, q, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_tmap_bf16(&tdo, do_bf, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)hkv, rows};
    const uint64_t str[2] = {(uint64_t)D * 2, (uint64_t)hkv * D * 2};
    const uint32_t box[3] = {64, 1, BKV};
    if (!encode_tmap_bf16(&tk, k, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_tmap_bf16(&tv, v, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  DQArgs da{{batch, L, B, hq, hkv, hq / hkv, (L + BQ - 1) / BQ, scale * 1.4426950408889634f,
             status, nullptr, 0},
            scale, lse, drow, dq};
  const long long items = (long long)da.f.nqt * 2 * hq * batch;
  static std::atomic<int> attr[64];
  const cudaError_t ea = set_smem_limit_once(dual_dq_kernel<D>, SP::TOTAL, attr);
  if (ea != cudaSuccess) return ea;
  const long long ctas = std::min<long long>(items, num_sms());
  dual_dq_kernel<D><<<(unsigned)ctas, DQ_THREADS, SP::TOTAL, stream>>>(tq, tdo, tk, tv, da);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_tc(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* o,
                      int batch, int L, int B, int hq, int hkv, float scale,
                      int32_t* status, float* lse, cudaStream_t stream) {
  using S = flash::Smem<D>;
  CUtensorMap tq, tk, tv, to;
  const uint64_t rows = (uint64_t)batch * 2 * L;
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)hq, rows};
    const uint64_t str[2] = {(uint64_t)D * 2, (uint64_t)hq * D * 2};
    const uint32_t box[3] = {64, 1, BQ};
    if (!encode_tmap_bf16(&tq, q, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)hkv, rows};
    const uint64_t str[2] = {(uint64_t)D * 2, (uint64_t)hkv * D * 2};
    const uint32_t box[3] = {64, 1, BKV};
    if (!encode_tmap_bf16(&tk, k, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_tmap_bf16(&tv, v, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)hq, (uint64_t)L, (uint64_t)batch * 2};
    const uint64_t str[3] = {(uint64_t)D * 4, (uint64_t)hq * D * 4, (uint64_t)L * hq * D * 4};
    const uint32_t box[4] = {32, 1, BQ, 1};
    // without O (a statistics-only run) the map is encoded over lse and never used
    const void* base = o ? static_cast<const void*>(o) : static_cast<const void*>(lse);
    if (!encode_tmap_f32(&to, base, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  DualArgs a{batch, L, B, hq, hkv, hq / hkv, (L + BQ - 1) / BQ,
             scale * 1.4426950408889634f, status, lse, o != nullptr};
  const long long items = (long long)a.nqt * 2 * hq * batch;
  using SP = flash::Smem<D, DualPolicy<D>::kStageBoxes>;
  static_assert(SP::TOTAL + sizeof(flash::Barriers) + sizeof(DualEpi) <= 227 * 1024,
                "persistent layout: Q, both rings and the staging fit shared memory");
  static std::atomic<int> attr[64];
  const cudaError_t ea = set_smem_limit_once(dual_stream_persistent_kernel<D>, SP::TOTAL, attr);
  if (ea != cudaSuccess) return ea;
  const long long ctas = std::min<long long>(items, num_sms());
  dual_stream_persistent_kernel<D><<<(unsigned)ctas, DUAL_THREADS, SP::TOTAL, stream>>>(
      tq, tk, tv, to, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dual_stream(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               float* o, int batch, int L, int B, int hq, int hkv, int d,
                               float scale, int32_t* status, cudaStream_t stream, float* lse) {
  if (!o && !lse) return cudaErrorInvalidValue;
  cudaError_t e =
      d == 64 ? launch_tc<64>(q, k, v, o, batch, L, B, hq, hkv, scale, status, lse, stream)
              : launch_tc<128>(q, k, v, o, batch, L, B, hq, hkv, scale, status, lse, stream);
  count_launches(1);
  return e;
}

cudaError_t launch_dual_stream_dq(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  const uint16_t* do_bf, const float* lse, const float* drow,
                                  float* dq, int batch, int L, int B, int hq, int hkv, int d,
                                  float scale, int32_t* status, cudaStream_t stream) {
  cudaError_t e = d == 64 ? launch_dq_tc<64>(q, k, v, do_bf, lse, drow, dq, batch, L, B, hq, hkv,
                                             scale, status, stream)
                          : launch_dq_tc<128>(q, k, v, do_bf, lse, drow, dq, batch, L, B, hq,
                                              hkv, scale, status, stream);
  count_launches(1);
  return e;
}

}  // namespace mars
