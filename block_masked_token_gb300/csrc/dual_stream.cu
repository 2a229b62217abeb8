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
  static constexpr bool kStagedStore = true;
  static constexpr bool kRowStats = true;
  static constexpr int kStageBoxes = D / 32 < 2 ? D / 32 : 2;
  const CUtensorMap* tm_o;   // O as [2*batch][L][hq][D] fp32, box [1][128][1][32]
  float* lse;                // optional: [batch][hq][2L] row log-sum-exp (log2 units)
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
  MARS_DEV uint8_t* stage(uint8_t* smem) const {
    return smem + flash::Smem<D, kStageBoxes>::OFF_STAGE;
  }
  // log2 of the row's softmax denominator in units of scale*log2(e)*score: m + log2(l)
  MARS_DEV void row_stats(int row, float m, float l) const {
    if (lse && row_valid(row))
      lse[((size_t)b * hq + h) * 2 * L + (size_t)stream * L + r0 + row] = m + log2f(l);
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

// One CTA per SM runs work items r*G + c (even rounds r) and
// r*G + G-1-c (odd rounds), G = gridDim.x, c = blockIdx.x, so heavy and light items even
// out. The rings, S buffers and barrier phases run on across items; the next item's Q is
// loaded as soon as the current item's last QK^T has completed, and its first K/V tiles
// stream in while the softmax warps write out the current item's O.
template <int D>
__global__ void __launch_bounds__(flash::NUM_THREADS, 1)
dual_stream_persistent_kernel(const __grid_constant__ CUtensorMap tm_q,
                              const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v,
                              const __grid_constant__ CUtensorMap tm_o, DualArgs a) {
  using namespace sm100;
  using Pol = DualPolicy<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ flash::Barriers bar;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tmem = cta_setup(bar, warp);
  volatile int* ab = &bar.abort;
  const int total = a.nqt * 2 * a.hq * a.batch;
  const int G = gridDim.x, c = blockIdx.x;
  auto item_id = [&](int r) { return r * G + ((r & 1) ? G - 1 - c : c); };
  const int rounds = (total + G - 1) / G;

  if (warp == 0 || warp == flash::V_LOADER_WARP) {
    const bool is_v = warp != 0;
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
  } else if (warp == 1 || warp == flash::PV_ISSUER_WARP) {
    if (lane == 0) {
      const bool pv = warp == flash::PV_ISSUER_WARP;
      int j0 = 0, i = 0, nq = 0;
      for (int r = 0; r < rounds; ++r) {
        const int id = item_id(r);
        if (id >= total) continue;
        const Pol pol = make_item<D>(a, id, &tm_o);
        if (pv) {
          if (!flash::pv_issuer<D>(bar, smem, pol.n_total, tmem, a.status, j0)) break;
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
  } else {
    int j0 = 0, i = 0, er = 0;
    for (int r = 0; r < rounds; ++r) {
      const int id = item_id(r);
      if (id >= total) continue;
      const Pol pol = make_item<D>(a, id, &tm_o);
      if (!flash::softmax_loop<D>(bar, smem, pol, pol.n_total, tmem, a.scale_log2, a.status, j0,
                                  i & 1, &er))
        break;
      j0 += pol.n_total;
      ++i;
    }
    if (threadIdx.x == 2 * 32) bulk_wait_read_all();   // last stores have read the staging
  }
  cta_teardown(tmem, warp);
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
  static_assert(SP::TOTAL + sizeof(flash::Barriers) <= 227 * 1024,
                "persistent layout: Q, both rings and the staging fit shared memory");
  static std::atomic<int> attr[64];
  const cudaError_t ea = set_smem_limit_once(dual_stream_persistent_kernel<D>, SP::TOTAL, attr);
  if (ea != cudaSuccess) return ea;
  const long long ctas = std::min<long long>(items, num_sms());
  dual_stream_persistent_kernel<D><<<(unsigned)ctas, flash::NUM_THREADS, SP::TOTAL, stream>>>(
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

}  // namespace mars
