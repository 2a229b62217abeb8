// Dual-stream (training-form) attention under the MARS mask M (papernotes.org notes of
// "MARS: Enabling Autoregressive Models Multi-Token Generation", Key design 1, eq. M,
// beta(t) = ceil(t/B); overall framework: clean stream x and masked stream x~ in one
// forward over z = [x; x~]).
//
// In 0-indexed stream-local terms a query row sees one or two contiguous key ranges:
//   clean row t (global t):    keys [0, t]
//   masked row t (global L+t): clean keys [0, B*(t/B)) and masked keys [L + B*(t/B), L + t]
// A CTA owns 128 consecutive rows of one stream for one (batch, query head) and visits
// only the 128-key tiles that intersect those ranges: for a clean tile the causal tiles
// 0..t/128, for a masked tile the clean tiles below its block start plus the tile(s)
// holding its own blocks. Fully masked tiles are never loaded; tiles every row sees in
// full skip the per-key test. The tile engine (flash_tc.cuh) runs QK^T and PV on tcgen05
// with S and O in TMEM.
#include <climits>

#include "common.cuh"
#include "flash_tc.cuh"
#include "internal.h"

namespace mars {

namespace {

using flash::BKV;
using flash::BQ;

template <int D>
struct DualPolicy {
  static constexpr bool kStagedStore = true;
  const CUtensorMap* tm_o;   // O as [2*batch][L][hq][D] fp32, box [1][128][1][32]
  int L, B, hq;
  int b, h, stream, r0;
  int n_clean, n_total, mstart, full_limit;

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
  // rows past L (a partial last query tile) fall outside the map's L extent and are not
  // written
  MARS_DEV void store_tile(const uint8_t* stage) const {
#pragma unroll
    for (int c = 0; c < D / 32; ++c)
      sm100::tma_store_4d(tm_o, stage + c * (BQ * 128), c * 32, h, r0, b * 2 + stream);
  }
};

struct DualArgs {
  int batch, L, B, hq, hkv, G, nqt;
  float scale_log2;
  int32_t* status;
};

template <int D>
__global__ void __launch_bounds__(flash::NUM_THREADS, 1)
dual_stream_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, DualArgs a) {
  using namespace sm100;
  using S = flash::Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ flash::Barriers bar;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // heaviest query tiles first
  int id = blockIdx.x;
  const int b = id % a.batch;
  id /= a.batch;
  const int h = id % a.hq;
  id /= a.hq;
  const int stream = id & 1;
  const int qt = a.nqt - 1 - (id >> 1);

  DualPolicy<D> pol;
  pol.tm_o = &tm_o;
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
  const int kvh = h / a.G;
  const int zb = b * 2 * a.L;

  if (threadIdx.x == 0) flash::init_barriers(bar);
  if (warp == 1) {
    tmem_alloc(&bar.tmem_base, S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // read once per warp and broadcast: a warp-uniform TMEM base
  const uint32_t tmem = __shfl_sync(0xffffffffu, bar.tmem_base, 0);

  // one 3D box of 128 rows per 64-column half; rows past the batch read as zeros
  auto issue = [&](const CUtensorMap* tm) {
    return [&, tm](int j, uint8_t* dst, uint64_t* b) {
      if (lane == 0) {
        const int z = zb + pol.tile_key0(j);
        for (int x = 0; x < D / 64; ++x) tma_load_3d(dst + x * (BKV * 128), tm, b, x * 64, kvh, z);
      }
    };
  };
  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar.q_full, S::Q_BYTES);
      for (int x = 0; x < D / 64; ++x)
        tma_load_3d(smem + S::OFF_Q + x * (BQ * 128), &tm_q, &bar.q_full, x * 64, h,
                    zb + stream * a.L + pol.r0);
    }
    flash::load_ring<D>(bar, smem, pol.n_total, a.status, false, issue(&tm_k));
    if (lane == 0) mbar_wait(&bar.q_full, 0, nullptr, a.status);
  } else if (warp == flash::V_LOADER_WARP) {
    flash::load_ring<D>(bar, smem, pol.n_total, a.status, true, issue(&tm_v));
  } else if (warp == 1 || warp == flash::PV_ISSUER_WARP) {
    if (lane == 0)
      flash::issuer<D, true>(bar, smem, pol.n_total, tmem, a.status,
                             warp == flash::PV_ISSUER_WARP);
  } else {
    flash::softmax_loop<D>(bar, smem, pol, pol.n_total, tmem, a.scale_log2, a.status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S::TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_tc(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* o,
                      int batch, int L, int B, int hq, int hkv, float scale,
                      int32_t* status, cudaStream_t stream) {
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
    if (!encode_tmap_f32(&to, o, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  DualArgs a{batch, L, B, hq, hkv, hq / hkv, (L + BQ - 1) / BQ,
             scale * 1.4426950408889634f, status};
  static std::atomic<int> attr[64];
  const cudaError_t ea = set_smem_limit_once(dual_stream_tc_kernel<D>, S::TOTAL, attr);
  if (ea != cudaSuccess) return ea;
  const long long ctas = (long long)a.nqt * 2 * hq * batch;
  dual_stream_tc_kernel<D><<<(unsigned)ctas, flash::NUM_THREADS, S::TOTAL, stream>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dual_stream(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               float* o, int batch, int L, int B, int hq, int hkv, int d,
                               float scale, int32_t* status, cudaStream_t stream) {
  cudaError_t e = d == 64 ? launch_tc<64>(q, k, v, o, batch, L, B, hq, hkv, scale, status, stream)
                          : launch_tc<128>(q, k, v, o, batch, L, B, hq, hkv, scale, status, stream);
  count_launches(1);
  return e;
}

}  // namespace mars
