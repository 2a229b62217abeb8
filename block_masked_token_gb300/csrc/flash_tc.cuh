// Flash-attention tile engine on tcgen05 shared by the dual-stream and decode kernels.
//
// A CTA runs a 128-row query tile held in shared memory over a list of 128-key tiles.
// Roles, as the decode kernel lays them out (256 threads):
//   warp 0      Q loader, then K loader: K tiles into a 3-stage ring (TMA, 128-byte
//               swizzle); warp 6 streams V tiles into their own ring (2 stages, 3 in the
//               decode kernel), so the two rings advance independently;
//   warp 1      TMEM owner and QK^T issuer: S_j = Q K_j^T into one of three 128-column
//               fp32 TMEM buffers; a K stage is released as soon as its QK^T finishes;
//   warp 7      PV issuer: O += P_j V_j with O and P in TMEM (P is the A operand, read
//               from TMEM); a V stage is released after its PV;
//   warps 2..5  softmax: thread = query row. It reads its S_j row (tcgen05.ld) into
//               registers, takes the row max, and writes P = exp2(S - m) as bf16 pairs
//               over the upper half of that S buffer (tcgen05.st). The running max is
//               raised lazily: O and l are rescaled (tcgen05.ld / st) only when the max
//               grows by more than 2^8, which keeps P <= 256 and the result exact up to
//               rounding.
// The two issuers (s_issuer, pv_issuer) run independently, so the softmax of tile j
// overlaps QK^T of later tiles and the PV of earlier ones. A kernel may instead let one
// thread issue both (mma_loop: S_j, then PV_{j-1}); the decode kernel does, its tile lists
// being short. The functions take warp
// roles from their caller, and the softmax derives its TMEM lane quadrant from warp & 3,
// so a kernel may place the roles differently: the persistent dual-stream kernel runs
// them as warpgroups and adds epilogue warps (staged_epilogue).
#pragma once

#include "sm100.cuh"

namespace mars {
namespace flash {

constexpr int BQ = 128;                    // query rows per CTA tile
constexpr int BKV = 128;                   // keys per tile
constexpr int NUM_THREADS = 256;          // 8 warps, roles below
constexpr int V_LOADER_WARP = 6;
constexpr int PV_ISSUER_WARP = 7;
constexpr int SOFTMAX_THREADS = 128;
constexpr float kRescaleLog2 = 8.0f;       // lazy max: rescale when it grows by > 2^8

// Ring depths of the K and V tile rings (with Q and a 32 KB O staging area they fill the
// 227 KB of shared memory).
#ifndef MARS_K_STAGES
#define MARS_K_STAGES 3
#endif
#ifndef MARS_V_STAGES
#define MARS_V_STAGES 2
#endif
constexpr int K_STAGES = MARS_K_STAGES;
constexpr int V_STAGES = MARS_V_STAGES;
constexpr int NBUF = 3;                    // S/P buffers in TMEM
constexpr int kMaxVStages = 4;             // V-ring barriers kept (a kernel may use fewer)

// VST: V-ring depth of the kernel (the decode kernel, whose CTAs stream long key lists
// with no O staging area, runs a deeper V ring than the default).
template <int D, int STAGE_BOXES = 0, int VST = V_STAGES>
struct Smem {
  static_assert(VST >= 1 && VST <= kMaxVStages, "V ring depth");
  static constexpr int Q_BYTES = BQ * D * 2;         // D/64 swizzled regions of [128][64]
  static constexpr int KV_BYTES = BKV * D * 2;       // one K or V tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = Q_BYTES;                          // K ring
  static constexpr int OFF_V = OFF_K + K_STAGES * KV_BYTES;      // V ring
  static constexpr int OFF_STAGE = OFF_V + VST * KV_BYTES;       // O staging (optional)
  static constexpr int TOTAL = OFF_STAGE + STAGE_BOXES * BQ * 128 + 1024;   // + alignment slack
  // TMEM columns: three S buffers (fp32) at 0, 128, 256 and O (fp32) at 384. P of a tile
  // (bf16 pairs, 64 columns) is written over the upper half of that tile's S buffer once
  // the softmax has read S; PV reads it from there.
  static constexpr int TMEM_S = 0;
  static constexpr int TMEM_O = NBUF * BKV;
  static constexpr int P_OFF = BKV / 2;              // P inside an S buffer
  static constexpr int TMEM_COLS = 512;
};

struct Barriers {
  uint64_t q_full;
  uint64_t k_full[K_STAGES], k_empty[K_STAGES], v_full[kMaxVStages], v_empty[kMaxVStages];
  uint64_t s_full[NBUF];
  uint64_t p_full[NBUF], pv_done[NBUF];
  uint64_t o_final, drain, drain_pv;
  uint64_t o_staged;      // softmax threads have written O to shared memory (staged store)
  uint64_t stage_free;    // the stores of the previous staging round have read it
  uint64_t q_empty;       // the QK^T MMAs of an item have completed (Q may be replaced)
  uint64_t epi_ready;     // softmax threads have handed over 1/l of their rows (hand-off)
  uint64_t epi_taken;     // epilogue threads have taken that hand-off (hand-off)
  uint64_t o_free;        // epilogue threads have read O out of TMEM (hand-off)
  uint32_t tmem_base;
  int abort;
};

// Thread 0: initialise every barrier (call before the CTA-wide sync that publishes them).
MARS_DEV void init_barriers(Barriers& bar) {
  using namespace sm100;
  bar.abort = 0;
  mbar_init(&bar.q_full, 1);
  for (int i = 0; i < K_STAGES; ++i) {
    mbar_init(&bar.k_full[i], 1);
    mbar_init(&bar.k_empty[i], 1);
  }
  for (int i = 0; i < kMaxVStages; ++i) {
    mbar_init(&bar.v_full[i], 1);
    mbar_init(&bar.v_empty[i], 1);
  }
  for (int i = 0; i < NBUF; ++i) {
    mbar_init(&bar.s_full[i], 1);
    mbar_init(&bar.p_full[i], SOFTMAX_THREADS);
    mbar_init(&bar.pv_done[i], 1);
  }
  mbar_init(&bar.o_staged, SOFTMAX_THREADS);
  mbar_init(&bar.stage_free, 1);
  mbar_init(&bar.q_empty, 1);
  mbar_init(&bar.epi_ready, SOFTMAX_THREADS);
  mbar_init(&bar.epi_taken, SOFTMAX_THREADS);
  mbar_init(&bar.o_free, SOFTMAX_THREADS);
  mbar_init(&bar.o_final, 1);
  mbar_init(&bar.drain, 1);
  mbar_init(&bar.drain_pv, 1);
  fence_barrier_init();
}

// Loader skeleton shared by the kernels: one warp streams one ring (the K ring or the V
// ring; the two run independently, so a slow V slot never holds back a K load). Lane 0
// waits for a free stage and arms its barrier with the tile's byte count, then every lane
// calls `issue(j, dst, bar)` (the kernel decides which lanes issue the TMA copies of tile
// j into dst, completing on bar). Returns after waiting (bounded) for every copy it
// issued, so the CTA never exits with copies in flight.
// j0: ring position of tile 0 (tiles of earlier work items of a persistent CTA); last[st]
// keeps the ring position of the latest copy into each stage, across calls, for the final
// drain (drain = true on the last call).
template <int D, int NST, class Issue>
MARS_DEV bool load_ring_n(Barriers& bar, uint64_t* full, uint64_t* empty, uint8_t* ring,
                          int ntiles, int j0, int (&last)[NST], bool drain, int32_t* status,
                          Issue& issue) {
  using namespace sm100;
  using S = Smem<D>;
  const int lane = threadIdx.x & 31;
  volatile int* ab = &bar.abort;
  bool good = true;
  for (int j = 0; j < ntiles; ++j) {
    const int jg = j0 + j;
    const int st = jg % NST;
    int ok = 1;
    if (lane == 0) {
      ok = mbar_wait(&empty[st], ((jg / NST) & 1) ^ 1, ab, status);
      if (ok) mbar_arrive_expect_tx(&full[st], S::KV_BYTES);
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) {
      good = false;
      break;
    }
    issue(j, ring + st * S::KV_BYTES, &full[st]);
    last[st] = jg;
  }
  if ((drain || !good) && lane == 0) {
    for (int st = 0; st < NST; ++st)
      if (last[st] >= 0) mbar_wait(&full[st], (last[st] / NST) & 1, nullptr, status);
  }
  __syncwarp();
  return good;
}

// One work item's K (or V) tiles into its ring; see load_ring_n. Returns false on abort.
template <int D, int NST, class Issue>
MARS_DEV bool load_ring_item(Barriers& bar, uint8_t* smem, int ntiles, int j0, int (&last)[NST],
                             bool drain, int32_t* status, bool is_v, Issue issue) {
  using S = Smem<D>;
  return is_v ? load_ring_n<D, NST>(bar, bar.v_full, bar.v_empty, smem + S::OFF_V, ntiles, j0,
                                    last, drain, status, issue)
              : load_ring_n<D, NST>(bar, bar.k_full, bar.k_empty, smem + S::OFF_K, ntiles, j0,
                                    last, drain, status, issue);
}

template <int D, int VST = V_STAGES, class Issue>
MARS_DEV void load_ring(Barriers& bar, uint8_t* smem, int ntiles, int32_t* status, bool is_v,
                        Issue issue) {
  if (is_v) {
    int last[VST];
    for (int i = 0; i < VST; ++i) last[i] = -1;
    load_ring_item<D, VST>(bar, smem, ntiles, 0, last, true, status, true, issue);
  } else {
    int last[K_STAGES];
    for (int i = 0; i < K_STAGES; ++i) last[i] = -1;
    load_ring_item<D, K_STAGES>(bar, smem, ntiles, 0, last, true, status, false, issue);
  }
}

// Row-visibility of a query row: keys jg (in the kernel's key index space) with
// jg < lo1_end, or lo2 <= jg <= hi2, are visible.
struct RowVis {
  int end1;     // first range [0, end1)
  int lo2, hi2; // second range [lo2, hi2]
};

MARS_DEV bool visible(const RowVis& v, int jg) {
  return jg < v.end1 || (jg >= v.lo2 && jg <= v.hi2);
}

// Visible columns of one row inside one key tile: [0, e1) or [s2, e2], restricted to the
// 16-key groups whose bit is set in pmask (pages of a paged tile; all ones otherwise).
struct ColRange {
  int e1, s2, e2;
  uint32_t pmask;
};

// Bits [lo, hi) of a 32-bit word (lo, hi clamped to [0, 32]).
MARS_DEV uint32_t bit_range(int lo, int hi) {
  lo = max(0, min(32, lo));
  hi = max(0, min(32, hi));
  if (hi <= lo) return 0u;
  const uint32_t upto_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
  const uint32_t upto_lo = (1u << lo) - 1u;
  return upto_hi & ~upto_lo;
}

// Visibility bits of columns 32c .. 32c+31 for one row.
MARS_DEV uint32_t chunk_mask(const ColRange& cr, int c) {
  const int base = c * 32;
  uint32_t mk = bit_range(0, cr.e1 - base) | bit_range(cr.s2 - base, cr.e2 + 1 - base);
  const uint32_t pg = cr.pmask >> (2 * c);            // two 16-key pages per chunk
  mk &= ((pg & 1u) ? 0x0000ffffu : 0u) | ((pg & 2u) ? 0xffff0000u : 0u);
  return mk;
}

// Swizzled byte offset of 16-byte chunk `chunk` (0..7) of row `r` inside a [rows][128 B]
// region (the layout TMA writes with 128-byte swizzle).
MARS_DEV uint32_t sw_off(int r, int chunk) {
  return (uint32_t)(r * 128 + ((chunk ^ (r & 7)) << 4));
}

MARS_DEV uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The MMAs are issued by two threads (tcgen05.mma issue blocks until the tensor pipe
// accepts the instruction, so a single issuer leaves the pipe idle whenever it waits on a
// barrier; with two, one thread's waits overlap the other's MMAs). Each commits only its
// own MMAs. ntiles >= 1 for both.

// QK^T issuer: S_j = Q K_j^T into S buffer j % NBUF.
// j0: global position of tile 0 in the rings and S buffers; q_parity: phase of q_full
// holding this item's Q. Returns false on abort.
template <int D>
MARS_DEV bool s_issuer(Barriers& bar, uint8_t* smem, int ntiles, uint32_t tmem,
                       int32_t* status, int j0 = 0, uint32_t q_parity = 0) {
  using namespace sm100;
  using S = Smem<D>;
  const uint32_t idesc_s = idesc_bf16_f32(BQ, BKV, false);   // S = Q K^T: B K-major
  const uint32_t q = smem_u32(smem + S::OFF_Q);
  volatile int* ab = &bar.abort;
  if (!mbar_wait(&bar.q_full, q_parity, ab, status)) return false;
  for (int jl = 0; jl < ntiles; ++jl) {
    const int j = j0 + jl;
    const int st = j % K_STAGES, sb = j % NBUF;
    if (!mbar_wait(&bar.k_full[st], (j / K_STAGES) & 1, ab, status)) return false;
    // S buffer sb last held tile j-NBUF, whose P the PV of that tile read from it
    if (j >= NBUF && !mbar_wait(&bar.pv_done[sb], ((j / NBUF) - 1) & 1, ab, status))
      return false;
    tc_fence_after();
    const uint64_t qd = sdesc_sw128(q, 16, 1024);
    const uint64_t kd = sdesc_sw128(smem_u32(smem + S::OFF_K + st * S::KV_BYTES), 16, 1024);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k >> 2) * (BQ * 128) + (k & 3) * 32;
      const uint32_t koff = (k >> 2) * (BKV * 128) + (k & 3) * 32;
      mma_bf16_ss(tmem + S::TMEM_S + sb * BKV, sdesc_advance(qd, off), sdesc_advance(kd, koff),
                  idesc_s, k != 0);
    }
    mma_commit(&bar.s_full[sb]);
    mma_commit(&bar.k_empty[st]);      // K stage free once this QK^T completes
  }
  return true;
}

// PV issuer: O += P_j V_j (P from the upper half of S buffer j % NBUF), then o_final.
// With o_free_parity >= 0 the first PV (which overwrites O) waits until the epilogue
// warps have read the previous item's O (the hand-off form).
template <int D>
MARS_DEV bool pv_issuer(Barriers& bar, uint8_t* smem, int ntiles, uint32_t tmem,
                        int32_t* status, int j0 = 0, int o_free_parity = -1) {
  using namespace sm100;
  using S = Smem<D>;
  const uint32_t idesc_o = idesc_bf16_f32(BQ, D, true);      // O = P V: B MN-major
  volatile int* ab = &bar.abort;
  for (int jl = 0; jl < ntiles; ++jl) {
    const int j = j0 + jl;
    const int pb = j % NBUF, st = j % V_STAGES;
    if (!mbar_wait(&bar.v_full[st], (j / V_STAGES) & 1, ab, status)) return false;
    if (!mbar_wait(&bar.p_full[pb], (j / NBUF) & 1, ab, status)) return false;
    if (jl == 0 && o_free_parity >= 0 &&
        !mbar_wait(&bar.o_free, (uint32_t)o_free_parity, ab, status))
      return false;
    tc_fence_after();
    // B = V [keys x D], MN-major: D/64 atoms of BKV*128 B, 8-key groups of 1024 B
    const uint64_t vd = sdesc_sw128(smem_u32(smem + S::OFF_V + st * S::KV_BYTES), BKV * 128, 1024);
#pragma unroll
    for (int k = 0; k < BKV / 16; ++k) {
      // A = P [128 rows x 128 keys] in TMEM: row = lane, 16 keys = 8 columns per K step
      const uint32_t a = tmem + S::TMEM_S + pb * BKV + S::P_OFF + k * 8;
      const uint64_t bd = sdesc_advance(vd, k * 2048);
      mma_bf16_ts(tmem + S::TMEM_O, a, bd, idesc_o, (jl | k) != 0);
    }
    mma_commit(&bar.pv_done[pb]);
    mma_commit(&bar.v_empty[st]);
  }
  mma_commit(&bar.o_final);
  return true;
}

// Single-thread alternative: one thread issues S_j, then PV_{j-1}, so the QK^T the softmax
// waits for is never queued behind PV work (used where the softmax is on the critical
// path). ntiles >= 1; VST is the V-ring depth the loaders use.
template <int D, int VST = V_STAGES>
MARS_DEV void mma_loop(Barriers& bar, uint8_t* smem, int ntiles, uint32_t tmem,
                       int32_t* status) {
  using namespace sm100;
  using S = Smem<D>;
  const uint32_t idesc_s = idesc_bf16_f32(BQ, BKV, false);   // S = Q K^T: B K-major
  const uint32_t idesc_o = idesc_bf16_f32(BQ, D, true);      // O = P V:   B MN-major
  const uint32_t q = smem_u32(smem + S::OFF_Q);
  volatile int* ab = &bar.abort;
  if (!mbar_wait(&bar.q_full, 0, ab, status)) return;
  auto issue_pv = [&](int j) -> bool {
    const int pb = j % NBUF, st = j % VST;
    if (!mbar_wait(&bar.v_full[st], (j / VST) & 1, ab, status)) return false;
    if (!mbar_wait(&bar.p_full[pb], (j / NBUF) & 1, ab, status)) return false;
    tc_fence_after();
    // B = V [keys x D], MN-major: D/64 atoms of BKV*128 B, 8-key groups of 1024 B
    const uint64_t vd = sdesc_sw128(smem_u32(smem + S::OFF_V + st * S::KV_BYTES), BKV * 128, 1024);
#pragma unroll
    for (int k = 0; k < BKV / 16; ++k) {
      // A = P [128 rows x 128 keys] in TMEM: row = lane, 16 keys = 8 columns per K step
      const uint32_t a = tmem + S::TMEM_S + pb * BKV + S::P_OFF + k * 8;
      const uint64_t bd = sdesc_advance(vd, k * 2048);
      mma_bf16_ts(tmem + S::TMEM_O, a, bd, idesc_o, (j | k) != 0);
    }
    mma_commit(&bar.pv_done[pb]);
    mma_commit(&bar.v_empty[st]);
    return true;
  };
  for (int j = 0; j < ntiles; ++j) {
    const int st = j % K_STAGES, sb = j % NBUF;
    if (!mbar_wait(&bar.k_full[st], (j / K_STAGES) & 1, ab, status)) return;
    // S buffer sb last held tile j-NBUF, whose P the PV of that tile read from it
    if (j >= NBUF && !mbar_wait(&bar.pv_done[sb], ((j / NBUF) - 1) & 1, ab, status)) return;
    tc_fence_after();
    const uint64_t qd = sdesc_sw128(q, 16, 1024);
    const uint64_t kd = sdesc_sw128(smem_u32(smem + S::OFF_K + st * S::KV_BYTES), 16, 1024);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k >> 2) * (BQ * 128) + (k & 3) * 32;
      const uint32_t koff = (k >> 2) * (BKV * 128) + (k & 3) * 32;
      mma_bf16_ss(tmem + S::TMEM_S + sb * BKV, sdesc_advance(qd, off), sdesc_advance(kd, koff),
                  idesc_s, k != 0);
    }
    mma_commit(&bar.s_full[sb]);
    mma_commit(&bar.k_empty[st]);      // K stage free once this QK^T completes
    if (j > 0 && !issue_pv(j - 1)) return;
  }
  if (!issue_pv(ntiles - 1)) return;
  mma_commit(&bar.o_final);
}

// Single-issuer form (run by lane 0 of warp 1): mma_loop, then a wait (bounded) for its
// own MMAs so none is in flight when the CTA tears down.
template <int D, int VST = V_STAGES>
MARS_DEV void single_issuer(Barriers& bar, uint8_t* smem, int ntiles, uint32_t tmem,
                            int32_t* status) {
  using namespace sm100;
  mma_loop<D, VST>(bar, smem, ntiles, tmem, status);
  mma_commit(&bar.drain);
  mbar_wait(&bar.drain, 0, nullptr, status);
}

MARS_DEV float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

MARS_DEV float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of one row's 128 S values (fp32 bits), scaled to log2 units: 8 independent
// chains of three-input max, then a short tree.
MARS_DEV float row_max_log2(const uint32_t (&r)[BKV], float scale_log2) {
  float pm[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) pm[i] = fmaxf(__uint_as_float(r[i]), __uint_as_float(r[8 + i]));
#pragma unroll
  for (int k = 2; k < BKV / 8; k += 2)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      pm[i] = max3f(pm[i], __uint_as_float(r[k * 8 + i]), __uint_as_float(r[(k + 1) * 8 + i]));
  return fmaxf(max3f(pm[0], pm[1], pm[2]), max3f(max3f(pm[3], pm[4], pm[5]), pm[6], pm[7])) *
         scale_log2;
}

// P = exp2(S * scale_log2 - m) for 64 S values starting at r[c0], packed as 32 bf16 pairs
// (even key in the low half); the fp32 values are added to acc (two lanes per float2).
// The scale-and-shift and the sums run as packed f32x2 operations.
MARS_DEV void exp2_pack64(const uint32_t (&r)[BKV], int c0, float scale_log2, float neg_m,
                          uint32_t (&packed)[32], float2 (&acc)[2]) {
  const float2 sc = make_float2(scale_log2, scale_log2), sh = make_float2(neg_m, neg_m);
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    const float2 t = __ffma2_rn(make_float2(__uint_as_float(r[c0 + e]), __uint_as_float(r[c0 + e + 1])),
                                sc, sh);
    const float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    packed[e >> 1] = pack_bf16x2(p.x, p.y);
    acc[(e >> 1) & 1] = __fadd2_rn(acc[(e >> 1) & 1], p);
  }
}

// Softmax + final normalisation for one query row per thread (threads 64..191).
// Policy provides: row_valid(row), row_vis(row), tile(j) -> Tile (with .full set when
// every row sees every key of tile j, so no per-key test runs), cols(vis, tile) ->
// ColRange (the columns of tile j visible to the row; a tile must admit only keys it
// owns, so no key is counted twice), with kRowStats row_stats(row, m, l) once the row is
// done, and either store_chunk(row, col, 32 fp32 of O, 1/l, m, l) or, with kHandOff,
// hand_off(row, 1/l) for the epilogue warps (staged_epilogue below).
// Each tile's S row is read from TMEM once (4 loads, one wait) into registers.
//
// A persistent kernel calls it once per work item with j0 (global position of the item's
// first tile) and o_parity (phase of o_final for the item, used without hand-off).
template <int D, class Policy>
MARS_DEV bool softmax_loop(Barriers& bar, uint8_t* smem, const Policy& pol, int ntiles,
                           uint32_t tmem, float scale_log2, int32_t* status, int j0 = 0,
                           uint32_t o_parity = 0) {
  using namespace sm100;
  using S = Smem<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int row = quad * 32 + lane;               // TMEM lane = query row of the tile
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  volatile int* ab = &bar.abort;
  const bool rv = pol.row_valid(row);
  const RowVis vis = pol.row_vis(row);
  float m = -INFINITY;                            // running max (log2 units, lazy)
  float l = 0.f;
  bool ok = true;
  // tcgen05.ld / st are warp-collective (.sync.aligned): every branch around them below is
  // warp-uniform, and so is every wait result (warp_wait).
  auto warp_wait = [&](uint64_t* b, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(b, parity, ab, status));
  };
  // tile descriptors are computed one tile ahead (for paged tiles this reads the block
  // table, whose latency then overlaps the wait for the next S)
  typename Policy::Tile next_tile = pol.tile(0);
  for (int j = 0; j < ntiles && ok; ++j) {
    const int jg = j0 + j;
    const int sb = jg % NBUF;
    const typename Policy::Tile tile = next_tile;
    if (j + 1 < ntiles) next_tile = pol.tile(j + 1);
    if (!(ok = warp_wait(&bar.s_full[sb], (jg / NBUF) & 1))) break;
    tc_fence_after();
    const uint32_t s_addr = tmem + S::TMEM_S + sb * BKV + lane_off;
    uint32_t r[BKV];
#pragma unroll
    for (int c = 0; c < BKV / 32; ++c)
      tmem_ld32(s_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(r + c * 32));
    tmem_ld_wait();
    if (!rv || !tile.full) {
      // visible columns of this row in this tile: [0, e1) or [s2, e2], on mapped pages
      // (none for a padding row past the end of the query tile)
      const ColRange cr = rv ? pol.cols(vis, tile) : ColRange{0, BKV, -1, 0u};
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c) {
        const uint32_t mk = chunk_mask(cr, c);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (!((mk >> e) & 1u)) r[c * 32 + e] = 0xff800000u;
      }
    }
    const float tmax = row_max_log2(r, scale_log2);
    // lazy rescale of O and l: a row raises its max only when it grows by more than 2^8.
    // Rows whose O already holds keys (m finite) rescale it in TMEM; the TMEM pass runs
    // for the whole warp when any of its rows needs it (alpha = 1 for the others).
    const bool raise = tmax > m + kRescaleLog2;
    const bool rescale_o = raise && m != -INFINITY;
    if (__any_sync(0xffffffffu, rescale_o)) {
      // PV of the previous tile must have landed in O before O is rescaled
      if (!(ok = warp_wait(&bar.pv_done[(jg - 1) % NBUF], ((jg - 1) / NBUF) & 1))) break;
      tc_fence_after();
      const float alpha = rescale_o ? ex2_approx(m - tmax) : 1.f;
      l *= alpha;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + S::TMEM_O + c * 32 + lane_off, o);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st32(tmem + S::TMEM_O + c * 32 + lane_off, o);
      }
      tmem_st_wait();
    }
    if (raise) m = tmax;
    // P = exp2(S*scale - m) -> bf16 pairs over the upper half of this tile's S buffer (S is
    // in registers now; row = lane, the A operand of the PV MMA), and the row sum
    const uint32_t p_addr = tmem + S::TMEM_S + sb * BKV + S::P_OFF + lane_off;
    const float neg_m = (m == -INFINITY) ? 0.f : -m;   // no visible key yet: all P are 0
    float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int h = 0; h < BKV / 64; ++h) {               // 64 keys = 32 columns per store
      uint32_t packed[32];
      exp2_pack64(r, h * 64, scale_log2, neg_m, packed, acc);
      tmem_st32(p_addr + h * 32, packed);
    }
    l += (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive_warp(&bar.p_full[sb]);
  }
  if (!ok) return false;
  if constexpr (Policy::kRowStats) pol.row_stats(row, m, l);
  const float inv = (l > 0.f) ? 1.f / l : 0.f;
  if constexpr (Policy::kHandOff) {
    // the epilogue warps read O and store it; these threads go on to the next item. A
    // short item can finish here before the epilogue has got to the previous one: hand
    // over only once that one's hand-off has been taken, so epi_ready never runs two
    // phases ahead of its waiter.
    if (pol.item > 0 && !warp_wait(&bar.epi_taken, (uint32_t)(pol.item - 1) & 1)) return false;
    pol.hand_off(row, inv);
    mbar_arrive_warp(&bar.epi_ready);
    return true;
  } else {
    if (!warp_wait(&bar.o_final, o_parity)) return false;
    tc_fence_after();
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tmem + S::TMEM_O + c * 32 + lane_off, o);
      tmem_ld_wait();
      if (rv) pol.store_chunk(row, c * 32, o, inv, m, l);
    }
    return true;
  }
}

// Epilogue warps of the hand-off form (one warp per TMEM lane quadrant, thread = row): per
// work item, once the softmax threads have handed over 1/l (epi_ready) and the last PV has
// completed (o_final), read O out of TMEM, release it to the next item's first PV
// (o_free), and write O/l to shared memory as 32-column boxes of [128 rows][32 fp32] in the
// 128-byte swizzled layout (a quarter-warp's 16-byte stores then hit distinct banks). One
// thread (store_thread) writes them out with TMA stores, kStageBoxes boxes per round;
// before a round overwrites the staging it waits until the previous round's stores have
// read it and releases the others through stage_free. er counts rounds across items; the
// caller drains the last stores (bulk_wait_read_all on store_thread) before exiting.
template <int D, class Policy>
MARS_DEV bool staged_epilogue(Barriers& bar, uint8_t* smem, const Policy& pol, uint32_t tmem,
                              uint32_t parity, float inv, int& er, int store_thread,
                              int32_t* status) {
  using namespace sm100;
  using S = Smem<D>;
  const int lane = threadIdx.x & 31;
  const int row = ((threadIdx.x >> 5) & 3) * 32 + lane;
  const uint32_t lane_off = (uint32_t)(row & ~31) << 16;
  volatile int* ab = &bar.abort;
  auto warp_wait = [&](uint64_t* b, uint32_t par) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(b, par, ab, status));
  };
  constexpr int NBOX = D / 32;
  constexpr int PER = Policy::kStageBoxes;
  static_assert(NBOX % PER == 0, "rounds cover O");
  if (!warp_wait(&bar.o_final, parity)) return false;
  tc_fence_after();
  uint32_t o[D];                                     // the whole O row: one TMEM wait
#pragma unroll
  for (int c = 0; c < NBOX; ++c)
    tmem_ld32(tmem + S::TMEM_O + c * 32 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(o + c * 32));
  tmem_ld_wait();
  tc_fence_before();
  mbar_arrive_warp(&bar.o_free);
  uint8_t* stage = pol.stage(smem);
#pragma unroll
  for (int b0 = 0; b0 < NBOX; b0 += PER) {
    if (er > 0) {
      if ((int)threadIdx.x == store_thread) {
        bulk_wait_read_all();
        mbar_arrive(&bar.stage_free);
      }
      if (!warp_wait(&bar.stage_free, (er - 1) & 1)) return false;
    }
#pragma unroll
    for (int c = 0; c < PER; ++c) {
      uint8_t* box = stage + c * (BQ * 128);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t* v = o + (b0 + c) * 32 + 4 * q;
        *reinterpret_cast<float4*>(box + sw_off(row, q)) =
            make_float4(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv,
                        __uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv);
      }
    }
    fence_proxy_async_smem();
    mbar_arrive_warp(&bar.o_staged);
    bool st_ok = true;
    if ((int)threadIdx.x == store_thread) {
      st_ok = mbar_wait(&bar.o_staged, er & 1, ab, status);
      if (st_ok) {
        pol.store_boxes(stage, b0, PER);
        bulk_commit();
      }
    }
    if (!__all_sync(0xffffffffu, st_ok)) return false;
    ++er;
  }
  return true;
}

}  // namespace flash
}  // namespace mars
