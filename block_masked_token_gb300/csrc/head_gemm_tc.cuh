// tcgen05 LM-head GEMM with the max / sum-exp / argmax reduction fused into its epilogue.
//
// logits[r, v] = sum_k h[r, k] * W[v, k] for a 128-row x 256-column tile lives only in
// TMEM; the epilogue reduces it to one partial {tile max, sum exp(l - tile max), first
// argmax, and the row's target logit when a target index falls in the tile} per (row,
// vocabulary tile), and the logits never reach global memory.
//
// Persistent, warp-specialised CTA (one per SM, 192 threads):
//   warp 0      TMA producer: h tile [128 x 64] and W tile [256 x 64] per k-block into a
//               4-stage ring (48 KB per stage, 128-byte swizzle);
//   warp 1      TMEM owner and MMA issuer: 4 x tcgen05.mma (M128 N256 K16) per k-block,
//               into one of two 256-column fp32 accumulators;
//   warps 2..5  epilogue: thread = accumulator row (TMEM lane), 256 columns read with
//               tcgen05.ld, online max / argmax / sum-exp, one 16-byte store per row
//               (the gradient mode instead stages bf16 dlogits boxes for TMA stores).
// Paired form (head_gemm_pair_kernel, two-CTA clusters): the pair computes a 256 x 256
// tile with tcgen05.mma.cta_group::2 (M256 N256 K16) issued by the even CTA; each CTA
// loads its own 128 rows of h and half of the W tile, k-blocks of 128 as two 64-column
// boxes each, into a 3-stage ring of 64 KB, both halves counted on the even CTA's
// barrier, and each CTA's epilogue reads its own rows.
// Tiles are ordered in groups of up to 16 row blocks (2048 rows): inside a group the row
// block is fastest, so the CTAs running at the same time share one W tile through L2, and
// the group's rows of h (at most 14.7 MB at hidden 3584) stay in L2 while the group sweeps
// the vocabulary. W therefore streams from HBM once per group (once per call for decode
// batches), and h once in all.
//
// Fused acceptance (the decode step, Params::sync set): within a group a CTA meets only a
// few row blocks (every gcd(grid, rows of the group)-th), so instead of one partial per
// tile the epilogue keeps one running partial per row and row block in shared memory
// over all of the CTA's tiles of the group, and writes it once, as a record, when the CTA
// leaves the group. Each record adds the number of vocabulary tiles it covers to its row
// block's count (an atomic ticket): the CTA whose record completes the count merges the
// row block's records (at most one per CTA), writes tokens and max-probs, and runs the
// left-to-right scan of every sequence whose rows lie in the block. A sequence whose rows
// straddle two row blocks is scanned by the second of the two merging CTAs (a second
// ticket per block boundary). Nothing waits on another CTA, and no second kernel runs.
#pragma once

#include <cuda_bf16.h>

#include "sm100.cuh"

namespace mars {
namespace head_tc {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr int TMEM_COLS = 512;                  // 2 accumulators x 256 fp32 columns
constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + 1024;   // + alignment slack
constexpr float kLog2e = 1.4426950408889634f;

constexpr int GROUP_M = 16;                     // row blocks per tile group
// running partials of the fused acceptance: [GROUP_M][BM] float4 after the ring
constexpr size_t SLOT_BYTES = (size_t)GROUP_M * BM * sizeof(float4);   // 32 KB
constexpr size_t SMEM_FUSED_BYTES = SMEM_BYTES + SLOT_BYTES;

// Paired form (head_gemm_pair_kernel): a cluster of two CTAs computes a 256-row x 256-column
// tile with two-SM MMAs (M256 N256 K16). Each CTA loads its own 128 rows of h and one half
// (128 vocabulary rows) of the W tile, so a CTA fills a third less shared memory per unit
// of MMA work. Its k-blocks are 128 wide (two 64-column boxes per operand), three 64 KB
// stages in the same space: fewer stage hand-offs per tile than six stages of 32 KB. The
// even CTA issues the MMAs; each CTA's epilogue reads its own 128 rows.
constexpr int GROUP_P = GROUP_M / 2;            // row-block pairs per tile group
constexpr int STAGES_P = 3;
constexpr int BK_P = 128;
constexpr int A_BYTES_P = BM * BK_P * 2;        // 32 KB: two [128][64] regions
constexpr int B_HALF_BYTES = (BN / 2) * BK_P * 2;       // 32 KB
constexpr int STAGE_BYTES_P = A_BYTES_P + B_HALF_BYTES;
static_assert(STAGES_P * STAGE_BYTES_P == STAGES * STAGE_BYTES, "both rings fill the same space");
constexpr int MAX_STAGES = STAGES_P > STAGES ? STAGES_P : STAGES;

struct Params {
  int rows, hidden, vocab;
  // num_tiles counts (row block, vocabulary tile) tiles, or in the paired form (row-block
  // pair, vocabulary tile) tiles, num_mp = (num_m + 1) / 2 pairs
  int num_m, num_n, num_k, num_tiles, num_mp;
  float4* part;          // [num_n][rows] {max, sumexp, argmax bits, target logit or 0}
  const int32_t* targets;  // [rows] vocabulary index per row, or NULL (no target logits)
  // Gradient mode (dlogits != NULL): instead of the partials, the epilogue writes
  // dlogits[r, v] = (exp(l_rv - row_lse[r]) - [v == y_r]) * row scale, in bf16, where the
  // row scale is stream_scale[(r % two_l) >= two_l / 2] for rows with a valid target, 0
  // otherwise.
  // It is written through the kernel's third tensor map (box 64 columns x 128 rows,
  // 128-byte swizzle, so vocab % 8 == 0), each box staged in the 32 KB after the ring,
  // which the launch then includes.
  uint16_t* dlogits;       // [rows, vocab] bf16
  const float* row_lse;    // [rows]
  const float* stream_scale;   // [2]: clean rows, masked rows
  int two_l;
  int32_t* status;
  // Fused acceptance mode (sync != NULL; part, targets and dlogits unused): counters
  // sync[0 .. num_m) = vocabulary tiles merged into records per row block, sync[num_m ..
  // 2 num_m) = records per row block, sync[2 num_m .. 3 num_m) = tickets of the boundary
  // between row blocks mb - 1 and mb; all zero at launch. rec[mb][i][row] = record i of
  // row block mb (at most max_rec, one per CTA) {max, sum exp(l - max), first argmax, 0}.
  uint32_t* sync;
  float4* rec;
  int max_rec;
  int B;                 // block positions per sequence (rows s*B .. s*B + B - 1)
  float tau;             // threshold, or per sequence from taus when taus != NULL
  const float* taus;
  int32_t* tokens;       // [rows]
  float* maxprob;        // [rows]
  int32_t* n_accept;     // [rows / B]
};

// 2^x on the special-function unit (ex2.approx.ftz: relative error about 2^-22, -inf -> 0),
// for the per-logit exponentials of the epilogues.
MARS_DEV float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (max, sum exp(l - max), lowest argmax) of the union of two sets of logits
MARS_DEV void merge_partial(float& m, float& s, int& a, float m2, float s2, int a2) {
  const float mx = fmaxf(m, m2);
  if (mx == -INFINITY) return;
  const float sm = (m == -INFINITY ? 0.f : s * exp2f((m - mx) * kLog2e)) +
                   (m2 == -INFINITY ? 0.f : s2 * exp2f((m2 - mx) * kLog2e));
  a = m > m2 ? a : (m2 > m ? a2 : min(a, a2));
  m = mx;
  s = sm;
}

// Left-to-right acceptance of sequence s from its B max-probs p[0..B-1]: the leading run
// of positions with p >= tau, at least 1 (a NaN threshold compares false).
MARS_DEV int accept_run(const float* pr, int B, float t) {
  int n = 0;
  while (n < B && pr[n] >= t) ++n;
  return n < 1 ? 1 : n;
}

// Row block (row-block pair when PAIR) and vocabulary tile of linear tile index `tile` (see
// the order above; a group is 16 row blocks, i.e. 8 pairs).
template <bool PAIR>
MARS_DEV void tile_coords(int tile, const Params& p, int& mr, int& nb) {
  constexpr int GR = PAIR ? GROUP_P : GROUP_M;
  const int nm = PAIR ? p.num_mp : p.num_m;
  const int per_group = GR * p.num_n;
  const int g = tile / per_group;
  const int gm = min(GR, nm - g * GR);                   // row blocks (pairs) in this group
  const int local = tile - g * per_group;
  mr = g * GR + local % gm;
  nb = local / gm;
}

// The kernel body, one-CTA (PAIR false) or paired form. tm_w's box is 256 vocabulary rows,
// or 128 in the paired form.
template <bool PAIR>
MARS_DEV void head_gemm_body(const CUtensorMap& tm_h, const CUtensorMap& tm_w,
                             const CUtensorMap& tm_d, const Params& p) {
  using namespace sm100;
  constexpr int NST = PAIR ? STAGES_P : STAGES;
  constexpr int SB = PAIR ? STAGE_BYTES_P : STAGE_BYTES;
  constexpr int KB = PAIR ? BK_P : BK;
  constexpr int AB = PAIR ? A_BYTES_P : A_BYTES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[MAX_STAGES], empty_bar[MAX_STAGES];
  __shared__ uint64_t acc_full[2], acc_empty[2], drain_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int issued_s, consumed_s;
  // fused acceptance: vocabulary tiles per running slot, broadcasts, merged max-probs
  __shared__ uint32_t slot_tiles_s[GROUP_M];
  __shared__ int rec_idx_s, last_s;
  __shared__ float p_s[BM];
  __shared__ uint64_t epi_bar;               // the four epilogue warps among themselves

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* stage_ptr = smem_raw + (sbase - raw);
  float4* slots = reinterpret_cast<float4*>(stage_ptr + (size_t)NST * SB);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the CTA pair (cluster) and this CTA's rank in it: rank 0 issues the MMAs
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int cid = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ncl = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    abort_s = 0;
    issued_s = 0;
    consumed_s = 0;
    for (int i = 0; i < GROUP_M; ++i) slot_tiles_s[i] = 0;
    // paired: rank 0's full barriers count the bytes of both CTAs' halves of a stage
    // (rank 1's are not used); rank 0's acc_empty counts both CTAs' epilogue threads
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], PAIR ? 2 * EPI_THREADS : EPI_THREADS);
    }
    mbar_init(&drain_bar, 1);
    mbar_init(&epi_bar, EPI_THREADS);
    fence_barrier_init();
    prefetch_tmap(&tm_h);
    prefetch_tmap(&tm_w);
    if (p.dlogits) prefetch_tmap(&tm_d);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(&tmem_base_s, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&tmem_base_s, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the peer's barriers are initialised before any arrival or commit reaches them
  if (PAIR) cluster_sync();
  const uint32_t tmem_base = __shfl_sync(0xffffffffu, tmem_base_s, 0);   // warp-uniform

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = cid; tile < p.num_tiles && ok; tile += ncl) {
        int mr, nb;
        tile_coords<PAIR>(tile, p, mr, nb);
        // this CTA's row block, and its vocabulary rows of the tile (paired: one half;
        // a row block past the last loads zeros and is skipped by the epilogue)
        const int mb = PAIR ? 2 * mr + (int)rank : mr;
        const int wrow = nb * BN + (PAIR ? (int)rank * (BN / 2) : 0);
        for (int kb = 0; kb < p.num_k; ++kb, ++it) {
          const int s = it % NST;
          const uint32_t ph = (it / NST) & 1;
          if (!(ok = mbar_wait_suspending(&empty_bar[s], ph ^ 1, &abort_s, p.status))) break;
          uint8_t* a = stage_ptr + s * SB;
          if (PAIR) {
            // both halves of the stage land on rank 0's barrier, which expects them both
            const uint32_t fb = cluster_addr(&full_bar[s], 0);
            if (rank == 0) mbar_arrive_expect_tx(&full_bar[s], 2 * SB);
            for (int x = 0; x < KB / 64; ++x) {
              tma_load_2d_pair(a + x * (BM * 128), &tm_h, fb, kb * KB + x * 64, mb * BM);
              tma_load_2d_pair(a + AB + x * ((BN / 2) * 128), &tm_w, fb, kb * KB + x * 64, wrow);
            }
          } else {
            mbar_arrive_expect_tx(&full_bar[s], SB);
            tma_load_2d(a, &tm_h, &full_bar[s], kb * BK, mb * BM);
            tma_load_2d(a + A_BYTES, &tm_w, &full_bar[s], kb * BK, wrow);
          }
          issued_s = it + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = idesc_bf16_f32(PAIR ? 2 * BM : BM, BN, false);
      int it = 0, t = 0;
      bool ok = true;
      for (int tile = cid; tile < p.num_tiles && ok; tile += ncl, ++t) {
        const int buf = t & 1;
        const uint32_t aph = (t >> 1) & 1;
        if (!(ok = mbar_wait_suspending(&acc_empty[buf], aph ^ 1, &abort_s, p.status))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = 0; kb < p.num_k; ++kb, ++it) {
          const int s = it % NST;
          const uint32_t ph = (it / NST) & 1;
          if (!(ok = mbar_wait_suspending(&full_bar[s], ph, &abort_s, p.status))) break;
          tc_fence_after();
          const uint32_t a = smem_u32(stage_ptr + s * SB);
          const uint32_t b = a + AB;
#pragma unroll
          for (int k = 0; k < KB / 16; ++k) {
            if (PAIR)
              mma_bf16_ss_pair(d_tmem,
                               sdesc_sw128(a + (k >> 2) * (BM * 128) + (k & 3) * 32, 16, 1024),
                               sdesc_sw128(b + (k >> 2) * ((BN / 2) * 128) + (k & 3) * 32, 16, 1024),
                               idesc, (kb | k) != 0);
            else
              mma_bf16_ss(d_tmem, sdesc_sw128(a + k * 32, 16, 1024),
                          sdesc_sw128(b + k * 32, 16, 1024), idesc, (kb | k) != 0);
          }
          // frees the stage (in both CTAs) once these MMAs finish
          if (PAIR) mma_commit_pair(&empty_bar[s], 0x3);
          else mma_commit(&empty_bar[s]);
          consumed_s = it + 1;
        }
        if (ok) {
          if (PAIR) mma_commit_pair(&acc_full[buf], 0x3);
          else mma_commit(&acc_full[buf]);
        }
      }
      // make sure no MMA is still in flight when the CTA tears down
      if (PAIR) mma_commit_pair(&drain_bar, 0x1);
      else mma_commit(&drain_bar);
      mbar_wait_suspending(&drain_bar, 0, nullptr, p.status);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int quad = warp & 3;                 // TMEM lane quadrant of this warp
    const int row_in_tile = quad * 32 + lane;
    const bool leader = threadIdx.x == 64;     // one thread of the four epilogue warps

    // Fused acceptance. The epilogue warps synchronise among themselves on an mbarrier
    // with the bounded wait (not a named barrier), so that a CTA whose pipeline gave up
    // cannot leave some of them waiting for ever.
    uint32_t epi_phase = 0;
    auto epi_sync = [&]() -> bool {
      mbar_arrive(&epi_bar);
      const bool ok = mbar_wait_suspending(&epi_bar, epi_phase & 1u, &abort_s, p.status);
      ++epi_phase;
      return ok;
    };

    // All rows of row block mb are merged: write tokens and max-probs, scan the sequences
    // inside the block, and take the block's boundary tickets.
    auto merge_block = [&](int mb) -> bool {
      __threadfence();
      const int nrec = min((int)atomicAdd(&p.sync[p.num_m + mb], 0u), p.max_rec);
      float m = -INFINITY, ssum = 0.f;
      int am = 0x7fffffff;
      const float4* rb = p.rec + (size_t)mb * p.max_rec * BM + row_in_tile;
      for (int i = 0; i < nrec; ++i) {
        const float4 v = __ldcg(rb + (size_t)i * BM);
        merge_partial(m, ssum, am, v.x, v.y, __float_as_int(v.z));
      }
      const float pr = 1.f / ssum;
      const int r0 = mb * BM;
      const int row = r0 + row_in_tile;
      if (row < p.rows) {
        p.tokens[row] = am;
        p.maxprob[row] = pr;
      }
      p_s[row_in_tile] = pr;
      __threadfence();
      if (!epi_sync()) return false;
      const int r1 = min(p.rows, r0 + BM);
      for (int sq = (r0 + p.B - 1) / p.B + row_in_tile; sq < r1 / p.B; sq += BM)
        p.n_accept[sq] = accept_run(p_s + (sq * p.B - r0), p.B, p.taus ? p.taus[sq] : p.tau);
      if (leader) {
        // a sequence straddling this block's first or last row: the second of the two
        // blocks to get here scans it from the max-probs both have written
        float pr2[32];
        for (int side = 0; side < 2; ++side) {
          const int edge = side == 0 ? r0 : r0 + BM;       // first row of the later block
          if (edge <= 0 || edge >= p.rows || edge % p.B == 0) continue;
          if (atomicAdd(&p.sync[2 * p.num_m + edge / BM], 1u) != 1u) continue;
          __threadfence();
          const int sq = edge / p.B;
          for (int k = 0; k < p.B; ++k) pr2[k] = __ldcg(p.maxprob + (size_t)sq * p.B + k);
          p.n_accept[sq] = accept_run(pr2, p.B, p.taus ? p.taus[sq] : p.tau);
        }
      }
      return epi_sync();                 // p_s is rewritten by the next merge
    };

    // The CTA leaves group g: write its running partials of the group as records and add
    // their vocabulary tiles to the row blocks' counts.
    auto flush_group = [&](int g, uint32_t visited) -> bool {
      for (uint32_t vm = visited; vm; vm &= vm - 1) {
        const int l = __ffs(vm) - 1;
        const int mb = g * GROUP_M + l;
        if (leader) rec_idx_s = (int)atomicAdd(&p.sync[p.num_m + mb], 1u);
        if (!epi_sync()) return false;
        const int idx = rec_idx_s;
        if (idx < p.max_rec)             // one record per CTA and row block: always true
          p.rec[((size_t)mb * p.max_rec + idx) * BM + row_in_tile] = slots[l * BM + row_in_tile];
        __threadfence();
        if (!epi_sync()) return false;
        if (leader) {
          const uint32_t n = slot_tiles_s[l];
          slot_tiles_s[l] = 0;
          last_s = atomicAdd(&p.sync[mb], n) + n == (uint32_t)p.num_n;
        }
        if (!epi_sync()) return false;
        if (last_s && !merge_block(mb)) return false;
      }
      return true;
    };

    int cur_g = -1;
    uint32_t visited = 0;
    int dl_box = 0;                            // dlogits boxes staged so far (TMA stores)
    // this tile's accumulator may be overwritten (paired: one arrival per warp of both
    // CTAs on rank 0's barrier)
    auto release_acc = [&](int buf) {
      tc_fence_before();
      if (PAIR) {
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(cluster_addr(&acc_empty[buf], 0), 32);
      } else {
        mbar_arrive(&acc_empty[buf]);
      }
    };
    int t = 0;
    for (int tile = cid; tile < p.num_tiles; tile += ncl, ++t) {
      int mr, nb;
      tile_coords<PAIR>(tile, p, mr, nb);
      const int mb = PAIR ? 2 * mr + (int)rank : mr;
      const int buf = t & 1;
      const uint32_t aph = (t >> 1) & 1;
      // warp-uniform result: the tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait_suspending(&acc_full[buf], aph, &abort_s, p.status))) break;
      tc_fence_after();
      if (PAIR && mb >= p.num_m) {             // the second half of an odd last pair: no rows
        release_acc(buf);
        continue;
      }
      const uint32_t taddr = tmem_base + buf * BN + ((uint32_t)(quad * 32) << 16);
      const int col0 = nb * BN;
      const int ncols = min(BN, p.vocab - col0);
      const int row = mb * BM + row_in_tile;
      // column of this row's target inside the tile (outside [0, ncols) when elsewhere)
      const int tcol = (p.targets && row < p.rows) ? p.targets[row] - col0 : -1;
      if (p.dlogits) {
        // gradient of the mean cross-entropy with respect to this tile of logits
        float lse = 0.f, scale = 0.f;
        if (row < p.rows) {
          const int y = p.targets[row];
          lse = p.row_lse[row];
          if (y >= 0 && y < p.vocab)
            scale = p.stream_scale[(row % p.two_l) >= p.two_l / 2 ? 1 : 0];
        }
        const float nl = -lse * kLog2e;
        // 32 columns c*32 .. c*32 + 31 of this row as 16 packed bf16 pairs
        auto grad32 = [&](int c, uint32_t (&g2)[16]) {
          uint32_t r[32];
          tmem_ld32(taddr + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float g0 = ex2_fast(fmaf(__uint_as_float(r[j]), kLog2e, nl));
            float g1 = ex2_fast(fmaf(__uint_as_float(r[j + 1]), kLog2e, nl));
            if (c * 32 + j == tcol) g0 -= 1.f;
            if (c * 32 + j + 1 == tcol) g1 -= 1.f;
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(g0 * scale, g1 * scale);
            g2[j >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
          }
        };
        // Four boxes of 64 columns, each staged as 128 rows x 128 bytes in the layout of
        // the map's 128-byte swizzle (16-byte unit q of row r at unit q ^ (r & 7)) in one
        // of two 16 KB halves of the area after the ring, and stored by one thread. Before
        // the barrier of a box the storing thread waits until its earlier stores have
        // read their halves, so the next box may overwrite the other half.
        bool ok = true;
#pragma unroll 1
        for (int bi = 0; bi < BN / 64; ++bi, ++dl_box) {
          uint8_t* half = reinterpret_cast<uint8_t*>(slots) + (dl_box & 1) * (BM * 128);
          uint8_t* srow = half + row_in_tile * 128;
#pragma unroll 1
          for (int h2 = 0; h2 < 2; ++h2) {
            const int c = bi * 2 + h2;
            uint32_t g2[16];
            grad32(c, g2);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int u = (h2 * 4 + q) ^ (row_in_tile & 7);
              *reinterpret_cast<uint4*>(srow + u * 16) =
                  make_uint4(g2[4 * q], g2[4 * q + 1], g2[4 * q + 2], g2[4 * q + 3]);
            }
          }
          fence_proxy_async_smem();
          if (leader) bulk_wait_read_all();
          if (!epi_sync()) {
            ok = false;
            break;
          }
          if (leader && col0 + bi * 64 < p.vocab) {
            tma_store_2d(&tm_d, half, col0 + bi * 64, mb * BM);
            bulk_commit();
          }
        }
        if (!ok) break;
        release_acc(buf);
        continue;
      }
      float tl = 0.f;
      float m = -INFINITY, ssum = 0.f;
      int am = 0x7fffffff;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(taddr + c * 32, r);
        tmem_ld_wait();
        const int rel = tcol - c * 32;
        if (rel >= 0 && rel < 32 && c * 32 + rel < ncols) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j == rel) tl = __uint_as_float(r[j]);
        }
        float cm = -INFINITY;
        int ca = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float x = (c * 32 + j < ncols) ? __uint_as_float(r[j]) : -INFINITY;
          if (x > cm) { cm = x; ca = col0 + c * 32 + j; }
        }
        if (cm > m) {
          ssum *= ex2_fast((m - cm) * kLog2e);
          m = cm;
          am = ca;
        }
        if (m != -INFINITY) {
          const float mb2 = m * kLog2e;
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = (c * 32 + j < ncols) ? __uint_as_float(r[j]) : -INFINITY;
            acc += ex2_fast(fmaf(x, kLog2e, -mb2));
          }
          ssum += acc;
        }
      }
      release_acc(buf);
      if (p.sync) {
        // fold this tile's partial into the running slot of its row block
        const int g = tile / ((PAIR ? GROUP_P : GROUP_M) * p.num_n);
        const int l = mb - g * GROUP_M;
        if (g != cur_g) {
          if (cur_g >= 0 && !flush_group(cur_g, visited)) break;
          cur_g = g;
          visited = 0;
        }
        float4& sl = slots[l * BM + row_in_tile];
        if ((visited >> l) & 1u) {
          float m0 = sl.x, s0 = sl.y;
          int a0 = __float_as_int(sl.z);
          merge_partial(m0, s0, a0, m, ssum, am);
          sl = make_float4(m0, s0, __int_as_float(a0), 0.f);
        } else {
          sl = make_float4(m, ssum, __int_as_float(am), 0.f);
        }
        visited |= 1u << l;
        if (leader) ++slot_tiles_s[l];
        continue;
      }
      if (row < p.rows)
        p.part[(size_t)nb * p.rows + row] = make_float4(m, ssum, __int_as_float(am), tl);
    }
    if (p.sync && cur_g >= 0 && !abort_s) flush_group(cur_g, visited);
    // the dlogits stores must have read shared memory and written global memory before exit
    if (leader) bulk_wait_all();
  }

  __syncthreads();
  // drain: if a wait gave up, wait (bounded) for TMA loads still in flight; rank 1's loads
  // complete on rank 0's barriers, so it gives them a fixed time instead
  if (threadIdx.x == 0 && abort_s) {
    if (PAIR && rank != 0) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 50000) {
      }
    } else {
      for (int it = consumed_s; it < issued_s; ++it)
        mbar_wait_suspending(&full_bar[it % NST], (it / NST) & 1, nullptr, p.status);
    }
  }
  tc_fence_before();
  __syncthreads();
  // paired: neither CTA leaves while the other may still arrive on its barriers
  if (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// static: every translation unit that launches them gets its own copy
static __global__ void __launch_bounds__(NUM_THREADS, 1)
head_gemm_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                 const __grid_constant__ CUtensorMap tm_d, Params p) {
  head_gemm_body<false>(tm_h, tm_w, tm_d, p);
}

// Paired form: the grid is a whole number of two-CTA clusters.
static __global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
head_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_h,
                      const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_d, Params p) {
  head_gemm_body<true>(tm_h, tm_w, tm_d, p);
}

}  // namespace head_tc
}  // namespace mars
