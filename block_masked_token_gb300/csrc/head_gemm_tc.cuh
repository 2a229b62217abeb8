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
//               tcgen05.ld, online max / argmax / sum-exp, one 16-byte store per row.
// Tiles are ordered in groups of up to 16 row blocks (2048 rows): inside a group the row
// block is fastest, so the CTAs running at the same time share one W tile through L2, and
// the group's rows of h (at most 14.7 MB at hidden 3584) stay in L2 while the group sweeps
// the vocabulary. W therefore streams from HBM once per group (once per call for decode
// batches), and h once in all.
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

struct Params {
  int rows, hidden, vocab;
  int num_m, num_n, num_k, num_tiles;
  float4* part;          // [num_n][rows] {max, sumexp, argmax bits, target logit or 0}
  const int32_t* targets;  // [rows] vocabulary index per row, or NULL (no target logits)
  // Gradient mode (dlogits != NULL): instead of the partials, the epilogue writes
  // dlogits[r, v] = (exp(l_rv - row_lse[r]) - [v == y_r]) * row scale, in bf16, where the
  // row scale is stream_scale[(r % two_l) >= two_l / 2] for rows with a valid target, 0
  // otherwise.
  uint16_t* dlogits;       // [rows, vocab] bf16
  const float* row_lse;    // [rows]
  const float* stream_scale;   // [2]: clean rows, masked rows
  int two_l;
  int32_t* status;
};

// Row block and vocabulary tile of linear tile index `tile` (see the order above).
MARS_DEV void tile_coords(int tile, const Params& p, int& mb, int& nb) {
  const int per_group = GROUP_M * p.num_n;
  const int g = tile / per_group;
  const int gm = min(GROUP_M, p.num_m - g * GROUP_M);    // row blocks in this group
  const int local = tile - g * per_group;
  mb = g * GROUP_M + local % gm;
  nb = local / gm;
}

// static: every translation unit that launches it gets its own copy
static __global__ void __launch_bounds__(NUM_THREADS, 1)
head_gemm_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                 Params p) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ uint64_t acc_full[2], acc_empty[2], drain_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int issued_s, consumed_s;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* stage_ptr = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_s = 0;
    issued_s = 0;
    consumed_s = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], EPI_THREADS);
    }
    mbar_init(&drain_bar, 1);
    fence_barrier_init();
    prefetch_tmap(&tm_h);
    prefetch_tmap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = __shfl_sync(0xffffffffu, tmem_base_s, 0);   // warp-uniform

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, p, mb, nb);
        for (int kb = 0; kb < p.num_k; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!(ok = mbar_wait(&empty_bar[s], ph ^ 1, &abort_s, p.status))) break;
          uint8_t* a = stage_ptr + s * STAGE_BYTES;
          mbar_arrive_expect_tx(&full_bar[s], STAGE_BYTES);
          tma_load_2d(a, &tm_h, &full_bar[s], kb * BK, mb * BM);
          tma_load_2d(a + A_BYTES, &tm_w, &full_bar[s], kb * BK, nb * BN);
          issued_s = it + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, BN, false);
      int it = 0, t = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x, ++t) {
        const int buf = t & 1;
        const uint32_t aph = (t >> 1) & 1;
        if (!(ok = mbar_wait(&acc_empty[buf], aph ^ 1, &abort_s, p.status))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = 0; kb < p.num_k; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!(ok = mbar_wait(&full_bar[s], ph, &abort_s, p.status))) break;
          tc_fence_after();
          const uint32_t a = smem_u32(stage_ptr + s * STAGE_BYTES);
          const uint32_t b = a + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            mma_bf16_ss(d_tmem, sdesc_sw128(a + k * 32, 16, 1024),
                        sdesc_sw128(b + k * 32, 16, 1024), idesc, (kb | k) != 0);
          }
          mma_commit(&empty_bar[s]);       // frees the stage once these MMAs finish
          consumed_s = it + 1;
        }
        if (ok) mma_commit(&acc_full[buf]);
      }
      // make sure no MMA is still in flight when the CTA tears down
      mma_commit(&drain_bar);
      mbar_wait(&drain_bar, 0, nullptr, p.status);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int quad = warp & 3;                 // TMEM lane quadrant of this warp
    const int row_in_tile = quad * 32 + lane;
    int t = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++t) {
      int mb, nb;
      tile_coords(tile, p, mb, nb);
      const int buf = t & 1;
      const uint32_t aph = (t >> 1) & 1;
      // warp-uniform result: the tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], aph, &abort_s, p.status))) break;
      tc_fence_after();
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
        uint16_t* drow = p.dlogits + (size_t)(row < p.rows ? row : 0) * p.vocab + col0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(taddr + c * 32, r);
          tmem_ld_wait();
          if (row < p.rows && c * 32 < ncols) {
            uint32_t g2[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              float g0 = exp2f(fmaf(__uint_as_float(r[j]), kLog2e, nl));
              float g1 = exp2f(fmaf(__uint_as_float(r[j + 1]), kLog2e, nl));
              if (c * 32 + j == tcol) g0 -= 1.f;
              if (c * 32 + j + 1 == tcol) g1 -= 1.f;
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(g0 * scale, g1 * scale);
              g2[j >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            if (c * 32 + 32 <= ncols && (p.vocab % 8) == 0) {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(drow + c * 32 + q * 8) =
                    make_uint4(g2[4 * q], g2[4 * q + 1], g2[4 * q + 2], g2[4 * q + 3]);
            } else {
              for (int j = 0; j < 32 && c * 32 + j < ncols; ++j)
                drow[c * 32 + j] = (uint16_t)((g2[j >> 1] >> ((j & 1) * 16)) & 0xffffu);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
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
          ssum *= exp2f((m - cm) * kLog2e);
          m = cm;
          am = ca;
        }
        if (m != -INFINITY) {
          const float mb2 = m * kLog2e;
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = (c * 32 + j < ncols) ? __uint_as_float(r[j]) : -INFINITY;
            acc += exp2f(fmaf(x, kLog2e, -mb2));
          }
          ssum += acc;
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
      if (row < p.rows)
        p.part[(size_t)nb * p.rows + row] = make_float4(m, ssum, __int_as_float(am), tl);
    }
  }

  __syncthreads();
  // drain: if a wait gave up, wait (bounded) for TMA loads still in flight
  if (threadIdx.x == 0 && abort_s) {
    for (int it = consumed_s; it < issued_s; ++it)
      mbar_wait(&full_bar[it % STAGES], (it / STAGES) & 1, nullptr, p.status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace head_tc
}  // namespace mars
