// Plain tcgen05 GEMM with an fp32 output, for the products of the LM-head gradient:
//   dh = dlogits W        (M = rows, N = hidden, K = vocab; A K-major, B MN-major)
//   dW = dlogits^T h      (M = vocab, N = hidden, K = rows; A and B MN-major)
// with dlogits [rows, vocab], W [vocab, hidden] and h [rows, hidden] all row-major bf16.
// Neither operand is copied or transposed in memory: a K-major tile is one TMA box of
// [128 or 256 rows][64 K] and an MN-major tile is 64-element-wide boxes of [64 K rows][64 MN]
// (128-byte swizzle either way), and the instruction descriptor's major bits tell the
// tensor core which it is.
//
// From two row blocks on it runs in the paired form described below.
// Persistent, warp-specialised CTA (one per SM, 192 threads), as the LM-head GEMM:
//   warp 0      TMA producer: the A and B tiles of each 64-deep K block into a 4-stage
//               ring (48 KB per stage);
//   warp 1      TMEM owner and MMA issuer: 4 x tcgen05.mma (M128 N256 K16) per K block
//               into one of two 256-column fp32 accumulators;
//   warps 2..5  epilogue: thread = accumulator row, 32 columns per tcgen05.ld, written to
//               C with 16-byte stores while the issuer fills the other accumulator.
// Tiles run column block fastest, so the CTAs running at the same time cover every column
// block of about 152 / num_n row blocks: each A tile is streamed from HBM once and shared
// through L2 by the CTAs of its row block, and each B tile by those of its column block.
#pragma once

#include "sm100.cuh"

namespace mars {
namespace gemm_tc {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr int TMEM_COLS = 512;                  // 2 accumulators x 256 fp32 columns
constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + 1024;   // + alignment slack
constexpr uint32_t MN_REGION = BK * 128;        // one [64 K rows][64 MN] box: 8 KB

// Paired form (gemm_pair_kernel, two-CTA clusters): the pair computes a 256 x 256 tile of C
// with tcgen05.mma.cta_group::2 (M256 N256 K16) issued by the even CTA. Each CTA loads its
// own 128 rows of A and 128 of the 256 columns of B, k-blocks of 128 (two 64-deep halves,
// each laid out as the one-CTA form's k-block), into a 3-stage ring of 64 KB; both halves
// of a stage are counted on the even CTA's barrier, and each CTA writes its own rows of C.
constexpr int BK_P = 128, STAGES_P = 3;
constexpr int HALF_BYTES_P = 128 * BK * 2;      // one 64-deep half of a 128-row tile: 16 KB
constexpr int OPER_BYTES_P = 2 * HALF_BYTES_P;  // a 128-row operand tile, 128 deep: 32 KB
constexpr int STAGE_BYTES_P = 2 * OPER_BYTES_P; // A and B: 64 KB
static_assert(STAGES_P * STAGE_BYTES_P == STAGES * STAGE_BYTES, "both rings fill the same space");
constexpr int MAX_STAGES = STAGES_P > STAGES ? STAGES_P : STAGES;

struct Params {
  int M, N, K;
  // paired: num_tiles counts (row-block pair, column block) tiles and num_k 128-deep blocks
  int num_m, num_n, num_k, num_tiles;
  float* c;              // [M, ldc] fp32, row-major (written)
  int ldc;
  int32_t* status;
};

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, each operand K- or MN-major;
// M = 128, or 256 over a CTA pair.
__host__ __device__ constexpr uint32_t idesc(bool a_mn_major, bool b_mn_major, int m = BM) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

// Shared-memory descriptor of K step k (16 deep) of an operand tile at byte address base.
//   K-major: rows of 64 K elements (128 B) in 1024-byte groups of 8 rows; a K step moves
//            32 bytes along the row.
//   MN-major: 64-element-wide MN regions of [64 K rows][128 B], MN_REGION bytes apart; a
//            K step moves 16 rows (2048 bytes).
template <bool MN_MAJOR>
MARS_DEV uint64_t operand_desc(uint32_t base, int k) {
  return MN_MAJOR ? sm100::sdesc_sw128(base + k * 2048, MN_REGION, 1024)
                  : sm100::sdesc_sw128(base + k * 32, 16, 1024);
}

// One operand tile of `rows` MN rows (128 for A, 256 for B) for K block kb into dst:
// a K-major map has box {64 K, rows}; an MN-major map has box {64 MN, 64 K}.
template <bool MN_MAJOR>
MARS_DEV void load_operand(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int mn0,
                           int kb, int rows) {
  if (MN_MAJOR) {
    for (int r = 0; r < rows / 64; ++r)
      sm100::tma_load_2d(dst + r * MN_REGION, map, bar, mn0 + r * 64, kb * BK);
  } else {
    sm100::tma_load_2d(dst, map, bar, kb * BK, mn0);
  }
}

// The same into this CTA's shared memory with the bytes counted on the even CTA's barrier
// (its cluster address), for the paired form.
template <bool MN_MAJOR>
MARS_DEV void load_operand_pair(uint8_t* dst, const CUtensorMap* map, uint32_t bar, int mn0,
                                int kb, int rows) {
  if (MN_MAJOR) {
    for (int r = 0; r < rows / 64; ++r)
      sm100::tma_load_2d_pair(dst + r * MN_REGION, map, bar, mn0 + r * 64, kb * BK);
  } else {
    sm100::tma_load_2d_pair(dst, map, bar, kb * BK, mn0);
  }
}

template <bool A_MN, bool B_MN, bool PAIR>
MARS_DEV void gemm_body(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const Params& p) {
  using namespace sm100;
  constexpr int NST = PAIR ? STAGES_P : STAGES;
  constexpr int SB = PAIR ? STAGE_BYTES_P : STAGE_BYTES;
  // (the callers' B is MN-major, whose boxes are 64 rows in either form)
  static_assert(!PAIR || B_MN, "the paired form loads B as MN-major boxes");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[MAX_STAGES], empty_bar[MAX_STAGES];
  __shared__ uint64_t acc_full[2], acc_empty[2], drain_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int issued_s, consumed_s;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* stage_ptr = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the CTA pair (cluster) and this CTA's rank in it: rank 0 issues the MMAs
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int cid = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ncl = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    abort_s = 0;
    issued_s = 0;
    consumed_s = 0;
    // paired: rank 0's full barriers count both CTAs' bytes; its acc_empty both CTAs'
    // epilogue threads
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], PAIR ? 2 * EPI_THREADS : EPI_THREADS);
    }
    mbar_init(&drain_bar, 1);
    fence_barrier_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
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
        const int mr = tile / p.num_n, nb = tile - (tile / p.num_n) * p.num_n;
        const int mb = PAIR ? 2 * mr + (int)rank : mr;   // past the last: loads zeros
        for (int kb = 0; kb < p.num_k; ++kb, ++it) {
          const int s = it % NST;
          const uint32_t ph = (it / NST) & 1;
          if (!(ok = mbar_wait_suspending(&empty_bar[s], ph ^ 1, &abort_s, p.status))) break;
          uint8_t* a = stage_ptr + s * SB;
          if (PAIR) {
            const uint32_t fb = cluster_addr(&full_bar[s], 0);
            if (rank == 0) mbar_arrive_expect_tx(&full_bar[s], 2 * SB);
            for (int h = 0; h < BK_P / BK; ++h) {
              load_operand_pair<A_MN>(a + h * HALF_BYTES_P, &tm_a, fb, mb * BM, kb * 2 + h, BM);
              load_operand_pair<B_MN>(a + OPER_BYTES_P + h * HALF_BYTES_P, &tm_b, fb,
                                      nb * BN + (int)rank * (BN / 2), kb * 2 + h, BN / 2);
            }
          } else {
            mbar_arrive_expect_tx(&full_bar[s], SB);
            load_operand<A_MN>(a, &tm_a, &full_bar[s], mb * BM, kb, BM);
            load_operand<B_MN>(a + A_BYTES, &tm_b, &full_bar[s], nb * BN, kb, BN);
          }
          issued_s = it + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && rank == 0) {
      constexpr uint32_t kIdesc = idesc(A_MN, B_MN, PAIR ? 2 * BM : BM);
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
          if (PAIR) {
            const uint32_t b = a + OPER_BYTES_P;
#pragma unroll
            for (int k = 0; k < BK_P / 16; ++k) {
              const uint32_t h = (uint32_t)(k >> 2) * HALF_BYTES_P;
              mma_bf16_ss_pair(d_tmem, operand_desc<A_MN>(a + h, k & 3),
                               operand_desc<B_MN>(b + h, k & 3), kIdesc, (kb | k) != 0);
            }
            mma_commit_pair(&empty_bar[s], 0x3);   // frees the stage in both CTAs
          } else {
            const uint32_t b = a + A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma_bf16_ss(d_tmem, operand_desc<A_MN>(a, k), operand_desc<B_MN>(b, k), kIdesc,
                          (kb | k) != 0);
            mma_commit(&empty_bar[s]);     // frees the stage once these MMAs finish
          }
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
      const int mr = tile / p.num_n, nb = tile - (tile / p.num_n) * p.num_n;
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
      const int row = mb * BM + row_in_tile;
      const int col0 = nb * BN;
      float* crow = p.c + (size_t)(row < p.M ? row : 0) * p.ldc;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(taddr + c * 32, r);
        tmem_ld_wait();
        const int cb = col0 + c * 32;
        if (row < p.M && cb < p.N) {
          if (cb + 32 <= p.N) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(crow + cb + e) =
                  make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                              __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (cb + e < p.N) crow[cb + e] = __uint_as_float(r[e]);
          }
        }
      }
      release_acc(buf);
    }
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

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
            Params p) {
  gemm_body<A_MN, B_MN, false>(tm_a, tm_b, p);
}

// Paired form: the grid is a whole number of two-CTA clusters.
template <bool A_MN, bool B_MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a,
                 const __grid_constant__ CUtensorMap tm_b, Params p) {
  gemm_body<A_MN, B_MN, true>(tm_a, tm_b, p);
}

}  // namespace gemm_tc
}  // namespace mars
