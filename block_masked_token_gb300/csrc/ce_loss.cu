// Dual-stream training loss L = L_mask + L_AR over the 2L positions of z = [x; x~]
// (papernotes.org notes of "MARS: Enabling Autoregressive Models Multi-Token Generation",
// Key design 2: the masked-stream loss plus the clean-stream next-token loss; gist.science
// explainer, 2.B "Combined Loss").
//
// For every row r of h (sequence s, stream position t < 2L) with a target index y_r,
// ce_r = logsumexp_v(l_rv) - l_{r y_r}, l = h W^T. L_AR is the mean of ce_r over the
// clean-stream rows (t < L) that carry a target, L_mask the mean over the masked-stream
// rows (t >= L) that carry one; rows with target -1 are left out. Which positions carry a
// target (the masked set, the right shift of the clean targets) is the caller's choice.
//
// Kernel 1 is the LM-head GEMM of head_gemm_tc.cuh, whose epilogue already reduces each
// 128 x 256 logit tile to {max, sum exp, argmax} per row and here also keeps the target's
// logit when it falls in the tile; the logits never reach memory. Kernel 2 merges the
// partials of each row into ce_r; kernel 3 reduces the rows of each stream in a fixed
// order (float64 accumulation), so the loss does not depend on scheduling.
//
// Gradient: dL/dl_rv = (softmax(l_r)_v - [v = y_r]) / N_x for a row of stream x with a
// target (N_x = that stream's rows with a target), 0 for the others. The head GEMM is run
// again with an epilogue that writes this dlogits tile in bf16 (using the forward's
// per-row log-sum-exp), then the tcgen05 GEMM of gemm_tc.cuh forms dh = dlogits W and
// dW = dlogits^T h from it in place (fp32 accumulation and output): W and h are read as
// MN-major operands and, for dW, dlogits as well, so nothing is transposed in memory.
#include "common.cuh"
#include "gemm_tc.cuh"
#include "head_gemm_tc.cuh"
#include "internal.h"

namespace mars {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// One warp per row.
__global__ void __launch_bounds__(256) ce_rows_kernel(const float4* __restrict__ part,
                                                      const int32_t* __restrict__ targets,
                                                      int rows, int nvt, int vocab,
                                                      float* __restrict__ row_ce,
                                                      float* __restrict__ row_lse,
                                                      int32_t* status) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float m = -INFINITY;
  for (int t = lane; t < nvt; t += 32) m = fmaxf(m, part[(size_t)t * rows + row].x);
  m = warp_max(m);
  float se = 0.f;
  for (int t = lane; t < nvt; t += 32) {
    const float4 v = part[(size_t)t * rows + row];
    se += v.y * exp2f((v.x - m) * kLog2e);
  }
  se = warp_sum(se);
  if (lane == 0) {
    const int y = targets[row];
    const float lse = m + log2f(se) * kLn2;
    if (row_lse) row_lse[row] = lse;
    float ce = 0.f;
    if (y >= 0 && y < vocab) {
      ce = lse - part[(size_t)(y / head_tc::BN) * rows + row].w;
    } else if (y != -1) {
      if (status) atomicOr(status, MARS_ST_BADTARGET);
    }
    row_ce[row] = ce;
  }
}

// One CTA: for each stream (0 clean, 1 masked) the mean of ce over its rows with a valid
// target, summed in a fixed order in float64. loss = {L_mask, L_AR, L_mask + L_AR}; a
// stream without any target contributes 0.
__global__ void __launch_bounds__(256) ce_reduce_kernel(const float* __restrict__ row_ce,
                                                        const int32_t* __restrict__ targets,
                                                        int batch, int L, int vocab,
                                                        float* __restrict__ loss) {
  __shared__ double s_sum[256];
  __shared__ int s_cnt[256];
  float mean[2];
  const long long n = (long long)batch * L;
  for (int stream = 0; stream < 2; ++stream) {
    double sum = 0.0;
    int cnt = 0;
    for (long long i = threadIdx.x; i < n; i += blockDim.x) {
      const long long s = i / L, t = i % L;
      const long long r = s * 2 * L + (long long)stream * L + t;
      const int y = targets[r];
      if (y >= 0 && y < vocab) {
        sum += (double)row_ce[r];
        ++cnt;
      }
    }
    s_sum[threadIdx.x] = sum;
    s_cnt[threadIdx.x] = cnt;
    __syncthreads();
    for (int o = blockDim.x / 2; o > 0; o >>= 1) {
      if (threadIdx.x < o) {
        s_sum[threadIdx.x] += s_sum[threadIdx.x + o];
        s_cnt[threadIdx.x] += s_cnt[threadIdx.x + o];
      }
      __syncthreads();
    }
    mean[stream] = s_cnt[0] ? (float)(s_sum[0] / s_cnt[0]) : 0.f;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    loss[0] = mean[1];
    loss[1] = mean[0];
    loss[2] = mean[1] + mean[0];
  }
}

// One CTA: the number of rows with a valid target in each stream; scale = 1 / count (0 for
// a stream without targets).
__global__ void __launch_bounds__(256) ce_scale_kernel(const int32_t* __restrict__ targets,
                                                       int batch, int L, int vocab,
                                                       float* __restrict__ scale) {
  __shared__ int s_cnt[2][256];
  int cnt[2] = {0, 0};
  const long long rows = (long long)batch * 2 * L;
  for (long long r = threadIdx.x; r < rows; r += blockDim.x) {
    const int y = targets[r];
    if (y >= 0 && y < vocab) ++cnt[(r % (2 * L)) >= L ? 1 : 0];
  }
  s_cnt[0][threadIdx.x] = cnt[0];
  s_cnt[1][threadIdx.x] = cnt[1];
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      s_cnt[0][threadIdx.x] += s_cnt[0][threadIdx.x + o];
      s_cnt[1][threadIdx.x] += s_cnt[1][threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x < 2) scale[threadIdx.x] = s_cnt[threadIdx.x][0] ? 1.f / s_cnt[threadIdx.x][0] : 0.f;
}

// C [M, N] (ldc = N) = A B with the tcgen05 GEMM, in its paired form from two row blocks
// on; the maps hold A and B in the layouts its template arguments name (B MN-major).
template <bool A_MN, bool B_MN>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K,
                        float* c, int32_t* status, cudaStream_t stream) {
  using namespace gemm_tc;
  Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_m = (M + BM - 1) / BM;
  p.num_n = (N + BN - 1) / BN;
  const bool pair = p.num_m >= 2;
  p.num_k = pair ? (K + BK_P - 1) / BK_P : (K + BK - 1) / BK;
  p.num_tiles = (pair ? (p.num_m + 1) / 2 : p.num_m) * p.num_n;
  p.c = c;
  p.ldc = N;
  p.status = status;
  static std::atomic<int> attr[64], attr_pair[64];
  const cudaError_t ea =
      pair ? set_smem_limit_once(gemm_pair_kernel<A_MN, B_MN>, (int)SMEM_BYTES, attr_pair)
           : set_smem_limit_once(gemm_kernel<A_MN, B_MN>, (int)SMEM_BYTES, attr);
  if (ea != cudaSuccess) return ea;
  if (pair) {
    const int pairs = num_sms() / 2;
    const int grid = 2 * (p.num_tiles < pairs ? p.num_tiles : pairs);
    gemm_pair_kernel<A_MN, B_MN><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
  } else {
    const int grid = p.num_tiles < num_sms() ? p.num_tiles : num_sms();
    gemm_kernel<A_MN, B_MN><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
  }
  count_launches(1);
  return cudaGetLastError();
}

// 2D bf16 tensor map of a row-major [outer, inner] matrix with box {box_inner, box_outer}.
bool map2d(CUtensorMap* m, const void* base, int inner, int outer, uint32_t box_inner,
           uint32_t box_outer) {
  const uint64_t dims[2] = {(uint64_t)inner, (uint64_t)outer};
  const uint64_t strides[1] = {(uint64_t)inner * 2};
  const uint32_t box[2] = {box_inner, box_outer};
  return encode_tmap_bf16(m, base, 2, dims, strides, box);
}

// Both head launches of this file share one copy of each kernel form and so one dynamic
// shared-memory limit: the larger of the two they use.
cudaError_t head_smem_limit(bool pair) {
  static std::atomic<int> attr[64], attr_pair[64];
  return pair ? set_smem_limit_once(head_tc::head_gemm_pair_kernel,
                                    (int)head_tc::SMEM_FUSED_BYTES, attr_pair)
              : set_smem_limit_once(head_tc::head_gemm_kernel, (int)head_tc::SMEM_FUSED_BYTES,
                                    attr);
}

// The LM-head GEMM over h [rows, hidden] and W [vocab, hidden] with p's epilogue (p's
// mode fields set by the caller; the sizes and tile counts are set here): the paired form
// from two row blocks on. tm_d is the dlogits map, or NULL.
cudaError_t launch_head_gemm(const uint16_t* h, const uint16_t* w, int rows, int hidden,
                             int vocab, head_tc::Params& p, const CUtensorMap* tm_d,
                             size_t smem, cudaStream_t stream) {
  using namespace head_tc;
  p.rows = rows;
  p.hidden = hidden;
  p.vocab = vocab;
  p.num_m = (rows + BM - 1) / BM;
  p.num_n = (vocab + BN - 1) / BN;
  const bool pair = p.num_m >= 2;
  p.num_k = pair ? (hidden + BK_P - 1) / BK_P : (hidden + BK - 1) / BK;
  p.num_mp = (p.num_m + 1) / 2;
  p.num_tiles = (pair ? p.num_mp : p.num_m) * p.num_n;
  CUtensorMap tm_h, tm_w;
  if (!map2d(&tm_h, h, hidden, rows, BK, BM) ||
      !map2d(&tm_w, w, hidden, vocab, BK, pair ? BN / 2 : BN))
    return cudaErrorInvalidValue;
  const cudaError_t ea = head_smem_limit(pair);
  if (ea != cudaSuccess) return ea;
  if (pair) {
    const int pairs = num_sms() / 2;
    const int grid = 2 * (p.num_tiles < pairs ? p.num_tiles : pairs);
    head_gemm_pair_kernel<<<grid, NUM_THREADS, smem, stream>>>(tm_h, tm_w, tm_d ? *tm_d : tm_w,
                                                                p);
  } else {
    const int grid = p.num_tiles < num_sms() ? p.num_tiles : num_sms();
    head_gemm_kernel<<<grid, NUM_THREADS, smem, stream>>>(tm_h, tm_w, tm_d ? *tm_d : tm_w, p);
  }
  return cudaGetLastError();
}

size_t grad_dlogits_bytes(int batch, int L, int vocab) {
  const size_t n = (size_t)batch * 2 * L * vocab * sizeof(uint16_t);
  return (n + 255) / 256 * 256;
}

}  // namespace

size_t ce_grad_workspace_bytes(int batch, int L, int vocab) {
  return grad_dlogits_bytes(batch, L, vocab) + 256;
}

cudaError_t launch_ce_loss_grad(const uint16_t* h, const uint16_t* w, const int32_t* targets,
                                const float* row_lse, int batch, int L, int hidden, int vocab,
                                float* dh, float* dw, void* workspace, int32_t* status,
                                cudaStream_t stream) {
  using namespace head_tc;
  const int rows = batch * 2 * L;
  uint16_t* dlogits = static_cast<uint16_t*>(workspace);
  float* scale = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                          grad_dlogits_bytes(batch, L, vocab));
  Params p{};
  p.targets = targets;
  p.dlogits = dlogits;
  p.row_lse = row_lse;
  p.stream_scale = scale;
  p.two_l = 2 * L;
  p.status = status;
  // dlogits, stored in boxes of 64 columns x 128 rows
  CUtensorMap tm_d;
  if (!map2d(&tm_d, dlogits, vocab, rows, 64, BM)) return cudaErrorInvalidValue;
  ce_scale_kernel<<<1, 256, 0, stream>>>(targets, batch, L, vocab, scale);
  cudaError_t e = launch_head_gemm(h, w, rows, hidden, vocab, p, &tm_d, SMEM_FUSED_BYTES, stream);
  if (e != cudaSuccess) return e;
  count_launches(2);
  if (!dh && !dw) return cudaSuccess;

  // dh [rows, H] = dlogits [rows, V] . W [V, H]: A K-major, B (W) MN-major
  if (dh) {
    CUtensorMap ta, tb;
    if (!map2d(&ta, dlogits, vocab, rows, gemm_tc::BK, gemm_tc::BM) ||
        !map2d(&tb, w, hidden, vocab, 64, gemm_tc::BK))
      return cudaErrorInvalidValue;
    if ((e = launch_gemm<false, true>(ta, tb, rows, hidden, vocab, dh, status, stream)) !=
        cudaSuccess)
      return e;
  }
  // dW [V, H] = dlogits^T [V, rows] . h [rows, H]: both operands MN-major
  if (dw) {
    CUtensorMap ta, tb;
    if (!map2d(&ta, dlogits, vocab, rows, 64, gemm_tc::BK) ||
        !map2d(&tb, h, hidden, rows, 64, gemm_tc::BK))
      return cudaErrorInvalidValue;
    if ((e = launch_gemm<true, true>(ta, tb, vocab, hidden, rows, dw, status, stream)) !=
        cudaSuccess)
      return e;
  }
  return cudaSuccess;
}

size_t ce_workspace_bytes(int batch, int L, int vocab) {
  const size_t rows = (size_t)batch * 2 * L;
  const size_t nvt = (size_t)(vocab + head_tc::BN - 1) / head_tc::BN;
  const size_t part = rows * nvt * sizeof(float4);
  return part + ((rows * sizeof(float) + 255) / 256) * 256;
}

cudaError_t launch_ce_loss(const uint16_t* h, const uint16_t* w, const int32_t* targets,
                           int batch, int L, int hidden, int vocab, float* loss,
                           float* row_ce, float* row_lse, void* workspace, int32_t* status,
                           cudaStream_t stream) {
  using namespace head_tc;
  const int rows = batch * 2 * L;
  Params p{};
  p.part = static_cast<float4*>(workspace);
  p.targets = targets;
  p.dlogits = nullptr;
  p.status = status;
  const cudaError_t e = launch_head_gemm(h, w, rows, hidden, vocab, p, nullptr, SMEM_BYTES,
                                         stream);
  if (e != cudaSuccess) return e;
  float* ce = row_ce ? row_ce
                     : reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                (size_t)rows * p.num_n * sizeof(float4));
  ce_rows_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(p.part, targets, rows, p.num_n, vocab,
                                                      ce, row_lse, status);
  ce_reduce_kernel<<<1, 256, 0, stream>>>(ce, targets, batch, L, vocab, loss);
  count_launches(3);
  return cudaGetLastError();
}

}  // namespace mars
