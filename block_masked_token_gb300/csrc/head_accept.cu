// Decode-step epilogue: LM-head logits, per-position max-prob and argmax, and the
// left-to-right threshold acceptance (papernotes.org notes of "MARS: Enabling
// Autoregressive Models Multi-Token Generation", Key design 3; gist.science explainer,
// 2.C "Confidence Thresholding").
//
// Kernel 1 (head_gemm_tc.cuh) is a tcgen05 GEMM whose epilogue turns each 128 x 256 tile
// of logits into one partial {tile max, sum exp(l - tile max), first argmax} per row; the
// logits never leave the chip. Kernel 2 merges the partials of each row, writes the token
// and max-prob = 1 / sum_v exp(l_v - max), and scans each sequence's B positions left to
// right: N = leading run of max-prob >= tau, at least 1, at most B. tau is one value per
// call, or one per sequence (per request: gist.science explainer, 2.C "Adaptive
// Throughput"; papernotes.org notes, highlights, third point).
#include "common.cuh"
#include "head_gemm_tc.cuh"
#include "internal.h"

namespace mars {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// One CTA per sequence, one warp per block position: merge partials, then the scan.
__global__ void __launch_bounds__(1024) head_finalize_kernel(
    const float4* __restrict__ part, int rows, int B, int nvt, float tau,
    const float* __restrict__ taus, int32_t* __restrict__ tokens, float* __restrict__ maxprob,
    int32_t* __restrict__ n_accept) {
  __shared__ float p_s[32];
  const int s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < B) {
    const int row = s * B + warp;
    float m = -INFINITY;
    int am = 0x7fffffff;
    for (int t = lane; t < nvt; t += 32) {
      const float4 v = part[(size_t)t * rows + row];
      const int a = __float_as_int(v.z);
      if (v.x > m || (v.x == m && a < am)) { m = v.x; am = a; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const int a2 = __shfl_xor_sync(0xffffffffu, am, o);
      if (m2 > m || (m2 == m && a2 < am)) { m = m2; am = a2; }
    }
    float se = 0.f;
    for (int t = lane; t < nvt; t += 32) {
      const float4 v = part[(size_t)t * rows + row];
      se += v.y * exp2f((v.x - m) * kLog2e);
    }
    se = warp_sum(se);
    const float p = 1.f / se;
    if (lane == 0) {
      tokens[row] = am;
      maxprob[row] = p;
      p_s[warp] = p;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const float t = taus ? taus[s] : tau;      // a NaN threshold accepts only the floor
    int n = 0;
    while (n < B && p_s[n] >= t) ++n;
    n_accept[s] = n < 1 ? 1 : n;
  }
}

}  // namespace

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return kNumSMs;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : kNumSMs;
  }
  return cached[dev];
}

size_t head_workspace_bytes(int batch, int B, int vocab) {
  const size_t nvt = (size_t)(vocab + head_tc::BN - 1) / head_tc::BN;
  return (size_t)batch * B * nvt * sizeof(float4);
}

cudaError_t launch_head_accept(const uint16_t* h, const uint16_t* w, int batch, int B,
                               int hidden, int vocab, float tau, const float* taus,
                               int32_t* tokens, float* maxprob, int32_t* n_accept,
                               void* workspace, int32_t* status, cudaStream_t stream) {
  using namespace head_tc;
  const int rows = batch * B;
  CUtensorMap tm_h, tm_w;
  {
    const uint64_t dims[2] = {(uint64_t)hidden, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)hidden * 2};
    const uint32_t box[2] = {BK, BM};
    if (!encode_tmap_bf16(&tm_h, h, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)hidden, (uint64_t)vocab};
    const uint64_t strides[1] = {(uint64_t)hidden * 2};
    const uint32_t box[2] = {BK, BN};
    if (!encode_tmap_bf16(&tm_w, w, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  Params p{};
  p.rows = rows;
  p.hidden = hidden;
  p.vocab = vocab;
  p.num_m = (rows + BM - 1) / BM;
  p.num_n = (vocab + BN - 1) / BN;
  p.num_k = (hidden + BK - 1) / BK;
  p.num_tiles = p.num_m * p.num_n;
  p.part = static_cast<float4*>(workspace);
  p.targets = nullptr;
  p.dlogits = nullptr;
  p.status = status;
  static std::atomic<int> attr[64];
  const cudaError_t ea = set_smem_limit_once(head_gemm_kernel, (int)SMEM_BYTES, attr);
  if (ea != cudaSuccess) return ea;
  const int grid = p.num_tiles < num_sms() ? p.num_tiles : num_sms();
  head_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(tm_h, tm_w, p);
  head_finalize_kernel<<<batch, 32 * B, 0, stream>>>(p.part, rows, B, p.num_n, tau, taus,
                                                     tokens, maxprob, n_accept);
  count_launches(2);
  return cudaGetLastError();
}

}  // namespace mars
