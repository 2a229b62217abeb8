// Decode-step epilogue: LM-head logits, per-position max-prob and argmax, and the
// left-to-right threshold acceptance (papernotes.org notes of "MARS: Enabling
// Autoregressive Models Multi-Token Generation", Key design 3; gist.science explainer,
// 2.C "Confidence Thresholding").
//
// Kernel 1 computes a tile of logits l = h W^T and reduces it in place to one partial
// (tile max, sum of exp(l - tile max), first argmax) per (row, vocabulary tile); the
// logits themselves never leave the chip. Kernel 2 merges the partials of each row,
// writes token and max-prob = 1 / sum_v exp(l_v - max), and scans each sequence's B
// positions left to right for N.
#include "common.cuh"
#include "internal.h"

namespace mars {

namespace {

constexpr int kTM = 64;     // rows per CTA tile
constexpr int kTN = 128;    // vocabulary columns per CTA tile
constexpr int kTK = 32;     // hidden chunk

// Partial: {max, sumexp, argmax (int bits), unused}
__global__ void __launch_bounds__(256) head_partials_kernel(
    const uint16_t* __restrict__ h, const uint16_t* __restrict__ w, int rows, int hidden,
    int vocab, int nvt, float4* __restrict__ part) {
  // the staging tiles and the logits tile share one buffer (they are live at different
  // times): kTM*(kTN+1) floats > kTK*(kTM+4) + kTK*(kTN+4)
  __shared__ float raw[kTM * (kTN + 1)];
  float (*a_s)[kTM + 4] = reinterpret_cast<float (*)[kTM + 4]>(raw);
  float (*b_s)[kTN + 4] = reinterpret_cast<float (*)[kTN + 4]>(raw + kTK * (kTM + 4));
  float (*c_s)[kTN + 1] = reinterpret_cast<float (*)[kTN + 1]>(raw);
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int row0 = blockIdx.y * kTM, col0 = blockIdx.x * kTN;
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < hidden; k0 += kTK) {
    __syncthreads();
    for (int idx = tid; idx < kTM * kTK; idx += 256) {
      const int r = idx / kTK, c = idx - r * kTK;
      const int gr = row0 + r, gc = k0 + c;
      a_s[c][r] = (gr < rows && gc < hidden) ? bf16_to_f32(h[(size_t)gr * hidden + gc]) : 0.f;
    }
    for (int idx = tid; idx < kTN * kTK; idx += 256) {
      const int r = idx / kTK, c = idx - r * kTK;
      const int gr = col0 + r, gc = k0 + c;
      b_s[c][r] = (gr < vocab && gc < hidden) ? bf16_to_f32(w[(size_t)gr * hidden + gc]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < kTK; ++kk) {
      float av[4], bv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = a_s[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 8; ++j) bv[j] = b_s[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) c_s[ty * 4 + i][tx + 16 * j] = acc[i][j];
  __syncthreads();
  // 4 threads per row, each over 32 consecutive columns, combined by shuffles.
  const int r = tid >> 2, part_id = tid & 3;
  const int ncol = min(kTN, vocab - col0);
  float m = -INFINITY;
  int am = 0x7fffffff;
  for (int c = part_id * 32; c < part_id * 32 + 32; ++c) {
    if (c < ncol) {
      const float x = c_s[r][c];
      if (x > m) { m = x; am = col0 + c; }
    }
  }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const int a2 = __shfl_xor_sync(0xffffffffu, am, o);
    if (m2 > m || (m2 == m && a2 < am)) { m = m2; am = a2; }
  }
  float se = 0.f;
  for (int c = part_id * 32; c < part_id * 32 + 32; ++c)
    if (c < ncol) se += __expf(c_s[r][c] - m);
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
  if (part_id == 0 && row0 + r < rows)
    part[(size_t)(row0 + r) * nvt + blockIdx.x] = make_float4(m, se, __int_as_float(am), 0.f);
}

// One CTA per sequence, one warp per block position: merge partials, then the scan.
__global__ void __launch_bounds__(1024) head_finalize_kernel(
    const float4* __restrict__ part, int B, int nvt, float tau, int32_t* __restrict__ tokens,
    float* __restrict__ maxprob, int32_t* __restrict__ n_accept) {
  __shared__ float p_s[32];
  const int s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < B) {
    const int row = s * B + warp;
    const float4* pr = part + (size_t)row * nvt;
    float m = -INFINITY;
    int am = 0x7fffffff;
    for (int t = lane; t < nvt; t += 32) {
      const float4 v = pr[t];
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
      const float4 v = pr[t];
      se += v.y * __expf(v.x - m);
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
    int n = 0;
    while (n < B && p_s[n] >= tau) ++n;
    n_accept[s] = n < 1 ? 1 : n;
  }
}

}  // namespace

size_t head_workspace_bytes(int batch, int B, int vocab) {
  const size_t nvt = (size_t)(vocab + kTN - 1) / kTN;
  return (size_t)batch * B * nvt * sizeof(float4);
}

cudaError_t launch_head_accept(const uint16_t* h, const uint16_t* w, int batch, int B,
                               int hidden, int vocab, float tau, int32_t* tokens,
                               float* maxprob, int32_t* n_accept, void* workspace,
                               cudaStream_t stream) {
  const int rows = batch * B;
  const int nvt = (vocab + kTN - 1) / kTN;
  float4* part = static_cast<float4*>(workspace);
  dim3 grid(nvt, (rows + kTM - 1) / kTM);
  head_partials_kernel<<<grid, 256, 0, stream>>>(h, w, rows, hidden, vocab, nvt, part);
  head_finalize_kernel<<<batch, 32 * B, 0, stream>>>(part, B, nvt, tau, tokens, maxprob, n_accept);
  count_launches(2);
  return cudaGetLastError();
}

}  // namespace mars
