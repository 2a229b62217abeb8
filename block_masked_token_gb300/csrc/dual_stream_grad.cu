// Gradient of the dual-stream attention under the MARS mask M (papernotes.org notes of
// "MARS: Enabling Autoregressive Models Multi-Token Generation", Key design 1, eq. M; the
// training step of the overall framework runs the backward of this forward).
//
// For each (batch, kv head) the G query heads that share it are handled together:
//   S_g  = Q_g K^T                   (cuBLAS, strided batch over g, fp32 out)
//   P_g  = softmax(scale S_g + M)    (here: one CTA per row, visible keys only, bf16 out)
//   dP_g = dO_g V^T                  (cuBLAS, batched, into the S buffer)
//   dV  += P_g^T dO_g                (cuBLAS, accumulated over g)
//   dS_g = P_g * (dP_g - D)          (here, in place over P; D_i = rowsum(dO_i * O_i))
//   dK  += scale dS_g^T Q_g          (cuBLAS, accumulated over g)
//   dQ_g = scale dS_g K              (cuBLAS, batched)
// The 2L x 2L score and probability matrices of one kv group are materialised in the
// workspace (fp32 and bf16). Masked entries are exactly 0 in P and dS, so the products are
// the masked ones; about half of the dense work multiplies zeros. This is the plain
// formulation with library GEMMs, correct at any size. A fused tile kernel in the manner
// of the forward (recompute S per tile, never store it) would avoid the materialisation.
#include <cublas_v2.h>
#include <cuda_bf16.h>

#include <climits>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mars {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// dO (fp32) -> bf16 copy, and D[b, i, h] = sum_d dO[b, i, h, d] * O[b, i, h, d]. One warp
// per (b, i, h) row.
__global__ void __launch_bounds__(256) grad_prep_kernel(const float* __restrict__ o,
                                                        const float* __restrict__ d_o,
                                                        __nv_bfloat16* __restrict__ do_bf,
                                                        float* __restrict__ drow,
                                                        long long nrows, int d) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= nrows) return;
  const float* a = o + row * d;
  const float* g = d_o + row * d;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) {
    const float x = g[c];
    acc += x * a[c];
    do_bf[row * d + c] = __float2bfloat16_rn(x);
  }
  acc = warp_sum(acc);
  if (lane == 0) drow[row] = acc;
}

// Visible keys of query row i (0-indexed over z = [x; x~]) under M: [0, e1) and [s2, e2]
// (the second range empty for clean rows).
MARS_DEV void visible_ranges(int i, int L, int B, int& e1, int& s2, int& e2) {
  if (i < L) {
    e1 = i + 1;
    s2 = INT_MAX;
    e2 = -1;
  } else {
    const int bs = ((i - L) / B) * B;
    e1 = bs;
    s2 = L + bs;
    e2 = i;
  }
}

// P = softmax(scale * S + M) for the rows of G score matrices (one CTA per row): one pass
// over the visible keys for the running max and sum (online), one to write the row, with
// masked entries 0. Only the visible keys are read. S: [G][2L][2L] fp32; P: bf16.
__global__ void __launch_bounds__(256) grad_softmax_kernel(const float* __restrict__ s,
                                                           __nv_bfloat16* __restrict__ p,
                                                           int L, int B, float scale_log2) {
  __shared__ float red_m[8], red_s[8];
  const int n = 2 * L;
  const long long grow = blockIdx.x;                  // g * 2L + i
  const int i = (int)(grow % n);
  const float* srow = s + grow * n;
  __nv_bfloat16* prow = p + grow * n;
  int e1, s2, e2;
  visible_ranges(i, L, B, e1, s2, e2);
  const int n2 = s2 <= e2 ? e2 - s2 + 1 : 0;        // keys of the second range
  const int nvis = e1 + n2;
  auto key = [&](int t) { return t < e1 ? t : s2 + (t - e1); };   // t-th visible key
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m = -INFINITY, sum = 0.f;                     // in log2 units
  for (int t = threadIdx.x; t < nvis; t += blockDim.x) {
    const float x = srow[key(t)] * scale_log2;
    if (x > m) {
      sum = sum * exp2f(m - x) + 1.f;
      m = x;
    } else {
      sum += exp2f(x - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2v = __shfl_xor_sync(0xffffffffu, sum, o);
    const float mm = fmaxf(m, m2);
    sum = (m == -INFINITY ? 0.f : sum * exp2f(m - mm)) +
          (m2 == -INFINITY ? 0.f : s2v * exp2f(m2 - mm));
    m = mm;
  }
  if (lane == 0) {
    red_m[warp] = m;
    red_s[warp] = sum;
  }
  __syncthreads();
  float mt = red_m[0];
  for (int w = 1; w < 8; ++w) mt = fmaxf(mt, red_m[w]);
  float st = 0.f;
  for (int w = 0; w < 8; ++w)
    if (red_m[w] != -INFINITY) st += red_s[w] * exp2f(red_m[w] - mt);
  const float inv = 1.f / st;                          // the diagonal is always visible
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const bool v = j < e1 || (j >= s2 && j <= e2);
    prow[j] = __float2bfloat16_rn(v ? exp2f(srow[j] * scale_log2 - mt) * inv : 0.f);
  }
}

// dS = P * (dP - D_i), in place over P (bf16), on the visible keys only (P, hence dS, is 0
// on the others). dP: [G][2L][2L] fp32; D of query head h0 + g at row i:
// drow[((b * 2L + i) * hq) + h0 + g].
__global__ void __launch_bounds__(256) grad_ds_kernel(__nv_bfloat16* __restrict__ p,
                                                      const float* __restrict__ dp,
                                                      const float* __restrict__ drow,
                                                      int L, int B, int hq, int h0, int b) {
  const int n = 2 * L;
  const long long grow = blockIdx.x;
  const int g = (int)(grow / n), i = (int)(grow % n);
  const float dv = drow[((long long)b * n + i) * hq + h0 + g];
  __nv_bfloat16* prow = p + grow * n;
  const float* dprow = dp + grow * n;
  int e1, s2, e2;
  visible_ranges(i, L, B, e1, s2, e2);
  const int n2 = s2 <= e2 ? e2 - s2 + 1 : 0;
  for (int t = threadIdx.x; t < e1 + n2; t += blockDim.x) {
    const int j = t < e1 ? t : s2 + (t - e1);
    const float pv = __bfloat162float(prow[j]);
    prow[j] = __float2bfloat16_rn(pv * (dprow[j] - dv));
  }
}

struct Blas {
  std::mutex mu;
  cublasHandle_t h[64] = {};
};
Blas& blas() {
  static Blas b;
  return b;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

size_t dual_grad_workspace_bytes(int batch, int L, int hq, int hkv, int d) {
  const size_t n = 2 * (size_t)L;
  const size_t G = (size_t)(hq / hkv);
  return align256(G * n * n * sizeof(float)) +            // S, then dP
         align256(G * n * n * sizeof(uint16_t)) +         // P, then dS
         align256((size_t)batch * n * hq * d * sizeof(uint16_t)) +   // dO in bf16
         align256((size_t)batch * n * hq * sizeof(float));           // D
}

cudaError_t launch_dual_stream_grad(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    const float* o, const float* d_o, int batch, int L, int B,
                                    int hq, int hkv, int d, float scale, float* dq, float* dk,
                                    float* dv, void* workspace, cudaStream_t stream) {
  const long long n = 2LL * L;
  const int G = hq / hkv;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* sbuf = reinterpret_cast<float*>(ws);
  ws += align256((size_t)G * n * n * sizeof(float));
  __nv_bfloat16* pbuf = reinterpret_cast<__nv_bfloat16*>(ws);
  ws += align256((size_t)G * n * n * sizeof(uint16_t));
  __nv_bfloat16* do_bf = reinterpret_cast<__nv_bfloat16*>(ws);
  ws += align256((size_t)batch * n * hq * d * sizeof(uint16_t));
  float* drow = reinterpret_cast<float*>(ws);

  const long long nrows = (long long)batch * n * hq;
  grad_prep_kernel<<<(unsigned)((nrows + 7) / 8), 256, 0, stream>>>(o, d_o, do_bf, drow,
                                                                    nrows, d);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  Blas& bl = blas();
  std::lock_guard<std::mutex> lock(bl.mu);
  if (!bl.h[dev] && cublasCreate(&bl.h[dev]) != CUBLAS_STATUS_SUCCESS) {
    bl.h[dev] = nullptr;
    return cudaErrorInitializationError;
  }
  cublasHandle_t hb = bl.h[dev];
  if (cublasSetStream(hb, stream) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  const float one = 1.f, zero = 0.f;
  const int ldq = hq * d, ldk = hkv * d, nn = (int)n;
  const long long strideS = n * n;
  auto ok = [](cublasStatus_t st) { return st == CUBLAS_STATUS_SUCCESS; };
  const float scale_log2 = scale * kLog2e;
  const unsigned grows = (unsigned)(G * n);

  for (int b = 0; b < batch; ++b) {
    for (int hk = 0; hk < hkv; ++hk) {
      const int h0 = hk * G;
      const uint16_t* Q0 = q + ((size_t)b * n * hq + h0) * d;
      const __nv_bfloat16* dO0 = do_bf + ((size_t)b * n * hq + h0) * d;
      const uint16_t* K = k + ((size_t)b * n * hkv + hk) * d;
      const uint16_t* V = v + ((size_t)b * n * hkv + hk) * d;
      float* dQ0 = dq + ((size_t)b * n * hq + h0) * d;
      float* dK = dk + ((size_t)b * n * hkv + hk) * d;
      float* dV = dv + ((size_t)b * n * hkv + hk) * d;
      // S_g[i][j] = sum_c Q_g[i][c] K[j][c]  (column-major: S_g^T = K Q_g^T)
      if (!ok(cublasGemmStridedBatchedEx(hb, CUBLAS_OP_T, CUBLAS_OP_N, nn, nn, d, &one, K,
                                         CUDA_R_16BF, ldk, 0, Q0, CUDA_R_16BF, ldq, d, &zero,
                                         sbuf, CUDA_R_32F, nn, strideS, G, CUBLAS_COMPUTE_32F,
                                         CUBLAS_GEMM_DEFAULT)))
        return cudaErrorUnknown;
      grad_softmax_kernel<<<grows, 256, 0, stream>>>(sbuf, pbuf, L, B, scale_log2);
      // dP_g = dO_g V^T, into the S buffer
      if (!ok(cublasGemmStridedBatchedEx(hb, CUBLAS_OP_T, CUBLAS_OP_N, nn, nn, d, &one, V,
                                         CUDA_R_16BF, ldk, 0, dO0, CUDA_R_16BF, ldq, d, &zero,
                                         sbuf, CUDA_R_32F, nn, strideS, G, CUBLAS_COMPUTE_32F,
                                         CUBLAS_GEMM_DEFAULT)))
        return cudaErrorUnknown;
      // dV += P_g^T dO_g  (column-major: dV^T = dO_g^T P_g)
      for (int g = 0; g < G; ++g) {
        if (!ok(cublasGemmEx(hb, CUBLAS_OP_N, CUBLAS_OP_T, d, nn, nn, &one, dO0 + g * d,
                             CUDA_R_16BF, ldq, pbuf + g * strideS, CUDA_R_16BF, nn,
                             g ? &one : &zero, dV, CUDA_R_32F, ldk, CUBLAS_COMPUTE_32F,
                             CUBLAS_GEMM_DEFAULT)))
          return cudaErrorUnknown;
      }
      grad_ds_kernel<<<grows, 256, 0, stream>>>(pbuf, sbuf, drow, L, B, hq, h0, b);
      // dK += scale dS_g^T Q_g  (column-major: dK^T = Q_g^T dS_g)
      for (int g = 0; g < G; ++g) {
        if (!ok(cublasGemmEx(hb, CUBLAS_OP_N, CUBLAS_OP_T, d, nn, nn, &scale, Q0 + g * d,
                             CUDA_R_16BF, ldq, pbuf + g * strideS, CUDA_R_16BF, nn,
                             g ? &one : &zero, dK, CUDA_R_32F, ldk, CUBLAS_COMPUTE_32F,
                             CUBLAS_GEMM_DEFAULT)))
          return cudaErrorUnknown;
      }
      // dQ_g = scale dS_g K  (column-major: dQ_g^T = K^T dS_g^T)
      if (!ok(cublasGemmStridedBatchedEx(hb, CUBLAS_OP_N, CUBLAS_OP_N, d, nn, nn, &scale, K,
                                         CUDA_R_16BF, ldk, 0, pbuf, CUDA_R_16BF, nn, strideS,
                                         &zero, dQ0, CUDA_R_32F, ldq, d, G,
                                         CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT)))
        return cudaErrorUnknown;
      count_launches(2);
    }
  }
  return cudaGetLastError();
}

}  // namespace mars
