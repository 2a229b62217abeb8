// Gradient of the dual-stream attention under the MARS mask M (papernotes.org notes of
// "MARS: Enabling Autoregressive Models Multi-Token Generation", Key design 1, eq. M; the
// training step of the overall framework runs the backward of this forward).
//
// Only two blocks of the 2L x 2L score matrix hold visible keys: every row against the
// clean keys (S_c, 2L x L: causal for clean rows, keys before the block start for masked
// rows) and each masked row against the keys of its own block (S_m, one Bb x Bb block per
// block of the masked stream, Bb = min(B, L)); clean rows never see masked keys. For each
// (batch, kv head) the G query heads that share it are handled together:
//   S_g  = Q_g K^T on those blocks       (cuBLAS; batched over g, and over blocks for S_m)
//   P_g  = softmax(scale S_g + M)        (here: one CTA per row, visible keys only)
//   dP_g = dO_g V^T on the same blocks   (cuBLAS, into the S buffers)
//   dV  += P_g^T dO_g                    (cuBLAS, accumulated over g)
//   dS_g = P_g * (dP_g - D)              (here, in place over P; D_i = rowsum(dO_i * O_i))
//   dK  += scale dS_g^T Q_g              (cuBLAS, accumulated over g)
//   dQ_g = scale dS_g K                  (cuBLAS)
// The blocks of one kv group are materialised in the workspace (scores fp32, P and dS
// bf16, masked entries exactly 0). This is the plain formulation with library GEMMs; a
// fused tile kernel in the manner of the forward would never store the blocks.
#include <cublas_v2.h>
#include <cuda_bf16.h>

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

// Geometry of the two score blocks of one head (see the header).
struct Blocks {
  int L, B, Bb, nb;   // stream length, block size, block width in S_m, blocks in S_m
};

MARS_DEV Blocks blocks_of(int L, int B) {
  Blocks g;
  g.L = L;
  g.B = B;
  g.Bb = B < L ? B : L;
  g.nb = (L + g.Bb - 1) / g.Bb;
  return g;
}

// Row i of head g (one CTA): the visible keys are S_c[i][0 .. e1) and, for a masked row
// t = i - L, S_m[t][0 .. cm] (cm = t - block start); P is written in full (0 elsewhere).
// S_c: [G][2L][L], S_m: [G][nb * Bb][Bb] fp32; P_c, P_m: same shapes, bf16.
__global__ void __launch_bounds__(256) grad_softmax_kernel(const float* __restrict__ s_c,
                                                           const float* __restrict__ s_m,
                                                           __nv_bfloat16* __restrict__ p_c,
                                                           __nv_bfloat16* __restrict__ p_m,
                                                           int L, int B, float scale_log2) {
  __shared__ float red_m[8], red_s[8];
  const Blocks geo = blocks_of(L, B);
  const int n = 2 * L;
  const long long grow = blockIdx.x;                   // g * 2L + i
  const int g = (int)(grow / n), i = (int)(grow % n);
  const float* crow = s_c + grow * L;
  __nv_bfloat16* pcrow = p_c + grow * L;
  int e1, cm;                                           // clean keys [0, e1); block keys [0, cm]
  const float* mrow = nullptr;
  __nv_bfloat16* pmrow = nullptr;
  if (i < L) {
    e1 = i + 1;
    cm = -1;
  } else {
    const int t = i - L, bs = (t / B) * B;
    e1 = bs;
    cm = t - bs;
    const long long mr = (long long)g * geo.nb * geo.Bb + t;
    mrow = s_m + mr * geo.Bb;
    pmrow = p_m + mr * geo.Bb;
  }
  const int nvis = e1 + cm + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m = -INFINITY, sum = 0.f;                       // in log2 units
  for (int t = threadIdx.x; t < nvis; t += blockDim.x) {
    const float x = (t < e1 ? crow[t] : mrow[t - e1]) * scale_log2;
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
  const float inv = 1.f / st;                           // the diagonal is always visible
  for (int j = threadIdx.x; j < L; j += blockDim.x)
    pcrow[j] = __float2bfloat16_rn(j < e1 ? exp2f(crow[j] * scale_log2 - mt) * inv : 0.f);
  if (pmrow)
    for (int c = threadIdx.x; c < geo.Bb; c += blockDim.x)
      pmrow[c] = __float2bfloat16_rn(c <= cm ? exp2f(mrow[c] * scale_log2 - mt) * inv : 0.f);
}

// dS = P * (dP - D_i), in place over P (bf16), on the visible keys of row i of head g (P,
// hence dS, is 0 on the others). dP in the S buffers; D of query head h0 + g at row i:
// drow[((b * 2L + i) * hq) + h0 + g].
__global__ void __launch_bounds__(256) grad_ds_kernel(__nv_bfloat16* __restrict__ p_c,
                                                      __nv_bfloat16* __restrict__ p_m,
                                                      const float* __restrict__ dp_c,
                                                      const float* __restrict__ dp_m,
                                                      const float* __restrict__ drow,
                                                      int L, int B, int hq, int h0, int b) {
  const Blocks geo = blocks_of(L, B);
  const int n = 2 * L;
  const long long grow = blockIdx.x;
  const int g = (int)(grow / n), i = (int)(grow % n);
  const float dv = drow[((long long)b * n + i) * hq + h0 + g];
  int e1 = i + 1, cm = -1;
  long long mr = 0;
  if (i >= L) {
    const int t = i - L, bs = (t / B) * B;
    e1 = bs;
    cm = t - bs;
    mr = ((long long)g * geo.nb * geo.Bb + t) * geo.Bb;
  }
  for (int t = threadIdx.x; t < e1 + cm + 1; t += blockDim.x) {
    if (t < e1) {
      const long long x = grow * L + t;
      p_c[x] = __float2bfloat16_rn(__bfloat162float(p_c[x]) * (dp_c[x] - dv));
    } else {
      const long long x = mr + (t - e1);
      p_m[x] = __float2bfloat16_rn(__bfloat162float(p_m[x]) * (dp_m[x] - dv));
    }
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

namespace {

struct GradBuffers {
  float* s_c;               // [G][2L][L]   scores against the clean keys, then dP
  float* s_m;               // [G][nb*Bb][Bb] scores inside the masked blocks, then dP
  __nv_bfloat16* p_c;       // P, then dS (same shapes)
  __nv_bfloat16* p_m;
  __nv_bfloat16* do_bf;     // dO in bf16, [b, 2L, hq, d]
  float* drow;              // D, [b, 2L, hq]
  size_t bytes;
};

GradBuffers carve(void* base, int batch, int L, int B, int hq, int hkv, int d) {
  const size_t n = 2 * (size_t)L;
  const size_t G = (size_t)(hq / hkv);
  const size_t Bb = (size_t)(B < L ? B : L);
  const size_t nb = ((size_t)L + Bb - 1) / Bb;
  GradBuffers g{};
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* at = p ? p + off : nullptr;
    off += align256(bytes);
    return at;
  };
  g.s_c = reinterpret_cast<float*>(take(G * n * L * sizeof(float)));
  g.s_m = reinterpret_cast<float*>(take(G * nb * Bb * Bb * sizeof(float)));
  g.p_c = reinterpret_cast<__nv_bfloat16*>(take(G * n * L * sizeof(uint16_t)));
  g.p_m = reinterpret_cast<__nv_bfloat16*>(take(G * nb * Bb * Bb * sizeof(uint16_t)));
  g.do_bf = reinterpret_cast<__nv_bfloat16*>(take((size_t)batch * n * hq * d * sizeof(uint16_t)));
  g.drow = reinterpret_cast<float*>(take((size_t)batch * n * hq * sizeof(float)));
  g.bytes = off;
  return g;
}

}  // namespace

size_t dual_grad_workspace_bytes(int batch, int L, int B, int hq, int hkv, int d) {
  return carve(nullptr, batch, L, B, hq, hkv, d).bytes;
}

cudaError_t launch_dual_stream_grad(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    const float* o, const float* d_o, int batch, int L, int B,
                                    int hq, int hkv, int d, float scale, float* dq, float* dk,
                                    float* dv, void* workspace, cudaStream_t stream) {
  const long long n = 2LL * L;
  const int G = hq / hkv;
  const GradBuffers w = carve(workspace, batch, L, B, hq, hkv, d);
  const int Bb = B < L ? B : L;
  const int nb = (L + Bb - 1) / Bb;
  const int nfull = L / Bb, rem = L % Bb;

  const long long nrows = (long long)batch * n * hq;
  grad_prep_kernel<<<(unsigned)((nrows + 7) / 8), 256, 0, stream>>>(o, d_o, w.do_bf, w.drow,
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
  const long long strideC = n * L;                      // one head's S_c
  const long long strideM = (long long)nb * Bb * Bb;    // one head's S_m
  const long long blkM = (long long)Bb * Bb;            // one block of S_m
  const float scale_log2 = scale * kLog2e;
  const unsigned grows = (unsigned)(G * n);
  bool good = true;
  auto ok = [&](cublasStatus_t st) { good = good && st == CUBLAS_STATUS_SUCCESS; };
  const cublasOperation_t N_ = CUBLAS_OP_N, T_ = CUBLAS_OP_T;
  const cudaDataType_t BF = CUDA_R_16BF, F32 = CUDA_R_32F;
  const cublasComputeType_t CT = CUBLAS_COMPUTE_32F;

  // S = X Y^T on the two blocks (X: query-side rows, Y: key-side rows; both bf16), into
  // (c, m): the batch over g for the clean-key block, and per g the batch over masked
  // blocks plus the short last block.
  auto scores = [&](const void* X0, int ldx, const void* Y, float* c, float* m) {
    // clean keys: c_g[i][j] = sum X_g[i] Y[j], i < 2L, j < L  (column-major C^T = Y X_g^T)
    ok(cublasGemmStridedBatchedEx(hb, T_, N_, L, nn, d, &one, Y, BF, ldk, 0, X0, BF, ldx, d,
                                  &zero, c, F32, L, strideC, G, CT, CUBLAS_GEMM_DEFAULT));
    for (int g = 0; g < G; ++g) {
      const uint16_t* Xg = static_cast<const uint16_t*>(X0) + g * d + (size_t)L * ldx;
      const uint16_t* Ym = static_cast<const uint16_t*>(Y) + (size_t)L * ldk;
      float* mg = m + g * strideM;
      if (nfull)
        ok(cublasGemmStridedBatchedEx(hb, T_, N_, Bb, Bb, d, &one, Ym, BF, ldk,
                                      (long long)Bb * ldk, Xg, BF, ldx, (long long)Bb * ldx,
                                      &zero, mg, F32, Bb, blkM, nfull, CT, CUBLAS_GEMM_DEFAULT));
      if (rem)
        ok(cublasGemmEx(hb, T_, N_, rem, rem, d, &one, Ym + (size_t)nfull * Bb * ldk, BF, ldk,
                        Xg + (size_t)nfull * Bb * ldx, BF, ldx, &zero, mg + nfull * blkM, F32,
                        Bb, CT, CUBLAS_GEMM_DEFAULT));
    }
  };
  // R += alpha sum_g P_g^T X_g for the key-side rows R (dV with P, X = dO; dK with dS,
  // X = Q): the clean keys from the clean block, the masked keys block by block.
  auto key_side = [&](const __nv_bfloat16* pc, const __nv_bfloat16* pm, const void* X0,
                      int ldx, float alpha, float* R) {
    for (int g = 0; g < G; ++g) {
      const float* beta = g ? &one : &zero;
      const uint16_t* Xg = static_cast<const uint16_t*>(X0) + g * d;
      // R[0:L]^T (d x L) = X_g^T (d x 2L) . P_c (2L x L)
      ok(cublasGemmEx(hb, N_, T_, d, L, nn, &alpha, Xg, BF, ldx, pc + g * strideC, BF, L, beta,
                      R, F32, ldk, CT, CUBLAS_GEMM_DEFAULT));
      const uint16_t* Xm = Xg + (size_t)L * ldx;
      float* Rm = R + (size_t)L * ldk;
      if (nfull)
        ok(cublasGemmStridedBatchedEx(hb, N_, T_, d, Bb, Bb, &alpha, Xm, BF, ldx,
                                      (long long)Bb * ldx, pm + g * strideM, BF, Bb, blkM, beta,
                                      Rm, F32, ldk, (long long)Bb * ldk, nfull, CT,
                                      CUBLAS_GEMM_DEFAULT));
      if (rem)
        ok(cublasGemmEx(hb, N_, T_, d, rem, rem, &alpha, Xm + (size_t)nfull * Bb * ldx, BF, ldx,
                        pm + g * strideM + nfull * blkM, BF, Bb, beta,
                        Rm + (size_t)nfull * Bb * ldk, F32, ldk, CT, CUBLAS_GEMM_DEFAULT));
    }
  };

  for (int b = 0; b < batch && good; ++b) {
    for (int hk = 0; hk < hkv && good; ++hk) {
      const int h0 = hk * G;
      const uint16_t* Q0 = q + ((size_t)b * n * hq + h0) * d;
      const __nv_bfloat16* dO0 = w.do_bf + ((size_t)b * n * hq + h0) * d;
      const uint16_t* K = k + ((size_t)b * n * hkv + hk) * d;
      const uint16_t* V = v + ((size_t)b * n * hkv + hk) * d;
      float* dQ0 = dq + ((size_t)b * n * hq + h0) * d;
      float* dK = dk + ((size_t)b * n * hkv + hk) * d;
      float* dV = dv + ((size_t)b * n * hkv + hk) * d;
      scores(Q0, ldq, K, w.s_c, w.s_m);
      grad_softmax_kernel<<<grows, 256, 0, stream>>>(w.s_c, w.s_m, w.p_c, w.p_m, L, B,
                                                     scale_log2);
      scores(dO0, ldq, V, w.s_c, w.s_m);                  // dP
      key_side(w.p_c, w.p_m, dO0, ldq, 1.f, dV);
      grad_ds_kernel<<<grows, 256, 0, stream>>>(w.p_c, w.p_m, w.s_c, w.s_m, w.drow, L, B, hq,
                                                h0, b);
      key_side(w.p_c, w.p_m, Q0, ldq, scale, dK);
      // dQ_g = scale (dS_c K_c + dS_m K_m)   (column-major: dQ_g^T = K^T dS_g^T)
      ok(cublasGemmStridedBatchedEx(hb, N_, N_, d, nn, L, &scale, K, BF, ldk, 0, w.p_c, BF, L,
                                    strideC, &zero, dQ0, F32, ldq, d, G, CT,
                                    CUBLAS_GEMM_DEFAULT));
      for (int g = 0; g < G; ++g) {
        const uint16_t* Km = K + (size_t)L * ldk;
        float* dQm = dQ0 + g * d + (size_t)L * ldq;
        if (nfull)
          ok(cublasGemmStridedBatchedEx(hb, N_, N_, d, Bb, Bb, &scale, Km, BF, ldk,
                                        (long long)Bb * ldk, w.p_m + g * strideM, BF, Bb, blkM,
                                        &one, dQm, F32, ldq, (long long)Bb * ldq, nfull, CT,
                                        CUBLAS_GEMM_DEFAULT));
        if (rem)
          ok(cublasGemmEx(hb, N_, N_, d, rem, rem, &scale, Km + (size_t)nfull * Bb * ldk, BF,
                          ldk, w.p_m + g * strideM + nfull * blkM, BF, Bb, &one,
                          dQm + (size_t)nfull * Bb * ldq, F32, ldq, CT, CUBLAS_GEMM_DEFAULT));
      }
      count_launches(2);
    }
  }
  if (!good) return cudaErrorUnknown;
  return cudaGetLastError();
}

}  // namespace mars
