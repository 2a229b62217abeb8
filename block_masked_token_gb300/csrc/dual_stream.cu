// Dual-stream (training-form) attention under the MARS mask M (papernotes.org notes of
// "MARS: Enabling Autoregressive Models Multi-Token Generation", Key design 1, eq. M,
// beta(t) = ceil(t/B); overall framework: clean stream x and masked stream x~ in one
// forward over z = [x; x~]).
//
// In 0-indexed stream-local terms a query row sees one or two contiguous key ranges:
//   clean row i < L:           keys [0, i]
//   masked row L + t:          clean keys [0, B*(t/B)) and masked keys [L + B*(t/B), L + t]
// so keys outside those ranges (fully masked under M) are never touched.
//
// Reference CUDA-core kernel: one warp per (batch, query head, row), 32 keys per step,
// online softmax in registers.
#include "common.cuh"
#include "internal.h"

namespace mars {

namespace {

struct DualArgs {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  float* o;
  int batch, L, B, hq, hkv, G;
  float scale;
};

template <int D>
__device__ void attend_range(const DualArgs& a, const float* qv, int b, int kvh, int j0,
                             int j1, float& m, float& l, float* acc) {
  const int lane = threadIdx.x & 31;
  const size_t rs = (size_t)a.hkv * D;           // row stride of k / v in elements
  const uint16_t* kb = a.k + ((size_t)b * 2 * a.L) * rs + (size_t)kvh * D;
  const uint16_t* vb = a.v + ((size_t)b * 2 * a.L) * rs + (size_t)kvh * D;
  for (int c0 = j0; c0 < j1; c0 += 32) {
    const int j = c0 + lane;
    float sc = -INFINITY;
    if (j < j1) {
      const uint16_t* kr = kb + (size_t)j * rs;
      float acc2 = 0.f;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        float kf[8];
        unpack8(*reinterpret_cast<const uint4*>(kr + c * 8), kf);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc2 = fmaf(qv[c * 8 + e], kf[e], acc2);
      }
      sc = acc2;
    }
    const float m_new = fmaxf(m, warp_max(sc));
    const float p = (j < j1) ? __expf(sc - m_new) : 0.f;
    const float alpha = (m == -INFINITY) ? 0.f : __expf(m - m_new);
    l = l * alpha + warp_sum(p);
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] *= alpha;
    const int n = min(32, j1 - c0);
    for (int jj = 0; jj < n; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const uint16_t* vr = vb + (size_t)(c0 + jj) * rs;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) acc[i] = fmaf(pj, bf16_to_f32(vr[lane + 32 * i]), acc[i]);
    }
    m = m_new;
  }
}

template <int D>
__global__ void __launch_bounds__(256) dual_stream_rowwise_kernel(DualArgs a) {
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int n = 2 * a.L;
  const long long total = (long long)a.batch * a.hq * n;
  if (gw >= total) return;
  const int i = (int)(gw % n);
  const int h = (int)((gw / n) % a.hq);
  const int b = (int)(gw / ((long long)n * a.hq));
  const int kvh = h / a.G;
  float qv[D];
  const uint16_t* qr = a.q + (((size_t)b * n + i) * a.hq + h) * D;
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    float f[8];
    unpack8(*reinterpret_cast<const uint4*>(qr + c * 8), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) qv[c * 8 + e] = f[e] * a.scale;
  }
  float m = -INFINITY, l = 0.f, acc[D / 32];
#pragma unroll
  for (int x = 0; x < D / 32; ++x) acc[x] = 0.f;
  if (i < a.L) {
    attend_range<D>(a, qv, b, kvh, 0, i + 1, m, l, acc);
  } else {
    const int t = i - a.L;
    const int bs = (t / a.B) * a.B;
    attend_range<D>(a, qv, b, kvh, 0, bs, m, l, acc);
    attend_range<D>(a, qv, b, kvh, a.L + bs, i + 1, m, l, acc);
  }
  float* orow = a.o + (((size_t)b * n + i) * a.hq + h) * D;
  const float inv = 1.f / l;
#pragma unroll
  for (int x = 0; x < D / 32; ++x) orow[lane + 32 * x] = acc[x] * inv;
}

}  // namespace

cudaError_t launch_dual_stream(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               float* o, int batch, int L, int B, int hq, int hkv, int d,
                               float scale, cudaStream_t stream) {
  DualArgs a{q, k, v, o, batch, L, B, hq, hkv, hq / hkv, scale};
  const long long warps = (long long)batch * hq * 2 * L;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  if (d == 64)
    dual_stream_rowwise_kernel<64><<<blocks, 256, 0, stream>>>(a);
  else
    dual_stream_rowwise_kernel<128><<<blocks, 256, 0, stream>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace mars
