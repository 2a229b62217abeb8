// Decode-form attention: B [MASK] queries per sequence over the paged committed prefix
// plus the block's own keys, causal inside the block (gist.science explainer of "MARS:
// Enabling Autoregressive Models Multi-Token Generation", 2.C sliding window and 2.D
// block-level KV cache; papernotes.org notes, Key design 3 and 4).
//
// Split-KV: grid (split, kv head, sequence). Each CTA serves all G*B query rows that
// share one KV head (GQA grouping: every key/value byte is read from HBM once per
// group), streams its split of the keys in 32-key chunks through shared memory, keeps
// an online softmax per row and writes an unnormalised partial (m, l, O) to the
// workspace. A second kernel merges the splits.
#include "common.cuh"
#include "internal.h"

namespace mars {

namespace {

constexpr int kChunk = 32;          // keys staged per iteration
constexpr int kThreads = 256;       // 8 warps
constexpr int kTargetCtas = 4 * kNumSMs;

struct DecodeArgs {
  const uint16_t* q;
  const uint16_t* k_blk;
  const uint16_t* v_blk;
  const uint16_t* k_pool;
  const uint16_t* v_pool;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* ws;
  float* o;
  int32_t* status;
  int num_pages, max_pages, B, hq, hkv, G, R, split_len, nsplit;
  float scale;
};

// Partial record per (sequence, kv head, split, row): m, l, 2 pad, then O[D].
template <int D>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(DecodeArgs a) {
  extern __shared__ float smem[];
  float* q_s = smem;                             // [R][D], pre-scaled
  float* k_s = q_s + a.R * D;                    // [kChunk][D+1]
  float* v_s = k_s + kChunk * (D + 1);           // [kChunk][D]
  float* o_s = v_s + kChunk * D;                 // [R][D]
  float* m_s = o_s + a.R * D;                    // [R]
  float* l_s = m_s + a.R;                        // [R]
  int* valid_s = reinterpret_cast<int*>(l_s + a.R);   // [kChunk]

  const int sp = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = a.seq_lens[s];
  const int T = P + a.B;
  const int t0 = sp * a.split_len;
  const int t1 = (sp == a.nsplit - 1) ? T : min(T, t0 + a.split_len);

  for (int idx = threadIdx.x; idx < a.R * D; idx += kThreads) {
    const int r = idx / D, dd = idx - r * D;
    const int g = r / a.B, k = r - g * a.B;
    const int h = kvh * a.G + g;
    q_s[idx] = a.scale * bf16_to_f32(a.q[(((size_t)s * a.B + k) * a.hq + h) * D + dd]);
    o_s[idx] = 0.f;
  }
  for (int r = threadIdx.x; r < a.R; r += kThreads) {
    m_s[r] = -INFINITY;
    l_s[r] = 0.f;
  }
  int st = 0;
  for (int c0 = t0; c0 < t1; c0 += kChunk) {
    __syncthreads();
    // stage keys c0 .. c0+31 (prefix rows from the pool, block rows from k_blk)
    for (int idx = threadIdx.x; idx < kChunk * (D / 8); idx += kThreads) {
      const int j = idx / (D / 8), c = idx - j * (D / 8);
      const int t = c0 + j;
      float kf[8], vf[8];
      bool ok = false;
      if (t < t1) {
        const uint16_t *kp = nullptr, *vp = nullptr;
        if (t < P) {
          const int lp = t / kPageSize;
          const int page = lp < a.max_pages ? a.block_table[(size_t)s * a.max_pages + lp] : -1;
          if (lp >= a.max_pages) st |= MARS_ST_OVERFLOW;
          else if (page < 0 || page >= a.num_pages) st |= MARS_ST_NOPAGE;
          else {
            const size_t off = (((size_t)page * a.hkv + kvh) * kPageSize + t % kPageSize) * D;
            kp = a.k_pool + off;
            vp = a.v_pool + off;
          }
        } else {
          const size_t off = (((size_t)s * a.B + (t - P)) * a.hkv + kvh) * D;
          kp = a.k_blk + off;
          vp = a.v_blk + off;
        }
        if (kp) {
          unpack8(*reinterpret_cast<const uint4*>(kp + c * 8), kf);
          unpack8(*reinterpret_cast<const uint4*>(vp + c * 8), vf);
          ok = true;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        k_s[j * (D + 1) + c * 8 + e] = ok ? kf[e] : 0.f;
        v_s[j * D + c * 8 + e] = ok ? vf[e] : 0.f;
      }
      if (c == 0) valid_s[j] = ok;
    }
    __syncthreads();
    const int t = c0 + lane;
    for (int r = warp; r < a.R; r += kThreads / 32) {
      const int k = r % a.B;
      const bool vis = valid_s[lane] && (t < P || (t - P) <= k);
      float sc = -INFINITY;
      if (vis) {
        float acc = 0.f;
        const float* qr = q_s + r * D;
        const float* kr = k_s + lane * (D + 1);
#pragma unroll 16
        for (int dd = 0; dd < D; ++dd) acc = fmaf(qr[dd], kr[dd], acc);
        sc = acc;
      }
      const float cmax = warp_max(sc);
      const float m_old = m_s[r];
      const float m_new = fmaxf(m_old, cmax);
      if (m_new == -INFINITY) continue;
      const float p = vis ? __expf(sc - m_new) : 0.f;
      const float alpha = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
      const float psum = warp_sum(p);
      float* orow = o_s + r * D;
      for (int dd = lane; dd < D; dd += 32) {
        float acc = orow[dd] * alpha;
#pragma unroll 8
        for (int j = 0; j < kChunk; ++j) acc = fmaf(__shfl_sync(0xffffffffu, p, j), v_s[j * D + dd], acc);
        orow[dd] = acc;
      }
      __syncwarp();
      if (lane == 0) {
        m_s[r] = m_new;
        l_s[r] = l_s[r] * alpha + psum;
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (st && a.status) atomicOr(a.status, st);
  const size_t rec = D + 4;
  float* base = a.ws + ((((size_t)s * a.hkv + kvh) * a.nsplit + sp) * a.R) * rec;
  for (int r = threadIdx.x; r < a.R; r += kThreads) {
    base[r * rec + 0] = m_s[r];
    base[r * rec + 1] = l_s[r];
  }
  for (int idx = threadIdx.x; idx < a.R * D; idx += kThreads) {
    const int r = idx / D, dd = idx - r * D;
    base[r * rec + 4 + dd] = o_s[idx];
  }
}

// One warp per (sequence, query head, block position): merge the split partials.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(DecodeArgs a) {
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int batch_rows = gridDim.y;   // unused guard helper
  (void)batch_rows;
  const int s = blockIdx.y;
  if (gw >= a.hq * a.B) return;
  const int h = gw / a.B, k = gw - h * a.B;
  const int kvh = h / a.G, g = h - kvh * a.G;
  const int r = g * a.B + k;
  const size_t rec = D + 4;
  const float* base = a.ws + (((size_t)s * a.hkv + kvh) * a.nsplit) * a.R * rec + r * rec;
  float m = -INFINITY;
  for (int sp = 0; sp < a.nsplit; ++sp) m = fmaxf(m, base[sp * a.R * rec]);
  float l = 0.f;
  float acc[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
  for (int sp = 0; sp < a.nsplit; ++sp) {
    const float* pr = base + sp * a.R * rec;
    const float ms = pr[0];
    if (ms == -INFINITY) continue;
    const float w = __expf(ms - m);
    l += pr[1] * w;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] += pr[4 + lane + 32 * i] * w;
  }
  const float inv = 1.f / l;
  float* orow = a.o + (((size_t)s * a.B + k) * a.hq + h) * D;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) orow[lane + 32 * i] = acc[i] * inv;
}

template <int D>
size_t split_smem_bytes(int R) {
  return sizeof(float) * (size_t)(2 * R * D + kChunk * (D + 1) + kChunk * D + 2 * R) +
         sizeof(int) * kChunk;
}

}  // namespace

DecodePlan plan_decode(int batch, int B, int hq, int hkv, int d, int max_len) {
  DecodePlan p{};
  const long long T = (long long)max_len + B;
  const long long pairs = (long long)batch * hkv;
  long long per = (pairs * T + kTargetCtas - 1) / kTargetCtas;
  if (per < 256) per = 256;
  per = (per + 127) / 128 * 128;
  p.split_len = (int)per;
  p.nsplit = (int)((T + per - 1) / per);
  if (p.nsplit < 1) p.nsplit = 1;
  p.rows = (hq / hkv) * B;
  p.ws_bytes = (size_t)batch * hkv * p.nsplit * p.rows * (d + 4) * sizeof(float);
  return p;
}

cudaError_t launch_decode_attn(const uint16_t* q, const uint16_t* k_blk,
                               const uint16_t* v_blk, const uint16_t* k_pool,
                               const uint16_t* v_pool, int num_pages,
                               const int32_t* block_table, int max_pages,
                               const int32_t* seq_lens, const DecodePlan& plan, float* o,
                               int batch, int B, int hq, int hkv, int d, float scale,
                               void* workspace, int32_t* status, cudaStream_t stream) {
  DecodeArgs a{q, k_blk, v_blk, k_pool, v_pool, block_table, seq_lens,
               static_cast<float*>(workspace), o, status, num_pages, max_pages, B, hq, hkv,
               hq / hkv, plan.rows, plan.split_len, plan.nsplit, scale};
  dim3 grid(plan.nsplit, hkv, batch);
  dim3 cgrid((hq * B + 7) / 8, batch);
  if (d == 64) {
    const size_t sm = split_smem_bytes<64>(plan.rows);
    cudaFuncSetAttribute(decode_split_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    decode_split_kernel<64><<<grid, kThreads, sm, stream>>>(a);
    decode_combine_kernel<64><<<cgrid, 256, 0, stream>>>(a);
  } else {
    const size_t sm = split_smem_bytes<128>(plan.rows);
    cudaFuncSetAttribute(decode_split_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    decode_split_kernel<128><<<grid, kThreads, sm, stream>>>(a);
    decode_combine_kernel<128><<<cgrid, 256, 0, stream>>>(a);
  }
  count_launches(2);
  return cudaGetLastError();
}

}  // namespace mars
