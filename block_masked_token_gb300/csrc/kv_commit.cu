// Commit of the accepted tokens' K/V into the paged block-level cache.
//
// Follows the per-sequence reading of the block-level KV cache on the papernotes.org notes
// of "MARS: Enabling Autoregressive Models Multi-Token Generation" (Key design 4) and the
// gist.science explainer (2.D): after each step the N_s accepted positions join the
// cached prefix of sequence s. One CTA per sequence: thread 0 resolves the page/slot of
// each accepted row (and any unmapped page), then the CTA copies the rows with 16-byte
// vector loads/stores and finally advances seq_lens[s]. Memory-bound and tiny
// (<= B * hkv * d * 4 bytes per sequence); its cost is the launch.
//
// Batch-synchronised variant (Key design 4 of the notes, second paragraph: the batch
// advances by the smallest accepted count of the step, faster samples wait; gist.science
// explainer, 2.D): every sequence commits N_min = min over the batch of its N, which each
// CTA reduces from n_accept itself, so the variant costs no extra launch.
#include "common.cuh"
#include "internal.h"

namespace mars {

__global__ void __launch_bounds__(128) kv_commit_kernel(
    const uint16_t* __restrict__ k_blk, const uint16_t* __restrict__ v_blk,
    const int32_t* __restrict__ n_accept, int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ block_table, int max_pages, uint16_t* __restrict__ k_pool,
    uint16_t* __restrict__ v_pool, int num_pages, int32_t* __restrict__ commit_slots,
    int batch, int B, int hkv, int d, int batch_sync, int32_t* status) {
  __shared__ int s_slot[32];
  __shared__ int s_n;
  __shared__ int s_min;
  const int s = blockIdx.x;
  if (batch_sync) {
    if (threadIdx.x == 0) s_min = B;
    __syncthreads();
    int m = B;
    for (int i = threadIdx.x; i < batch; i += blockDim.x) {
      const int v = n_accept[i];
      m = min(m, v < 0 ? 0 : (v > B ? B : v));
    }
    atomicMin(&s_min, m);
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int P = seq_lens[s];
    int N = n_accept[s];
    N = N < 0 ? 0 : (N > B ? B : N);
    if (batch_sync) N = s_min;
    int done = N;
    int st = 0;
    for (int i = 0; i < B; ++i) {
      int slot = -1;
      if (i < done) {
        const int pos = P + i;
        const int lp = pos / kPageSize;
        if (pos < 0 || lp >= max_pages) {
          st |= MARS_ST_OVERFLOW;
          done = i;
        } else {
          const int page = block_table[(size_t)s * max_pages + lp];
          if (page < 0 || page >= num_pages) {
            st |= MARS_ST_NOPAGE;
            done = i;
          } else {
            slot = page * kPageSize + pos % kPageSize;
          }
        }
      }
      s_slot[i] = slot;
    }
    s_n = done;
    seq_lens[s] = P + done;
    if (st && status) atomicOr(status, st);
  }
  __syncthreads();
  const int n = s_n;
  const int vph = d / 8;                       // 16-byte vectors per head row
  const int total = n * hkv * vph;
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int i = idx / (hkv * vph);
    const int rem = idx - i * hkv * vph;
    const int h = rem / vph;
    const int c = rem - h * vph;
    const int gs = s_slot[i];
    const size_t page = (size_t)(gs / kPageSize);
    const int slot = gs % kPageSize;
    const size_t src = (((size_t)s * B + i) * hkv + h) * d + (size_t)c * 8;
    const size_t dst = ((page * hkv + h) * kPageSize + slot) * d + (size_t)c * 8;
    *reinterpret_cast<uint4*>(k_pool + dst) = *reinterpret_cast<const uint4*>(k_blk + src);
    *reinterpret_cast<uint4*>(v_pool + dst) = *reinterpret_cast<const uint4*>(v_blk + src);
  }
  if (commit_slots)
    for (int i = threadIdx.x; i < B; i += blockDim.x) commit_slots[(size_t)s * B + i] = s_slot[i];
}

cudaError_t launch_kv_commit(const uint16_t* k_blk, const uint16_t* v_blk,
                             const int32_t* n_accept, int32_t* seq_lens,
                             const int32_t* block_table, int max_pages, uint16_t* k_pool,
                             uint16_t* v_pool, int num_pages, int32_t* commit_slots,
                             int batch, int B, int hkv, int d, bool batch_sync,
                             int32_t* status, cudaStream_t stream) {
  kv_commit_kernel<<<batch, 128, 0, stream>>>(k_blk, v_blk, n_accept, seq_lens, block_table,
                                               max_pages, k_pool, v_pool, num_pages,
                                               commit_slots, batch, B, hkv, d,
                                               batch_sync ? 1 : 0, status);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace mars
