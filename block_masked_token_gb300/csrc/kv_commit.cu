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

// Block-level commit with a batch-wide B_cache boundary (Key design 4 of the notes, both
// paragraphs: the prefix cache is frozen in blocks of B_cache tokens, samples that fill
// their block first wait at the boundary, and once every sample has filled it the whole
// block is written to the persistent cache; gist.science explainer, 2.D). One CTA per
// sequence. Accepted rows go to the sequence's block buffer (stage); the pool is written
// only in whole blocks. Whether every block is full is known only once every CTA has
// taken its rows, so the last CTA to finish (an atomic ticket, no waiting) records it in
// sync[0], and the next call's CTAs write their blocks to the pool before taking new
// rows. Between the two calls the decode attention reads the full block from the stage,
// so it sees the same keys as if the block were already in the pool.
//   sync[0] = every block full after the previous call (the flush is pending)
//   sync[1] = CTAs of this call that have finished (the ticket; reset by the last one)
//   sync[2] = sequences whose block is full (reset when the blocks are written)
__global__ void __launch_bounds__(128) kv_commit_block_kernel(
    const uint16_t* __restrict__ k_blk, const uint16_t* __restrict__ v_blk,
    const int32_t* __restrict__ n_accept, int32_t* __restrict__ seq_lens,
    int32_t* __restrict__ fill, uint16_t* __restrict__ k_stage, uint16_t* __restrict__ v_stage,
    int B_cache, int32_t* sync, const int32_t* __restrict__ block_table, int max_pages,
    uint16_t* __restrict__ k_pool, uint16_t* __restrict__ v_pool, int num_pages,
    int32_t* __restrict__ commit_slots, int batch, int B, int hkv, int d, int32_t* status) {
  __shared__ int s_slot[64];
  __shared__ int s_flush, s_nflush, s_fill0, s_n;
  __shared__ int s_slot_new[32];
  const int s = blockIdx.x;
  const int vph = d / 8;                       // 16-byte vectors per head row
  const size_t row_elems = (size_t)hkv * d;    // one row of k_blk / stage
  // page slot of logical position pos of this sequence, or -1 (and a status bit)
  auto slot_of = [&](int pos, int& st) -> int {
    const int lp = pos / kPageSize;
    if (pos < 0 || lp >= max_pages) {
      st |= MARS_ST_OVERFLOW;
      return -1;
    }
    const int page = block_table[(size_t)s * max_pages + lp];
    if (page < 0 || page >= num_pages) {
      st |= MARS_ST_NOPAGE;
      return -1;
    }
    return page * kPageSize + pos % kPageSize;
  };
  if (threadIdx.x == 0) {
    int st = 0;
    const int P = seq_lens[s];
    int F = fill[s];
    F = F < 0 ? 0 : (F > B_cache ? B_cache : F);
    // 1. the blocks were all full after the previous call: write this one to the pool
    const int flush = *reinterpret_cast<volatile int32_t*>(sync) != 0;
    int nflush = 0;
    if (flush) {
      for (int i = 0; i < B_cache; ++i) {
        const int sl = slot_of(P + i, st);
        if (sl < 0) break;                     // an unmapped page ends the block's write
        s_slot[i] = sl;
        nflush = i + 1;
      }
      F = 0;
    }
    const int P1 = P + nflush;
    // 2. this step's accepted rows, as many as the block can still take
    int N = n_accept[s];
    N = N < 0 ? 0 : (N > B ? B : N);
    int n = min(N, B_cache - F);
    for (int i = 0; i < B; ++i) {
      int sl = -1;
      if (i < n) {
        sl = slot_of(P1 + F + i, st);
        if (sl < 0) n = i;
      }
      s_slot_new[i] = sl;
    }
    s_flush = flush;
    s_nflush = nflush;
    s_fill0 = F;
    s_n = n;
    seq_lens[s] = P1;
    fill[s] = F + n;
    if (st && status) atomicOr(status, st);
  }
  __syncthreads();
  const int nflush = s_nflush, F = s_fill0, n = s_n;
  // block buffer -> pool (all stage reads of the flush happen before the appends below)
  for (int idx = threadIdx.x; idx < nflush * hkv * vph; idx += blockDim.x) {
    const int i = idx / (hkv * vph);
    const int rem = idx - i * hkv * vph;
    const int h = rem / vph, c = rem - h * vph;
    const int gs = s_slot[i];
    const size_t src = ((size_t)s * B_cache + i) * row_elems + (size_t)h * d + (size_t)c * 8;
    const size_t dst = (((size_t)(gs / kPageSize) * hkv + h) * kPageSize + gs % kPageSize) * d +
                       (size_t)c * 8;
    *reinterpret_cast<uint4*>(k_pool + dst) = *reinterpret_cast<const uint4*>(k_stage + src);
    *reinterpret_cast<uint4*>(v_pool + dst) = *reinterpret_cast<const uint4*>(v_stage + src);
  }
  __syncthreads();
  // accepted rows -> block buffer rows F .. F + n - 1
  for (int idx = threadIdx.x; idx < n * hkv * vph; idx += blockDim.x) {
    const int i = idx / (hkv * vph);
    const int rem = idx - i * hkv * vph;
    const size_t src = ((size_t)s * B + i) * row_elems + (size_t)rem * 8;
    const size_t dst = ((size_t)s * B_cache + F + i) * row_elems + (size_t)rem * 8;
    *reinterpret_cast<uint4*>(k_stage + dst) = *reinterpret_cast<const uint4*>(k_blk + src);
    *reinterpret_cast<uint4*>(v_stage + dst) = *reinterpret_cast<const uint4*>(v_blk + src);
  }
  if (commit_slots)
    for (int i = threadIdx.x; i < B; i += blockDim.x)
      commit_slots[(size_t)s * B + i] = s_slot_new[i];
  __syncthreads();
  // 3. the ticket: the last CTA records whether every block is now full
  if (threadIdx.x == 0) {
    if (F + n == B_cache && (F < B_cache || s_flush)) {
      __threadfence();
      atomicAdd(&sync[2], 1);
    }
    __threadfence();
    const int ticket = atomicAdd(&sync[1], 1);
    if (ticket == batch - 1) {
      __threadfence();
      const int full = atomicAdd(&sync[2], 0);
      const int all = full >= batch;
      if (all) atomicExch(&sync[2], 0);
      atomicExch(&sync[0], all);
      atomicExch(&sync[1], 0);
    }
  }
}

cudaError_t launch_kv_commit_block(const uint16_t* k_blk, const uint16_t* v_blk,
                                   const int32_t* n_accept, int32_t* seq_lens, int32_t* fill,
                                   uint16_t* k_stage, uint16_t* v_stage, int B_cache,
                                   int32_t* sync, const int32_t* block_table, int max_pages,
                                   uint16_t* k_pool, uint16_t* v_pool, int num_pages,
                                   int32_t* commit_slots, int batch, int B, int hkv, int d,
                                   int32_t* status, cudaStream_t stream) {
  kv_commit_block_kernel<<<batch, 128, 0, stream>>>(
      k_blk, v_blk, n_accept, seq_lens, fill, k_stage, v_stage, B_cache, sync, block_table,
      max_pages, k_pool, v_pool, num_pages, commit_slots, batch, B, hkv, d, status);
  count_launches(1);
  return cudaGetLastError();
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
