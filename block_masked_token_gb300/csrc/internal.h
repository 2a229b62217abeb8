// Internal launchers behind the C ABI (mars_api.cu). Arguments are validated there;
// every launcher enqueues on `stream` and returns the cudaError_t of its launches.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <stddef.h>
#include <stdint.h>

namespace mars {

// Host-side count of kernels enqueued by the library (read by mars_launch_count()).
void count_launches(int n);

// ---- KV commit ([notes] Key design 4): one CTA per sequence.
cudaError_t launch_kv_commit(const uint16_t* k_blk, const uint16_t* v_blk,
                             const int32_t* n_accept, int32_t* seq_lens,
                             const int32_t* block_table, int max_pages, uint16_t* k_pool,
                             uint16_t* v_pool, int num_pages, int32_t* commit_slots,
                             int batch, int B, int hkv, int d, bool batch_sync,
                             int32_t* status, cudaStream_t stream);

// ---- Block-level commit with a B_cache boundary (block buffer, batch-wide flush).
cudaError_t launch_kv_commit_block(const uint16_t* k_blk, const uint16_t* v_blk,
                                   const int32_t* n_accept, int32_t* seq_lens, int32_t* fill,
                                   uint16_t* k_stage, uint16_t* v_stage, int B_cache,
                                   int32_t* sync, const int32_t* block_table, int max_pages,
                                   uint16_t* k_pool, uint16_t* v_pool, int num_pages,
                                   int32_t* commit_slots, int batch, int B, int hkv, int d,
                                   int32_t* status, cudaStream_t stream);

// ---- Decode attention: split-KV partials then a combine pass.
struct DecodePlan {
  int split_len;   // keys per split (multiple of 128)
  int nsplit;      // splits per (sequence, kv head)
  int rows;        // query rows per (sequence, kv head) = (hq / hkv) * B
  bool ordered;    // CTAs take the sequences longest first (order array in the workspace)
  size_t order_bytes;
  size_t ws_bytes;
};
DecodePlan plan_decode(int batch, int B, int hq, int hkv, int d, int max_len);

cudaError_t launch_decode_attn(const uint16_t* q, const uint16_t* k_blk,
                               const uint16_t* v_blk, const uint16_t* k_pool,
                               const uint16_t* v_pool, int num_pages,
                               const int32_t* block_table, int max_pages,
                               const int32_t* seq_lens, const DecodePlan& plan, float* o,
                               int batch, int B, int hq, int hkv, int d, float scale,
                               void* workspace, int32_t* status, cudaStream_t stream,
                               const uint16_t* k_stage = nullptr,
                               const uint16_t* v_stage = nullptr,
                               const int32_t* stage_fill = nullptr, int B_cache = 0);

// ---- LM head + max-prob/argmax + acceptance.
size_t head_workspace_bytes(int batch, int B, int vocab);
// taus: one threshold per sequence (device, [batch]), or NULL to use tau for all.
cudaError_t launch_head_accept(const uint16_t* h, const uint16_t* w, int batch, int B,
                               int hidden, int vocab, float tau, const float* taus,
                               int32_t* tokens, float* maxprob, int32_t* n_accept,
                               void* workspace, int32_t* status, cudaStream_t stream);

// ---- Gradient of the dual-stream attention: a statistics-only forward run, then the
// tcgen05 dK/dV kernel over key tiles and the row-parallel tcgen05 dQ kernel.
size_t dual_grad_workspace_bytes(int batch, int L, int B, int hq, int hkv, int d);
cudaError_t launch_dual_stream_grad(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    const float* o, const float* d_o, int batch, int L, int B,
                                    int hq, int hkv, int d, float scale, float* dq, float* dk,
                                    float* dv, void* workspace, int32_t* status,
                                    cudaStream_t stream, const float* lse = nullptr);

// ---- Dual-stream training loss (L_mask + L_AR) over the 2L rows of each sequence.
size_t ce_workspace_bytes(int batch, int L, int vocab);
cudaError_t launch_ce_loss(const uint16_t* h, const uint16_t* w, const int32_t* targets,
                           int batch, int L, int hidden, int vocab, float* loss,
                           float* row_ce, float* row_lse, void* workspace, int32_t* status,
                           cudaStream_t stream);
size_t ce_grad_workspace_bytes(int batch, int L, int vocab);
cudaError_t launch_ce_loss_grad(const uint16_t* h, const uint16_t* w, const int32_t* targets,
                                const float* row_lse, int batch, int L, int hidden, int vocab,
                                float* dh, float* dw, void* workspace, int32_t* status,
                                cudaStream_t stream);

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

// Function attributes belong to the device they were set on: raise a kernel's dynamic
// shared-memory limit once per device (flags indexed by device ordinal).
template <class Kernel>
cudaError_t set_smem_limit_once(Kernel* fn, int bytes, std::atomic<int> (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(1, std::memory_order_release);
  return e;
}

// ---- One CTA waiting on an mbarrier that nothing completes (the wait-limit self-check).
cudaError_t launch_wait_timeout_check(int32_t* status, cudaStream_t stream);

// ---- Dual-stream attention under mask M. o may be null when lse is given (the row
// statistics alone: lse[b][h][stream][t], t < Lp = L rounded up to 128, = log2 of the
// softmax denominator in units of scale*log2(e)*score; pad rows are written as 0).
cudaError_t launch_dual_stream(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               float* o, int batch, int L, int B, int hq, int hkv, int d,
                               float scale, int32_t* status, cudaStream_t stream,
                               float* lse = nullptr);

// dQ of the dual-stream attention gradient from the forward's row statistics: lse and
// D = rowsum(dO * O) as [b][hq][2][Lp] fp32, dO in bf16 like q. Writes every row of dq.
cudaError_t launch_dual_stream_dq(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  const uint16_t* do_bf, const float* lse, const float* drow,
                                  float* dq, int batch, int L, int B, int hq, int hkv, int d,
                                  float scale, int32_t* status, cudaStream_t stream);

}  // namespace mars
