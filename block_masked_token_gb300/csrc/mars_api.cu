// C ABI of libmars (declared in include/mars.h): argument validation on the host, then
// launches on the caller's stream. No allocation, no host synchronisation.
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace mars {

namespace {

// Thread 0 waits on a fresh mbarrier whose phase nothing completes.
__global__ void wait_timeout_check_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);
    sm100::fence_barrier_init();
    sm100::mbar_wait(&bar, 0, nullptr, status);   // gives up after the wait limit
  }
}

}  // namespace

cudaError_t launch_wait_timeout_check(int32_t* status, cudaStream_t stream) {
  wait_timeout_check_kernel<<<1, 32, 0, stream>>>(status);
  count_launches(1);
  return cudaGetLastError();
}
static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
}  // namespace mars

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MARS_OK : MARS_ECUDA; }

int check_heads(int hq, int hkv, int d) {
  if (hq <= 0 || hkv <= 0 || hq % hkv) return MARS_EINVAL;
  if (d != 64 && d != 128) return MARS_EUNSUPPORTED;
  return MARS_OK;
}

// Shared-memory bound of the decode split kernel: query rows per KV head.
constexpr int kMaxDecodeRows = 128;

}  // namespace

extern "C" {

size_t mars_workspace_bytes(int op, int batch, int B, int hq, int hkv, int d, int hidden,
                            int vocab, int max_len) {
  (void)hidden;
  if (batch <= 0 || B < 1) return 0;
  if (op == MARS_OP_DUAL_GRAD) {                 // B is the block size of mask M here
    if (check_heads(hq, hkv, d) != MARS_OK || max_len < 1) return 0;
    return mars::dual_grad_workspace_bytes(batch, max_len, B, hq, hkv, d);
  }
  if (B > 32) return 0;
  if (op == MARS_OP_DECODE_ATTN) {
    if (check_heads(hq, hkv, d) != MARS_OK || max_len < 0) return 0;
    return mars::plan_decode(batch, B, hq, hkv, d, max_len).ws_bytes;
  }
  if (op == MARS_OP_HEAD_ACCEPT) {
    if (vocab <= 0) return 0;
    return mars::head_workspace_bytes(batch, B, vocab);
  }
  if (op == MARS_OP_CE_LOSS) {
    if (vocab <= 0 || max_len < 1) return 0;
    return mars::ce_workspace_bytes(batch, max_len, vocab);
  }
  if (op == MARS_OP_CE_LOSS_GRAD) {
    if (vocab <= 0 || max_len < 1) return 0;
    return mars::ce_grad_workspace_bytes(batch, max_len, vocab);
  }
  return 0;
}

int mars_attn_dual_stream(const mars_bf16* q, const mars_bf16* k, const mars_bf16* v,
                          float* o, int batch, int L, int B, int hq, int hkv, int d,
                          float scale, int32_t* status, void* stream) {
  if (batch < 0 || L < 1 || B < 1) return MARS_EINVAL;
  int rc = check_heads(hq, hkv, d);
  if (rc) return rc;
  if (batch == 0) return MARS_OK;
  if (!q || !k || !v || !o) return MARS_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return MARS_EALIGN;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)d);
  if (isinf(scale)) return MARS_EINVAL;
  return cuda_rc(mars::launch_dual_stream(q, k, v, o, batch, L, B, hq, hkv, d, scale, status,
                                          static_cast<cudaStream_t>(stream)));
}

int mars_attn_dual_stream_lse(const mars_bf16* q, const mars_bf16* k, const mars_bf16* v,
                              float* o, float* lse, int batch, int L, int B, int hq, int hkv,
                              int d, float scale, int32_t* status, void* stream) {
  if (batch < 0 || L < 1 || B < 1) return MARS_EINVAL;
  int rc = check_heads(hq, hkv, d);
  if (rc) return rc;
  if (batch == 0) return MARS_OK;
  if (!q || !k || !v || !o || !lse) return MARS_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return MARS_EALIGN;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)d);
  if (isinf(scale)) return MARS_EINVAL;
  return cuda_rc(mars::launch_dual_stream(q, k, v, o, batch, L, B, hq, hkv, d, scale, status,
                                          static_cast<cudaStream_t>(stream), lse));
}

int mars_decode_attn(const mars_bf16* q, const mars_bf16* k_blk, const mars_bf16* v_blk,
                     const mars_bf16* k_pool, const mars_bf16* v_pool, int num_pages,
                     const int32_t* block_table, int max_pages_per_seq,
                     const int32_t* seq_lens, int max_len_hint, float* o, int batch, int B,
                     int hq, int hkv, int d, int page_size, float scale, void* workspace,
                     size_t ws_bytes, int32_t* status, void* stream) {
  if (batch < 0 || B < 1 || B > 32 || max_len_hint < 0 || num_pages < 0 ||
      max_pages_per_seq < 0)
    return MARS_EINVAL;
  int rc = check_heads(hq, hkv, d);
  if (rc) return rc;
  if (page_size != mars::kPageSize) return MARS_EUNSUPPORTED;
  if ((hq / hkv) * B > kMaxDecodeRows) return MARS_EUNSUPPORTED;
  if (batch == 0) return MARS_OK;
  if (!q || !k_blk || !v_blk || !o || !seq_lens || !workspace) return MARS_EINVAL;
  if (max_pages_per_seq > 0 && (!k_pool || !v_pool || !block_table)) return MARS_EINVAL;
  if (!aligned16(q) || !aligned16(k_blk) || !aligned16(v_blk) || !aligned16(o) ||
      !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(workspace))
    return MARS_EALIGN;
  const mars::DecodePlan plan = mars::plan_decode(batch, B, hq, hkv, d, max_len_hint);
  if (ws_bytes < plan.ws_bytes) return MARS_ENOSPACE;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)d);
  if (isinf(scale)) return MARS_EINVAL;
  return cuda_rc(mars::launch_decode_attn(q, k_blk, v_blk, k_pool, v_pool, num_pages,
                                          block_table, max_pages_per_seq, seq_lens, plan, o,
                                          batch, B, hq, hkv, d, scale, workspace, status,
                                          static_cast<cudaStream_t>(stream)));
}

int mars_decode_attn_block_cache(const mars_bf16* q, const mars_bf16* k_blk,
                                 const mars_bf16* v_blk, const mars_bf16* k_pool,
                                 const mars_bf16* v_pool, int num_pages,
                                 const int32_t* block_table, int max_pages_per_seq,
                                 const int32_t* seq_lens, int max_len_hint,
                                 const mars_bf16* k_stage, const mars_bf16* v_stage,
                                 const int32_t* block_fill, int B_cache, float* o, int batch,
                                 int B, int hq, int hkv, int d, int page_size, float scale,
                                 void* workspace, size_t ws_bytes, int32_t* status,
                                 void* stream) {
  if (batch < 0 || B < 1 || B > 32 || max_len_hint < 0 || num_pages < 0 ||
      max_pages_per_seq < 0)
    return MARS_EINVAL;
  if (B_cache < 8 || B_cache > 64 || B_cache % 8) return MARS_EUNSUPPORTED;
  int rc = check_heads(hq, hkv, d);
  if (rc) return rc;
  if (page_size != mars::kPageSize) return MARS_EUNSUPPORTED;
  if ((hq / hkv) * B > kMaxDecodeRows) return MARS_EUNSUPPORTED;
  if (batch == 0) return MARS_OK;
  if (!q || !k_blk || !v_blk || !o || !seq_lens || !workspace || !k_stage || !v_stage ||
      !block_fill)
    return MARS_EINVAL;
  if (max_pages_per_seq > 0 && (!k_pool || !v_pool || !block_table)) return MARS_EINVAL;
  if (!aligned16(q) || !aligned16(k_blk) || !aligned16(v_blk) || !aligned16(o) ||
      !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(workspace) ||
      !aligned16(k_stage) || !aligned16(v_stage))
    return MARS_EALIGN;
  const mars::DecodePlan plan = mars::plan_decode(batch, B, hq, hkv, d, max_len_hint);
  if (ws_bytes < plan.ws_bytes) return MARS_ENOSPACE;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)d);
  if (isinf(scale)) return MARS_EINVAL;
  return cuda_rc(mars::launch_decode_attn(q, k_blk, v_blk, k_pool, v_pool, num_pages,
                                          block_table, max_pages_per_seq, seq_lens, plan, o,
                                          batch, B, hq, hkv, d, scale, workspace, status,
                                          static_cast<cudaStream_t>(stream), k_stage, v_stage,
                                          block_fill, B_cache));
}

namespace {

int head_accept_checked(const mars_bf16* h, const mars_bf16* w, int batch, int B, int hidden,
                        int vocab, float tau, const float* taus, int32_t* tokens,
                        float* maxprob, int32_t* n_accept, void* workspace, size_t ws_bytes,
                        int32_t* status, void* stream) {
  if (batch < 0 || B < 1 || B > 32 || hidden < 8 || vocab < 1) return MARS_EINVAL;
  if (hidden % 8) return MARS_EUNSUPPORTED;
  if (batch == 0) return MARS_OK;
  if (!h || !w || !tokens || !maxprob || !n_accept || !workspace) return MARS_EINVAL;
  if (!aligned16(h) || !aligned16(w) || !aligned16(workspace)) return MARS_EALIGN;
  if (ws_bytes < mars::head_workspace_bytes(batch, B, vocab)) return MARS_ENOSPACE;
  return cuda_rc(mars::launch_head_accept(h, w, batch, B, hidden, vocab, tau, taus, tokens,
                                          maxprob, n_accept, workspace, status,
                                          static_cast<cudaStream_t>(stream)));
}

int kv_commit_checked(const mars_bf16* k_blk, const mars_bf16* v_blk, const int32_t* n_accept,
                      int32_t* seq_lens, const int32_t* block_table, int max_pages_per_seq,
                      mars_bf16* k_pool, mars_bf16* v_pool, int num_pages,
                      int32_t* commit_slots, int batch, int B, int hkv, int d, int page_size,
                      bool batch_sync, int32_t* status, void* stream) {
  if (batch < 0 || B < 1 || B > 32 || hkv < 1 || num_pages < 0 || max_pages_per_seq < 0)
    return MARS_EINVAL;
  if (d != 64 && d != 128) return MARS_EUNSUPPORTED;
  if (page_size != mars::kPageSize) return MARS_EUNSUPPORTED;
  if (batch == 0) return MARS_OK;
  if (!k_blk || !v_blk || !n_accept || !seq_lens || !block_table || !k_pool || !v_pool)
    return MARS_EINVAL;
  if (!aligned16(k_blk) || !aligned16(v_blk) || !aligned16(k_pool) || !aligned16(v_pool))
    return MARS_EALIGN;
  return cuda_rc(mars::launch_kv_commit(k_blk, v_blk, n_accept, seq_lens, block_table,
                                        max_pages_per_seq, k_pool, v_pool, num_pages,
                                        commit_slots, batch, B, hkv, d, batch_sync, status,
                                        static_cast<cudaStream_t>(stream)));
}

}  // namespace

int mars_head_accept(const mars_bf16* h, const mars_bf16* w, int batch, int B, int hidden,
                     int vocab, float tau, int32_t* tokens, float* maxprob,
                     int32_t* n_accept, void* workspace, size_t ws_bytes, int32_t* status,
                     void* stream) {
  if (isnan(tau) || isinf(tau)) return MARS_EINVAL;
  return head_accept_checked(h, w, batch, B, hidden, vocab, tau, nullptr, tokens, maxprob,
                             n_accept, workspace, ws_bytes, status, stream);
}

int mars_head_accept_per_request(const mars_bf16* h, const mars_bf16* w, int batch, int B,
                                 int hidden, int vocab, const float* taus, int32_t* tokens,
                                 float* maxprob, int32_t* n_accept, void* workspace,
                                 size_t ws_bytes, int32_t* status, void* stream) {
  if (batch > 0 && !taus) return MARS_EINVAL;
  return head_accept_checked(h, w, batch, B, hidden, vocab, 0.f, taus, tokens, maxprob,
                             n_accept, workspace, ws_bytes, status, stream);
}

int mars_kv_commit(const mars_bf16* k_blk, const mars_bf16* v_blk, const int32_t* n_accept,
                   int32_t* seq_lens, const int32_t* block_table, int max_pages_per_seq,
                   mars_bf16* k_pool, mars_bf16* v_pool, int num_pages,
                   int32_t* commit_slots, int batch, int B, int hkv, int d, int page_size,
                   int32_t* status, void* stream) {
  return kv_commit_checked(k_blk, v_blk, n_accept, seq_lens, block_table, max_pages_per_seq,
                           k_pool, v_pool, num_pages, commit_slots, batch, B, hkv, d,
                           page_size, false, status, stream);
}

int mars_kv_commit_batch_sync(const mars_bf16* k_blk, const mars_bf16* v_blk,
                              const int32_t* n_accept, int32_t* seq_lens,
                              const int32_t* block_table, int max_pages_per_seq,
                              mars_bf16* k_pool, mars_bf16* v_pool, int num_pages,
                              int32_t* commit_slots, int batch, int B, int hkv, int d,
                              int page_size, int32_t* status, void* stream) {
  return kv_commit_checked(k_blk, v_blk, n_accept, seq_lens, block_table, max_pages_per_seq,
                           k_pool, v_pool, num_pages, commit_slots, batch, B, hkv, d,
                           page_size, true, status, stream);
}

int mars_kv_commit_block(const mars_bf16* k_blk, const mars_bf16* v_blk,
                         const int32_t* n_accept, int32_t* seq_lens, int32_t* block_fill,
                         mars_bf16* k_stage, mars_bf16* v_stage, int B_cache,
                         int32_t* sync_state, const int32_t* block_table,
                         int max_pages_per_seq, mars_bf16* k_pool, mars_bf16* v_pool,
                         int num_pages, int32_t* commit_slots, int batch, int B, int hkv,
                         int d, int page_size, int32_t* status, void* stream) {
  if (batch < 0 || B < 1 || B > 32 || hkv < 1 || num_pages < 0 || max_pages_per_seq < 0)
    return MARS_EINVAL;
  if (B_cache < 8 || B_cache > 64 || B_cache % 8) return MARS_EUNSUPPORTED;
  if (d != 64 && d != 128) return MARS_EUNSUPPORTED;
  if (page_size != mars::kPageSize) return MARS_EUNSUPPORTED;
  if (batch == 0) return MARS_OK;
  if (!k_blk || !v_blk || !n_accept || !seq_lens || !block_fill || !k_stage || !v_stage ||
      !sync_state || !block_table || !k_pool || !v_pool)
    return MARS_EINVAL;
  if (!aligned16(k_blk) || !aligned16(v_blk) || !aligned16(k_pool) || !aligned16(v_pool) ||
      !aligned16(k_stage) || !aligned16(v_stage))
    return MARS_EALIGN;
  return cuda_rc(mars::launch_kv_commit_block(
      k_blk, v_blk, n_accept, seq_lens, block_fill, k_stage, v_stage, B_cache, sync_state,
      block_table, max_pages_per_seq, k_pool, v_pool, num_pages, commit_slots, batch, B, hkv,
      d, status, static_cast<cudaStream_t>(stream)));
}

namespace {

int dual_grad_checked(const mars_bf16* q, const mars_bf16* k, const mars_bf16* v,
                      const float* o, const float* d_o, const float* lse, int batch, int L,
                      int B, int hq, int hkv, int d, float scale, float* dq, float* dk,
                      float* dv, void* workspace, size_t ws_bytes, int32_t* status,
                      void* stream) {
  if (batch < 0 || L < 1 || B < 1) return MARS_EINVAL;
  int rc = check_heads(hq, hkv, d);
  if (rc) return rc;
  if (batch == 0) return MARS_OK;
  if (!q || !k || !v || !o || !d_o || !dq || !dk || !dv || !workspace) return MARS_EINVAL;
  if (lse && !aligned16(lse)) return MARS_EALIGN;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(d_o) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return MARS_EALIGN;
  if (ws_bytes < mars::dual_grad_workspace_bytes(batch, L, B, hq, hkv, d)) return MARS_ENOSPACE;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)d);
  if (isinf(scale)) return MARS_EINVAL;
  return cuda_rc(mars::launch_dual_stream_grad(q, k, v, o, d_o, batch, L, B, hq, hkv, d, scale,
                                               dq, dk, dv, workspace, status,
                                               static_cast<cudaStream_t>(stream), lse));
}

}  // namespace

int mars_attn_dual_stream_grad(const mars_bf16* q, const mars_bf16* k, const mars_bf16* v,
                               const float* o, const float* d_o, int batch, int L, int B,
                               int hq, int hkv, int d, float scale, float* dq, float* dk,
                               float* dv, void* workspace, size_t ws_bytes, int32_t* status,
                               void* stream) {
  return dual_grad_checked(q, k, v, o, d_o, nullptr, batch, L, B, hq, hkv, d, scale, dq, dk, dv,
                           workspace, ws_bytes, status, stream);
}

int mars_attn_dual_stream_grad_lse(const mars_bf16* q, const mars_bf16* k, const mars_bf16* v,
                                   const float* o, const float* d_o, const float* lse,
                                   int batch, int L, int B, int hq, int hkv, int d, float scale,
                                   float* dq, float* dk, float* dv, void* workspace,
                                   size_t ws_bytes, int32_t* status, void* stream) {
  if (batch > 0 && !lse) return MARS_EINVAL;
  return dual_grad_checked(q, k, v, o, d_o, lse, batch, L, B, hq, hkv, d, scale, dq, dk, dv,
                           workspace, ws_bytes, status, stream);
}

int mars_dual_stream_ce_loss(const mars_bf16* h, const mars_bf16* w, const int32_t* targets,
                             int batch, int L, int hidden, int vocab, float* loss,
                             float* row_ce, float* row_lse, void* workspace, size_t ws_bytes,
                             int32_t* status, void* stream) {
  if (batch < 0 || L < 1 || hidden < 8 || vocab < 1) return MARS_EINVAL;
  if (hidden % 8) return MARS_EUNSUPPORTED;
  if ((long long)batch * 2 * L > 0x7fffffffLL) return MARS_EINVAL;
  if (!loss) return MARS_EINVAL;
  if (batch == 0) return cuda_rc(cudaMemsetAsync(loss, 0, 3 * sizeof(float),
                                                 static_cast<cudaStream_t>(stream)));
  if (!h || !w || !targets || !workspace) return MARS_EINVAL;
  if (!aligned16(h) || !aligned16(w) || !aligned16(workspace)) return MARS_EALIGN;
  if (ws_bytes < mars::ce_workspace_bytes(batch, L, vocab)) return MARS_ENOSPACE;
  return cuda_rc(mars::launch_ce_loss(h, w, targets, batch, L, hidden, vocab, loss, row_ce,
                                      row_lse, workspace, status,
                                      static_cast<cudaStream_t>(stream)));
}

int mars_dual_stream_ce_loss_grad(const mars_bf16* h, const mars_bf16* w,
                                  const int32_t* targets, const float* row_lse, int batch,
                                  int L, int hidden, int vocab, float* dh, float* dw,
                                  void* workspace, size_t ws_bytes, int32_t* status,
                                  void* stream) {
  if (batch < 0 || L < 1 || hidden < 8 || vocab < 1) return MARS_EINVAL;
  if (hidden % 8 || vocab % 8) return MARS_EUNSUPPORTED;
  if ((long long)batch * 2 * L > 0x7fffffffLL) return MARS_EINVAL;
  if (batch == 0) return MARS_OK;
  if (!h || !w || !targets || !row_lse || !workspace) return MARS_EINVAL;
  if (!aligned16(h) || !aligned16(w) || !aligned16(workspace)) return MARS_EALIGN;
  if (ws_bytes < mars::ce_grad_workspace_bytes(batch, L, vocab)) return MARS_ENOSPACE;
  return cuda_rc(mars::launch_ce_loss_grad(h, w, targets, row_lse, batch, L, hidden, vocab, dh,
                                           dw, workspace, status,
                                           static_cast<cudaStream_t>(stream)));
}

const char* mars_strerror(int code) {
  switch (code) {
    case MARS_OK: return "ok";
    case MARS_EINVAL: return "invalid argument";
    case MARS_EALIGN: return "tensor base pointer not 16-byte aligned";
    case MARS_EUNSUPPORTED: return "unsupported size (d must be 64/128, page_size 16)";
    case MARS_ECUDA: return "CUDA launch failed";
    case MARS_ENOSPACE: return "workspace too small";
    default: return "unknown error";
  }
}

int mars_check_wait_timeout(int32_t* status, void* stream) {
  if (!status) return MARS_EINVAL;
  return cuda_rc(mars::launch_wait_timeout_check(status, static_cast<cudaStream_t>(stream)));
}

uint64_t mars_launch_count(void) { return mars::g_launches.load(std::memory_order_relaxed); }

const char* mars_version(void) { return "libmars sm_103a v2 (tcgen05/TMA kernels)"; }

}  // extern "C"
