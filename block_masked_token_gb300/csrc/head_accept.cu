// Decode-step epilogue: LM-head logits, per-position max-prob and argmax, and the
// left-to-right threshold acceptance (papernotes.org notes of "MARS: Enabling
// Autoregressive Models Multi-Token Generation", Key design 3; gist.science explainer,
// 2.C "Confidence Thresholding").
//
// One kernel: the tcgen05 LM-head GEMM of head_gemm_tc.cuh in its fused-acceptance mode.
// Each 128 x 256 tile of logits lives only in TMEM; the epilogue folds it into a running
// {max, sum exp(l - max), first argmax} per row, and the CTA that completes a row block
// merges the block's partial records, writes the tokens and max-probs = 1 / sum_v
// exp(l_v - max), and scans each sequence's B positions left to right: N = leading run of
// max-prob >= tau, at least 1, at most B. tau is one value per call, or one per sequence
// (per request: gist.science explainer, 2.C "Adaptive Throughput"; papernotes.org notes,
// highlights, third point). The counters the merge relies on are zeroed on the stream
// before the kernel (cudaMemsetAsync), so a workspace needs no preparation.
#include "common.cuh"
#include "head_gemm_tc.cuh"
#include "internal.h"

namespace mars {

namespace {

// Workspace of the fused head: counters (3 per row block), then the partial records
// (one per CTA and row block).
struct HeadLayout {
  int num_m, num_n, grid, max_rec;
  bool pair;             // the paired (two-SM) kernel: from two row blocks on
  int pair_grid;         // its CTAs, a whole number of pairs
  size_t sync_bytes, rec_bytes;
};

HeadLayout head_layout(int batch, int B, int vocab) {
  using namespace head_tc;
  HeadLayout L{};
  const long long rows = (long long)batch * B;
  L.num_m = (int)((rows + BM - 1) / BM);
  L.num_n = (vocab + BN - 1) / BN;
  const long long tiles = (long long)L.num_m * L.num_n;
  L.grid = (int)(tiles < num_sms() ? tiles : num_sms());
  // at most one record per CTA and row block; the paired grid meets a row block with at
  // most one CTA per pair, min(pair tiles, SMs / 2) <= grid
  L.max_rec = L.grid;
  L.pair = L.num_m >= 2;
  const long long pair_tiles = (long long)((L.num_m + 1) / 2) * L.num_n;
  const long long pairs = num_sms() / 2;
  L.pair_grid = 2 * (int)(pair_tiles < pairs ? pair_tiles : pairs);
  L.sync_bytes = ((size_t)3 * L.num_m * sizeof(uint32_t) + 255) / 256 * 256;
  L.rec_bytes = (size_t)L.num_m * L.max_rec * BM * sizeof(float4);
  return L;
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
  const HeadLayout L = head_layout(batch, B, vocab);
  return L.sync_bytes + L.rec_bytes;
}

cudaError_t launch_head_accept(const uint16_t* h, const uint16_t* w, int batch, int B,
                               int hidden, int vocab, float tau, const float* taus,
                               int32_t* tokens, float* maxprob, int32_t* n_accept,
                               void* workspace, int32_t* status, cudaStream_t stream) {
  using namespace head_tc;
  const int rows = batch * B;
  const HeadLayout L = head_layout(batch, B, vocab);
  CUtensorMap tm_h, tm_w;
  {
    const uint64_t dims[2] = {(uint64_t)hidden, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)hidden * 2};
    const uint32_t box[2] = {BK, BM};
    if (!encode_tmap_bf16(&tm_h, h, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    // paired: each CTA of a pair loads one half (128 vocabulary rows) of the W tile
    const uint64_t dims[2] = {(uint64_t)hidden, (uint64_t)vocab};
    const uint64_t strides[1] = {(uint64_t)hidden * 2};
    const uint32_t box[2] = {BK, (uint32_t)(L.pair ? BN / 2 : BN)};
    if (!encode_tmap_bf16(&tm_w, w, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  Params p{};
  p.rows = rows;
  p.hidden = hidden;
  p.vocab = vocab;
  p.num_m = L.num_m;
  p.num_n = L.num_n;
  p.num_k = L.pair ? (hidden + BK_P - 1) / BK_P : (hidden + BK - 1) / BK;
  p.num_mp = (p.num_m + 1) / 2;
  p.num_tiles = (L.pair ? p.num_mp : p.num_m) * p.num_n;
  p.part = nullptr;
  p.targets = nullptr;
  p.dlogits = nullptr;
  p.status = status;
  p.sync = static_cast<uint32_t*>(workspace);
  p.rec = reinterpret_cast<float4*>(static_cast<uint8_t*>(workspace) + L.sync_bytes);
  p.max_rec = L.max_rec;
  p.B = B;
  p.tau = tau;
  p.taus = taus;
  p.tokens = tokens;
  p.maxprob = maxprob;
  p.n_accept = n_accept;
  static std::atomic<int> attr[64], attr_pair[64];
  cudaError_t e = L.pair ? set_smem_limit_once(head_gemm_pair_kernel, (int)SMEM_FUSED_BYTES, attr_pair)
                         : set_smem_limit_once(head_gemm_kernel, (int)SMEM_FUSED_BYTES, attr);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.sync, 0, (size_t)3 * L.num_m * sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  if (L.pair)
    head_gemm_pair_kernel<<<L.pair_grid, NUM_THREADS, SMEM_FUSED_BYTES, stream>>>(tm_h, tm_w,
                                                                                 tm_w, p);
  else
    head_gemm_kernel<<<L.grid, NUM_THREADS, SMEM_FUSED_BYTES, stream>>>(tm_h, tm_w, tm_w, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace mars
