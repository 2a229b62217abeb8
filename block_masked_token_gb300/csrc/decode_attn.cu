// Decode-form attention: B [MASK] queries per sequence over the paged committed prefix
// plus the block's own keys, causal inside the block (gist.science explainer of "MARS:
// Enabling Autoregressive Models Multi-Token Generation", 2.C sliding window and 2.D
// block-level KV cache; papernotes.org notes, Key design 3 and 4).
//
// Split-KV over the prefix: grid (split, kv head, sequence). A CTA stacks the G*B query
// rows that share one KV head (row r = block position r / G, head kvh*G + r % G) into one
// 128-row tile, so every key/value byte is read from HBM once per KV head, and runs the
// tcgen05 flash engine (flash_tc.cuh) over its split: prefix tiles of 128 keys gathered
// page by page from the paged pool (8 producer lanes, one 16-token page each, TMA with
// 128-byte swizzle), and for the last split one more tile with the B block keys (causal:
// query k sees block keys 0..k). With several splits each writes an unnormalised partial
// (m in log2 units, l, O) to the workspace and a second kernel merges them. Splits are
// used only when there are fewer (sequence, kv head) pairs than SMs and the prefixes are
// long (each split at least kMinSplitKeys keys); otherwise there is one split per pair and
// its CTA writes the normalised output directly. When the CTAs take more than one wave, a
// small kernel first orders the sequences by length so that the longest start first.
#include <climits>

#include "common.cuh"
#include "flash_tc.cuh"
#include "internal.h"

namespace mars {

namespace {

using flash::BKV;
using flash::BQ;

// Split-KV sizing. A split costs a partial record and a merge launch, which at 7B shapes
// outweighs the balance it buys unless a split still streams at least this many keys:
// with batch 32 and prefixes up to 2048, one split per (sequence, kv head) ran in 33 us
// against 46-50 us with 2 to 4 splits and the merge.
constexpr int kMinSplitKeys = 2048;
// Largest batch whose CTAs are ordered by sequence length (the order is built in shared
// memory by one CTA); larger batches run in index order.
constexpr int kMaxOrderBatch = 4096;
constexpr int kPagesPerTile = BKV / kPageSize;   // 8
// V-ring depth: one more than the engine's default (the decode CTA has no O staging area,
// so Q, three K stages and three V stages fill its shared memory). With two, a V slot came
// free only when the PV two tiles back had completed, and each tile waited about one
// DRAM round trip of its own.
constexpr int kVStages = 3;

struct DecodeArgs {
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* order;  // sequences by decreasing length (CTA z -> sequence), or NULL
  float* ws;
  float* o;
  int32_t* status;
  int num_pages, max_pages, B, hq, hkv, G, R, split_len, nsplit;
  float scale_log2;
  // block-level cache: rows accepted into each sequence's block buffer and not yet in the
  // pool (stage_fill[s] of B_cache), read between the prefix and the block keys; NULL
  // without a block buffer
  const int32_t* stage_fill;
  int B_cache;
};

MARS_DEV bool page_ok(const DecodeArgs& a, const int32_t* bt_row, int lp) {
  if (lp >= a.max_pages) return false;
  const int e = bt_row[lp];
  return e >= 0 && e < a.num_pages;
}

template <int D>
struct DecodePolicy {
  static constexpr bool kHandOff = false;
  static constexpr bool kRowStats = false;
  const DecodeArgs* a;
  const int32_t* bt_row;
  float* part;           // [R][D + 4] records of this (sequence, kv head, split)
  int P, start, n_prefix;
  int fill;              // buffered block rows visible before the block keys
  int s_idx, s_kvh;      // sequence and kv head of this CTA

  struct Tile {
    int kp0;             // logical key position of column 0
    uint32_t pmask;      // prefix tile: bit i = page i of the tile is mapped
    bool block;          // the block-key tile
    bool full;
  };
  MARS_DEV bool row_valid(int row) const { return row < a->R; }
  MARS_DEV flash::RowVis row_vis(int row) const { return {P, P, P + row / a->G}; }
  MARS_DEV Tile tile(int j) const {
    Tile t;
    if (j < n_prefix) {
      t.kp0 = start + j * BKV;
      t.block = false;
      t.pmask = 0;
      for (int i = 0; i < kPagesPerTile; ++i)
        if (page_ok(*a, bt_row, t.kp0 / kPageSize + i)) t.pmask |= 1u << i;
      t.full = (t.kp0 + BKV <= P) && t.pmask == 0xffu;
    } else {
      t.kp0 = P;
      t.block = true;
      t.pmask = 0;
      t.full = false;
    }
    return t;
  }
  MARS_DEV flash::ColRange cols(const flash::RowVis& v, const Tile& t) const {
    flash::ColRange c;
    c.s2 = BKV;
    c.e2 = -1;
    if (t.block && a->stage_fill) {      // buffered rows [0, fill), block keys 0..k at B_cache
      c.e1 = fill;
      c.s2 = a->B_cache;
      c.e2 = a->B_cache + (v.hi2 - P);
      c.pmask = 0xffu;
    } else if (t.block) {                // block keys 0..k (k = v.hi2 - P)
      c.e1 = v.hi2 - P + 1;
      c.pmask = 0xffu;
    } else {                             // prefix keys below P on mapped pages
      c.e1 = min(P - t.kp0, BKV);
      c.pmask = t.pmask;
    }
    return c;
  }
  MARS_DEV void store_chunk(int row, int col, const uint32_t (&r)[32], float inv, float m,
                            float l) const {
    if (a->nsplit == 1) {            // the only split: final output, normalised
      const int k = row / a->G, h = s_kvh * a->G + row % a->G;
      float* dst = a->o + (((size_t)s_idx * a->B + k) * a->hq + h) * D + col;
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4*>(dst + e) =
            make_float4(__uint_as_float(r[e]) * inv, __uint_as_float(r[e + 1]) * inv,
                        __uint_as_float(r[e + 2]) * inv, __uint_as_float(r[e + 3]) * inv);
      return;
    }
    float* rec = part + (size_t)row * (D + 4);
    if (col == 0) {
      rec[0] = m;
      rec[1] = l;
    }
#pragma unroll
    for (int e = 0; e < 32; e += 4)
      *reinterpret_cast<float4*>(rec + 4 + col + e) =
          make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                      __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
  }
};

template <int D>
__global__ void __launch_bounds__(flash::NUM_THREADS, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_kp,
                 const __grid_constant__ CUtensorMap tm_vp,
                 const __grid_constant__ CUtensorMap tm_kb,
                 const __grid_constant__ CUtensorMap tm_vb,
                 const __grid_constant__ CUtensorMap tm_ks,
                 const __grid_constant__ CUtensorMap tm_vs, DecodeArgs a) {
  using namespace sm100;
  using S = flash::Smem<D, 0, kVStages>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ flash::Barriers bar;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sp = blockIdx.x, kvh = blockIdx.y;
  const int s = a.order ? a.order[blockIdx.z] : (int)blockIdx.z;

  // Start what the first tile waits for at once: the loaders' block-table entries of prefix
  // tile 0 (its pages do not depend on the length) and the tensor maps, so that their
  // latencies overlap the length's and the set-up below.
  const int32_t* bt_row = a.block_table + (size_t)s * a.max_pages;
  int bt0 = INT_MIN;
  if ((warp == 0 || warp == flash::V_LOADER_WARP) && lane < kPagesPerTile) {
    const int lp = (sp * a.split_len) / kPageSize + lane;
    if (lp < a.max_pages) bt0 = bt_row[lp];
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_kp);
    prefetch_tmap(&tm_vp);
    prefetch_tmap(&tm_kb);
    prefetch_tmap(&tm_vb);
    if (a.stage_fill) {
      prefetch_tmap(&tm_ks);
      prefetch_tmap(&tm_vs);
    }
  }

  DecodePolicy<D> pol;
  pol.a = &a;
  pol.bt_row = bt_row;
  pol.part = a.ws + ((((size_t)s * a.hkv + kvh) * a.nsplit + sp) * a.R) * (D + 4);
  pol.P = a.seq_lens[s];
  pol.fill = a.stage_fill ? min(max(a.stage_fill[s], 0), a.B_cache) : 0;
  pol.s_idx = s;
  pol.s_kvh = kvh;
  pol.start = sp * a.split_len;
  const bool last = sp == a.nsplit - 1;
  const int end = last ? pol.P : min(pol.P, pol.start + a.split_len);
  pol.n_prefix = end > pol.start ? (end - pol.start + BKV - 1) / BKV : 0;
  const int n_total = pol.n_prefix + (last ? 1 : 0);
  if (n_total == 0) {                // split past this sequence's prefix: empty partial
    for (int r = threadIdx.x; r < a.R; r += blockDim.x) {
      pol.part[(size_t)r * (D + 4)] = -INFINITY;
      pol.part[(size_t)r * (D + 4) + 1] = 0.f;
    }
    return;
  }

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  if (threadIdx.x == 0) flash::init_barriers(bar);
  if (warp == 1) {
    tmem_alloc(&bar.tmem_base, S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // read once per warp and broadcast: a warp-uniform TMEM base keeps the MMA operands in
  // uniform registers, which tcgen05.mma issue depends on for its rate
  const uint32_t tmem = __shfl_sync(0xffffffffu, bar.tmem_base, 0);

  if (warp == 0 || warp == flash::V_LOADER_WARP) {
    // --------------------------------------------- loaders: K ring (warp 0, and Q first),
    // V ring (its own warp)
    const bool is_v = warp == flash::V_LOADER_WARP;
    if (!is_v && lane == 0) {
      mbar_arrive_expect_tx(&bar.q_full, a.R * 128 * (D / 64));
      for (int x = 0; x < D / 64; ++x)
        tma_load_3d(smem + S::OFF_Q + x * (BQ * 128), &tm_q, &bar.q_full, x * 64, kvh * a.G,
                    s * a.B);
    }
    int st_flags = 0;
    // block-table entry of this lane's page in prefix tile j (INT_MIN past the table); the
    // entry of the next tile is read as each tile is issued, so its latency overlaps the
    // wait for the next free ring slot instead of delaying that tile's copies
    auto entry = [&](int j) -> int {
      if (j >= pol.n_prefix || lane >= kPagesPerTile) return 0;
      const int lp = (pol.start + j * BKV) / kPageSize + lane;
      return lp < a.max_pages ? pol.bt_row[lp] : INT_MIN;
    };
    int next_entry = (pol.n_prefix > 0 && lane < kPagesPerTile) ? bt0 : 0;   // entry(0)
    // prefix tile j: lane i < 8 copies 16-token page i of the tile (unmapped pages load
    // page 0 and are masked by the softmax); the block tile: lane 0 copies a 128-row box
    // from row s*B of k_blk / v_blk (rows past the batch read as zeros), or, with a block
    // buffer, its B_cache rows into tile rows 0..B_cache-1 and a (128 - B_cache)-row box of
    // k_blk / v_blk after them
    auto issue = [&](const CUtensorMap* tm_pool, const CUtensorMap* tm_blk,
                     const CUtensorMap* tm_stage) {
      return [&, tm_pool, tm_blk, tm_stage](int j, uint8_t* dst, uint64_t* b) {
        const int e = next_entry;
        next_entry = entry(j + 1);
        if (j < pol.n_prefix) {
          if (lane < kPagesPerTile) {
            const int kp = pol.start + j * BKV + lane * kPageSize;
            int page = 0;
            if (e >= 0 && e < a.num_pages) {
              page = e;
            } else if (kp < pol.P) {
              st_flags |= e == INT_MIN ? MARS_ST_OVERFLOW : MARS_ST_NOPAGE;
            }
            // with an empty pool the map (over q, one page long) is never read: the box
            // starts past its end and loads zeros
            const int row = a.num_pages > 0 ? (page * a.hkv + kvh) * kPageSize : kPageSize;
            for (int x = 0; x < D / 64; ++x)
              tma_load_2d(dst + x * (BKV * 128) + lane * (kPageSize * 128), tm_pool, b, x * 64,
                          row);
          }
        } else if (lane == 0) {
          for (int x = 0; x < D / 64; ++x) {
            uint8_t* reg = dst + x * (BKV * 128);
            if (a.stage_fill) {
              tma_load_3d(reg, tm_stage, b, x * 64, kvh, s * a.B_cache);
              tma_load_3d(reg + a.B_cache * 128, tm_blk, b, x * 64, kvh, s * a.B);
            } else {
              tma_load_3d(reg, tm_blk, b, x * 64, kvh, s * a.B);
            }
          }
        }
      };
    };
    if (is_v)
      flash::load_ring<D, kVStages>(bar, smem, n_total, a.status, true,
                                    issue(&tm_vp, &tm_vb, &tm_vs));
    else
      flash::load_ring<D, kVStages>(bar, smem, n_total, a.status, false,
                                    issue(&tm_kp, &tm_kb, &tm_ks));
    if (!is_v && lane == 0) mbar_wait(&bar.q_full, 0, nullptr, a.status);
    if (st_flags && a.status) atomicOr(a.status, st_flags);
  } else if (warp == 1 || warp == flash::PV_ISSUER_WARP) {
    // one thread issues both QK^T and PV (short tile lists); the PV warp idles
    if (warp == 1 && lane == 0)
      flash::single_issuer<D, kVStages>(bar, smem, n_total, tmem, a.status);
  } else {
    flash::softmax_loop<D>(bar, smem, pol, n_total, tmem, a.scale_log2, a.status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S::TMEM_COLS);
  }
}

// One warp per (sequence, query head, block position): merge the split partials.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(DecodeArgs a) {
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int s = blockIdx.y;
  if (gw >= a.hq * a.B) return;
  const int h = gw / a.B, k = gw - h * a.B;
  const int kvh = h / a.G, g = h - kvh * a.G;
  const int r = k * a.G + g;
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
    const float w = exp2f(ms - m);
    l += pr[1] * w;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] += pr[4 + lane + 32 * i] * w;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float* orow = a.o + (((size_t)s * a.B + k) * a.hq + h) * D;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) orow[lane + 32 * i] = acc[i] * inv;
}

// Longest sequences first: CTAs start in blockIdx order, so this keeps the long pairs out
// of the last wave, which otherwise leaves SMs idle while a few long CTAs finish. One CTA;
// rank_i = #{j : len_j > len_i, or len_j == len_i and j < i}; order[rank_i] = i.
__global__ void __launch_bounds__(1024) decode_order_kernel(const int32_t* __restrict__ seq_lens,
                                                            int batch,
                                                            int32_t* __restrict__ order) {
  __shared__ int lens[kMaxOrderBatch];
  for (int i = threadIdx.x; i < batch; i += blockDim.x) lens[i] = seq_lens[i];
  __syncthreads();
  for (int i = threadIdx.x; i < batch; i += blockDim.x) {
    const int li = lens[i];
    int rank = 0;
    for (int j = 0; j < batch; ++j) {
      const int lj = lens[j];
      rank += (lj > li) || (lj == li && j < i);
    }
    order[rank] = i;
  }
}

template <int D>
cudaError_t launch_tc(const uint16_t* q, const uint16_t* k_blk, const uint16_t* v_blk,
                      const uint16_t* k_pool, const uint16_t* v_pool, const uint16_t* k_stage,
                      const uint16_t* v_stage, DecodeArgs& a, int batch, cudaStream_t stream) {
  using S = flash::Smem<D, 0, kVStages>;
  CUtensorMap tq, tkp, tvp, tkb, tvb;
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.hq, (uint64_t)batch * a.B};
    const uint64_t str[2] = {(uint64_t)D * 2, (uint64_t)a.hq * D * 2};
    const uint32_t box[3] = {64, (uint32_t)a.G, (uint32_t)a.B};
    if (!encode_tmap_bf16(&tq, q, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t rows = (uint64_t)(a.num_pages > 0 ? a.num_pages : 1) * a.hkv * kPageSize;
    const uint64_t dims[2] = {(uint64_t)D, rows};
    const uint64_t str[1] = {(uint64_t)D * 2};
    const uint32_t box[2] = {64, (uint32_t)kPageSize};
    // an empty pool is never read (its boxes start past the end, see the loader); encode
    // over q instead
    const void* kp = a.num_pages > 0 ? (const void*)k_pool : (const void*)q;
    const void* vp = a.num_pages > 0 ? (const void*)v_pool : (const void*)q;
    const uint64_t dims_e[2] = {(uint64_t)D, (uint64_t)kPageSize};
    if (!encode_tmap_bf16(&tkp, kp, 2, a.num_pages > 0 ? dims : dims_e, str, box))
      return cudaErrorInvalidValue;
    if (!encode_tmap_bf16(&tvp, vp, 2, a.num_pages > 0 ? dims : dims_e, str, box))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.hkv, (uint64_t)batch * a.B};
    const uint64_t str[2] = {(uint64_t)D * 2, (uint64_t)a.hkv * D * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)(a.stage_fill ? BKV - a.B_cache : BKV)};
    if (!encode_tmap_bf16(&tkb, k_blk, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_tmap_bf16(&tvb, v_blk, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  CUtensorMap tks = tkb, tvs = tvb;        // unused without a block buffer
  if (a.stage_fill) {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.hkv, (uint64_t)batch * a.B_cache};
    const uint64_t str[2] = {(uint64_t)D * 2, (uint64_t)a.hkv * D * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)a.B_cache};
    if (!encode_tmap_bf16(&tks, k_stage, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_tmap_bf16(&tvs, v_stage, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  static std::atomic<int> attr[64];
  const cudaError_t ea = set_smem_limit_once(decode_tc_kernel<D>, S::TOTAL, attr);
  if (ea != cudaSuccess) return ea;
  dim3 grid(a.nsplit, a.hkv, batch);
  decode_tc_kernel<D><<<grid, flash::NUM_THREADS, S::TOTAL, stream>>>(tq, tkp, tvp, tkb, tvb,
                                                                      tks, tvs, a);
  if (a.nsplit > 1) {
    dim3 cgrid((a.hq * a.B + 7) / 8, batch);
    decode_combine_kernel<D><<<cgrid, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

DecodePlan plan_decode(int batch, int B, int hq, int hkv, int d, int max_len) {
  DecodePlan p{};
  const long long T = (long long)max_len > 0 ? max_len : 1;
  const long long pairs = (long long)batch * hkv;
  const long long sms = num_sms();
  // one split per (sequence, kv head) when the pairs fill the GPU; otherwise enough splits
  // for about one wave of CTAs, but only as many as keep every split at least
  // kMinSplitKeys long (none when the prefixes are shorter than two such splits)
  long long nsplit = 1;
  if (pairs < sms) {
    const long long want = (sms + pairs - 1) / pairs;
    const long long most = T / kMinSplitKeys;
    nsplit = want < most ? want : most;
    if (nsplit < 1) nsplit = 1;
  }
  long long per = (T + nsplit - 1) / nsplit;
  per = (per + BKV - 1) / BKV * BKV;
  p.split_len = (int)per;
  p.nsplit = (int)((T + per - 1) / per);
  if (p.nsplit < 1) p.nsplit = 1;
  p.rows = (hq / hkv) * B;
  // more than one wave of CTAs: order the sequences by length (see decode_order_kernel)
  p.ordered = pairs * p.nsplit > sms && batch > 1 && batch <= kMaxOrderBatch;
  p.order_bytes = p.ordered ? ((size_t)batch * sizeof(int32_t) + 255) / 256 * 256 : 0;
  p.ws_bytes = p.order_bytes + (size_t)batch * hkv * p.nsplit * p.rows * (d + 4) * sizeof(float);
  return p;
}

cudaError_t launch_decode_attn(const uint16_t* q, const uint16_t* k_blk,
                               const uint16_t* v_blk, const uint16_t* k_pool,
                               const uint16_t* v_pool, int num_pages,
                               const int32_t* block_table, int max_pages,
                               const int32_t* seq_lens, const DecodePlan& plan, float* o,
                               int batch, int B, int hq, int hkv, int d, float scale,
                               void* workspace, int32_t* status, cudaStream_t stream,
                               const uint16_t* k_stage, const uint16_t* v_stage,
                               const int32_t* stage_fill, int B_cache) {
  int32_t* order = plan.ordered ? static_cast<int32_t*>(workspace) : nullptr;
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.order_bytes);
  if (order) {
    decode_order_kernel<<<1, 1024, 0, stream>>>(seq_lens, batch, order);
    count_launches(1);
  }
  DecodeArgs a{block_table, seq_lens, order, part, o, status, num_pages, max_pages, B, hq,
               hkv, hq / hkv, plan.rows, plan.split_len, plan.nsplit,
               scale * 1.4426950408889634f, stage_fill, stage_fill ? B_cache : 0};
  const cudaError_t e =
      d == 64 ? launch_tc<64>(q, k_blk, v_blk, k_pool, v_pool, k_stage, v_stage, a, batch, stream)
              : launch_tc<128>(q, k_blk, v_blk, k_pool, v_pool, k_stage, v_stage, a, batch,
                               stream);
  count_launches(plan.nsplit > 1 ? 2 : 1);
  return e;
}

}  // namespace mars
