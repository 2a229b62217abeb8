/*
 * mars.h — C ABI of libmars: the GB300 (sm_103a) hot path of MARS block-masked
 * multi-token decoding ("MARS: Enabling Autoregressive Models Multi-Token Generation",
 * Jin, Wang, Luo, Sun, arXiv 2604.07023).
 *
 * Sources cited below: [notes] = the papernotes.org NeurIPS 2026 reading notes of the
 * paper (the page that prints the formulas), sections "Key design 1..4" (关键设计 1..4);
 * [gist] = the gist.science explainer, "2. Methodology", parts C and D.
 *
 * Conventions shared by every entry point
 *   - Tensor arguments are DEVICE pointers to caller-owned memory (for example PyTorch
 *     tensors). Scalars are passed by value. The library never allocates, frees or
 *     keeps a pointer after the call returns.
 *   - bf16 tensors are raw bfloat16 bits (mars_bf16). All tensors are row-major and
 *     contiguous in the layout stated per argument; base pointers must be 16-byte
 *     aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is enqueued
 *     on it and the call returns without synchronising the host.
 *   - Return value: MARS_OK, or a negative MARS_E* code for an error found on the host
 *     before anything was launched (nothing was enqueued then), or MARS_ECUDA if a launch
 *     failed. mars_strerror() names each code.
 *   - Errors only the device can see (a block-table entry outside the pool, a position
 *     past the mapped pages) OR a MARS_ST_* bit into *status (a device int32 the caller
 *     zeroes) and skip the offending write; nothing traps. status may be NULL where
 *     stated.
 *   - Head dimension d is 64 or 128; hq % hkv == 0 (query head h uses KV head
 *     h / (hq / hkv), consecutive query heads share a KV head); 1 <= B <= 32.
 */
#ifndef MARS_H
#define MARS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mars_bf16;

#define MARS_OK 0
#define MARS_EINVAL (-1)        /* bad argument: null pointer, size out of range, NaN tau */
#define MARS_EALIGN (-2)        /* a tensor base pointer is not 16-byte aligned */
#define MARS_EUNSUPPORTED (-3)  /* valid but not built: d not in {64,128}, page_size != 16 */
#define MARS_ECUDA (-4)         /* a CUDA launch or driver call failed */
#define MARS_ENOSPACE (-5)      /* workspace smaller than mars_workspace_bytes() */

#define MARS_ST_NOPAGE 1        /* block-table entry < 0 or >= num_pages: write skipped */
#define MARS_ST_OVERFLOW 2      /* position beyond max_pages_per_seq: write skipped */
#define MARS_ST_TIMEOUT 4       /* an in-kernel pipeline wait passed its time limit (2 s);
                                   the kernel stopped early and its outputs are invalid */
#define MARS_ST_BADTARGET 8     /* a loss target outside [-1, vocab): that row is left out */

#define MARS_OP_DECODE_ATTN 1
#define MARS_OP_HEAD_ACCEPT 2
#define MARS_OP_CE_LOSS 3
#define MARS_OP_CE_LOSS_GRAD 4
#define MARS_OP_DUAL_GRAD 5

/* Workspace (device scratch, caller-allocated, >= 256-byte aligned) needed by `op`.
 * MARS_OP_DECODE_ATTN uses batch, B, hq, hkv, d, max_len (the max_len_hint of the call);
 * MARS_OP_HEAD_ACCEPT uses batch, B, vocab; MARS_OP_CE_LOSS and MARS_OP_CE_LOSS_GRAD use
 * batch, vocab and max_len as the stream length L (pass B = 1 for these two);
 * MARS_OP_DUAL_GRAD uses batch, B (the block size of mask M, any value >= 1), hq, hkv, d
 * and max_len as L. Other arguments are ignored.
 * Returns 0 for an unknown op or invalid sizes. */
size_t mars_workspace_bytes(int op, int batch, int B, int hq, int hkv, int d, int hidden,
                            int vocab, int max_len);

/* Dual-stream (training-form) attention under mask M ([notes] Key design 1, eq. M, with
 * beta(t) = ceil(t/B); overall framework: one forward over z = [x; x~]).
 *   q  [batch, 2L, hq,  d] bf16   rows 0..L-1 clean stream x, rows L..2L-1 masked x~
 *   k  [batch, 2L, hkv, d] bf16
 *   v  [batch, 2L, hkv, d] bf16
 *   o  [batch, 2L, hq,  d] float  (written)
 * Row i attends to key j (0-indexed) iff: i,j < L and j <= i; or i,j >= L,
 * (i-L)/B == (j-L)/B and j <= i; or i >= L, j < L and j/B < (i-L)/B. Softmax of
 * scale * q.k over the visible keys, scale <= 0 meaning 1/sqrt(d). Fully masked key tiles
 * are never loaded. L >= 1; B > L is allowed (one block). status may be NULL
 * (MARS_ST_TIMEOUT only). */
int mars_attn_dual_stream(const mars_bf16* q, const mars_bf16* k, const mars_bf16* v,
                          float* o, int batch, int L, int B, int hq, int hkv, int d,
                          float scale, int32_t* status, void* stream);

/* mars_attn_dual_stream that also writes each query row's softmax log-sum-exp, the
 * statistic its gradient needs (the training step's forward keeps it for the backward):
 *   lse [batch, hq, 2, Lp] float (written), Lp = L rounded up to a multiple of 128;
 *       lse[b][h][s][t] = log2 of sum over the keys visible to row s*L + t of
 *       exp2(scale * log2(e) * q.k), for t < L; rows L <= t < Lp are written as 0.
 * lse is 16-byte aligned. Other arguments, layouts and errors as mars_attn_dual_stream;
 * o is written identically. */
int mars_attn_dual_stream_lse(const mars_bf16* q, const mars_bf16* k, const mars_bf16* v,
                              float* o, float* lse, int batch, int L, int B, int hq, int hkv,
                              int d, float scale, int32_t* status, void* stream);

/* Decode-form attention ([gist] 2.C sliding window; [notes] Key design 3 and 4): each
 * sequence s appends B [MASK] queries after its committed prefix of P_s = seq_lens[s]
 * tokens held in a paged cache; block query k sees all P_s prefix keys and block keys
 * 0..k.
 *   q           [batch, B, hq,  d] bf16
 *   k_blk,v_blk [batch, B, hkv, d] bf16   K/V of the B block positions
 *   k_pool,v_pool [num_pages, hkv, page_size, d] bf16   the paged prefix cache
 *   block_table [batch, max_pages_per_seq] int32        page of logical page p
 *   seq_lens    [batch] int32 (device)                  P_s
 *   max_len_hint  host upper bound on every P_s; it sizes the split-KV grid without a
 *                 host sync. A larger P_s is still computed correctly (the last split
 *                 runs to the end), only slower.
 *   o           [batch, B, hq, d] float (written)
 *   workspace   >= mars_workspace_bytes(MARS_OP_DECODE_ATTN, ...) bytes
 *   status      may be NULL; MARS_ST_NOPAGE / MARS_ST_OVERFLOW when a needed page is
 *               unmapped (those keys are then skipped).
 * page_size must be 16. */
int mars_decode_attn(const mars_bf16* q, const mars_bf16* k_blk, const mars_bf16* v_blk,
                     const mars_bf16* k_pool, const mars_bf16* v_pool, int num_pages,
                     const int32_t* block_table, int max_pages_per_seq,
                     const int32_t* seq_lens, int max_len_hint, float* o, int batch, int B,
                     int hq, int hkv, int d, int page_size, float scale, void* workspace,
                     size_t ws_bytes, int32_t* status, void* stream);

/* Step epilogue ([notes] Key design 3; [gist] 2.C "Confidence Thresholding"): LM-head
 * logits l = h W^T for the B positions of each sequence, then per position the argmax
 * token (lowest index on ties) and max-prob p = max_v softmax(l)_v = 1 / sum_v
 * exp(l_v - max l), then N_s = the number of leading positions with p >= tau, at least 1
 * and at most B. The logits never reach global memory.
 *   h         [batch*B, hidden] bf16   row s*B + k = sequence s, block position k
 *   w         [vocab, hidden] bf16     the LM head, vocabulary-major (row v = word v)
 *   tau       the confidence threshold, per call (the live speed knob); finite
 *   tokens    [batch, B] int32, maxprob [batch, B] float, n_accept [batch] int32 (written)
 *   workspace >= mars_workspace_bytes(MARS_OP_HEAD_ACCEPT, ...) bytes; needs no
 *             initialisation (the call clears the counters it uses on the stream)
 * One GEMM kernel does it all: the CTA that completes a block of 128 rows merges its
 * partial maxima and sums, writes the tokens and max-probs, and runs the scan.
 * hidden % 8 == 0 (row pitch of h and w a multiple of 16 bytes). status may be NULL. */
int mars_head_accept(const mars_bf16* h, const mars_bf16* w, int batch, int B, int hidden,
                     int vocab, float tau, int32_t* tokens, float* maxprob,
                     int32_t* n_accept, void* workspace, size_t ws_bytes, int32_t* status,
                     void* stream);

/* mars_head_accept with one threshold per request ([gist] 2.C "Adaptive Throughput": the
 * speed is adjusted per request in real time; [notes] highlights, third point: each
 * request's confidence threshold is tuned online). Sequence s accepts its leading run of
 * positions with p >= taus[s] (at least 1, at most B); everything else is mars_head_accept.
 *   taus      [batch] float, device memory, read when the kernels run; a NaN entry
 *             compares false, so that sequence accepts exactly one token
 * Returns MARS_EINVAL when taus is NULL (batch > 0). */
int mars_head_accept_per_request(const mars_bf16* h, const mars_bf16* w, int batch, int B,
                                 int hidden, int vocab, const float* taus, int32_t* tokens,
                                 float* maxprob, int32_t* n_accept, void* workspace,
                                 size_t ws_bytes, int32_t* status, void* stream);

/* Scratch reserved by mars_head_accept_noalloc on every GPU that loads the library. */
#define MARS_NOALLOC_SCRATCH_BYTES (8u << 20)

/* mars_head_accept without a workspace argument. The paper has no counterpart: this is
 * a deployment variant for callers that cannot allocate device memory when they run a
 * decode step (memory reserved up front with no allocation allowed afterwards, a host
 * framework that owns every device allocation, a real-time path where an allocation and
 * its possible synchronisation are not allowed). Inputs, outputs and results are those
 * of mars_head_accept; it allocates nothing (no cudaMalloc, cudaFree or allocating
 * library call).
 * Scratch: one library-owned device array of MARS_NOALLOC_SCRATCH_BYTES per GPU, held
 * from library load until the process exits. A call needing more than that (the
 * workspace mars_head_accept would need, mars_workspace_bytes(MARS_OP_HEAD_ACCEPT, ...):
 * on a 152-SM GB300 at vocab 152064, more than 26 blocks of 128 rows, i.e. 3328 rows)
 * returns MARS_ENOSPACE before anything is launched.
 * The first call on a device (made while that device is current) looks up the array's
 * device address; make that first call before any CUDA stream capture. The address is
 * looked up again when the calling thread's current context differs from the one of the
 * lookup (for example after cudaDeviceReset); such a first call in a new context must
 * likewise come before any capture.
 * Every call uses the same array and leaves its contents behind; the counters that must
 * start at zero are cleared on the stream at the start of every call. Calls whose kernels
 * may overlap on the GPU (different streams without ordering between them) race on the
 * array and give wrong results, so order such calls on one stream. */
int mars_head_accept_noalloc(const mars_bf16* h, const mars_bf16* w, int batch, int B,
                             int hidden, int vocab, float tau, int32_t* tokens,
                             float* maxprob, int32_t* n_accept, int32_t* status,
                             void* stream);

/* Commit of the accepted tokens' K/V into the block-level cache ([notes] Key design 4;
 * [gist] 2.D), per sequence every step: for i < N_s = n_accept[s] (clamped to [0, B]),
 * pos = seq_lens[s] + i, page = block_table[s][pos / page_size], slot = pos % page_size;
 * k_pool[page, :, slot, :] = k_blk[s, i] and the same for v; commit_slots[s][i] =
 * page * page_size + slot, -1 for i >= N_s; then seq_lens[s] += (rows committed).
 * A row whose page is unmapped (entry < 0 or >= num_pages, or past max_pages_per_seq)
 * is not written, flags MARS_ST_NOPAGE / MARS_ST_OVERFLOW, gets slot -1, and ends the
 * commit of that sequence (seq_lens advances by the rows before it).
 *   k_blk,v_blk [batch, B, hkv, d] bf16; n_accept [batch] int32; seq_lens [batch] int32
 *   (in/out); block_table [batch, max_pages_per_seq] int32; k_pool, v_pool [num_pages,
 *   hkv, page_size, d] bf16 (updated in place); commit_slots [batch, B] int32 (written,
 *   may be NULL). page_size must be 16. status may be NULL. */
int mars_kv_commit(const mars_bf16* k_blk, const mars_bf16* v_blk, const int32_t* n_accept,
                   int32_t* seq_lens, const int32_t* block_table, int max_pages_per_seq,
                   mars_bf16* k_pool, mars_bf16* v_pool, int num_pages,
                   int32_t* commit_slots, int batch, int B, int hkv, int d, int page_size,
                   int32_t* status, void* stream);

/* Batch-synchronised commit ([notes] Key design 4, second paragraph: the batch state
 * advances by the smallest number of tokens any sample accepted in the step, faster
 * samples waiting for the others; [gist] 2.D: the cache moves only with what the whole
 * batch accepted). Exactly mars_kv_commit with every N_s replaced by
 * N_min = min over the batch of clamp(n_accept[s], 0, B); seq_lens advance by N_min (less
 * for a sequence stopped by an unmapped page). Same arguments, layouts and errors. */
int mars_kv_commit_batch_sync(const mars_bf16* k_blk, const mars_bf16* v_blk,
                              const int32_t* n_accept, int32_t* seq_lens,
                              const int32_t* block_table, int max_pages_per_seq,
                              mars_bf16* k_pool, mars_bf16* v_pool, int num_pages,
                              int32_t* commit_slots, int batch, int B, int hkv, int d,
                              int page_size, int32_t* status, void* stream);

/* Words of the device state that mars_kv_commit_block keeps between calls. */
#define MARS_BLOCK_SYNC_WORDS 4

/* Block-level commit with a batch-wide B_cache boundary ([notes] Key design 4: the prefix
 * cache is frozen in blocks of B_cache tokens; within a batch, a sample that has filled
 * its block waits at the boundary until every sample has filled it, and then the whole
 * block is written to the persistent prefix cache; [gist] 2.D: the cache is updated only
 * when a full block of tokens has been accepted across all samples of the batch).
 * State, all device memory owned by the caller and zeroed by it before the first call:
 *   seq_lens    [batch] int32   tokens of each sequence in the persistent cache (the pool)
 *   block_fill  [batch] int32   accepted tokens held in the sequence's block buffer
 *   k_stage, v_stage [batch, B_cache, hkv, d] bf16   the block buffers (row i = the i-th
 *               accepted token of the current block); contents need no initialisation
 *   sync_state  [MARS_BLOCK_SYNC_WORDS] int32        batch-wide flags (zeroed once)
 * One call, for every sequence s:
 *   1. if every block was full after the previous call, block rows 0..B_cache-1 are
 *      written to the pool at positions seq_lens[s] .. seq_lens[s] + B_cache - 1 (page =
 *      block_table[s][pos / page_size], slot = pos % page_size), seq_lens[s] += B_cache
 *      and block_fill[s] = 0. (Whether every block is full is known only after every
 *      sequence of a call has taken its rows; the kernel records it without any wait
 *      and the next call writes the blocks. The decode attention of the step in between
 *      reads the full blocks from the buffers, i.e. the same keys.)
 *   2. it takes n = min(clamp(n_accept[s], 0, B), B_cache - block_fill[s]) accepted rows
 *      (block rows 0..n-1 of k_blk / v_blk, [batch, B, hkv, d]) into buffer rows
 *      block_fill[s] .. block_fill[s] + n - 1: a sequence whose block is full takes none
 *      and waits. commit_slots[s][i] (may be NULL) = page * page_size + slot of position
 *      seq_lens[s] + block_fill[s] + i, where row i will be written with its block, for
 *      i < n, and -1 otherwise; block_fill[s] += n.
 * A page that is unmapped (entry < 0 or >= num_pages, or past max_pages_per_seq) flags
 * MARS_ST_NOPAGE / MARS_ST_OVERFLOW: a block's write stops before a row on such a page
 * (seq_lens advances by the rows written, the rest of the block is dropped), and an
 * accepted row whose position falls on one is not taken, nor are the rows after it.
 * 8 <= B_cache <= 64, B_cache % 8 == 0; page_size must be 16. Calls must be ordered on one
 * stream (each reads the state the previous one wrote). The decode attention over this
 * cache is mars_decode_attn_block_cache. */
int mars_kv_commit_block(const mars_bf16* k_blk, const mars_bf16* v_blk,
                         const int32_t* n_accept, int32_t* seq_lens, int32_t* block_fill,
                         mars_bf16* k_stage, mars_bf16* v_stage, int B_cache,
                         int32_t* sync_state, const int32_t* block_table,
                         int max_pages_per_seq, mars_bf16* k_pool, mars_bf16* v_pool,
                         int num_pages, int32_t* commit_slots, int batch, int B, int hkv,
                         int d, int page_size, int32_t* status, void* stream);

/* mars_decode_attn over the block-level cache of mars_kv_commit_block ([notes] Key design
 * 3 and 4; [gist] 2.C, 2.D): the keys of sequence s are its seq_lens[s] prefix tokens in
 * the paged pool, then the block_fill[s] accepted tokens of its block buffer (k_stage /
 * v_stage rows 0..block_fill[s]-1), then the B block keys of this step; block query k
 * sees the prefix, the buffered tokens and block keys 0..k. Arguments, layouts, workspace
 * and errors as mars_decode_attn; 8 <= B_cache <= 64, B_cache % 8 == 0. */
int mars_decode_attn_block_cache(const mars_bf16* q, const mars_bf16* k_blk,
                                 const mars_bf16* v_blk, const mars_bf16* k_pool,
                                 const mars_bf16* v_pool, int num_pages,
                                 const int32_t* block_table, int max_pages_per_seq,
                                 const int32_t* seq_lens, int max_len_hint,
                                 const mars_bf16* k_stage, const mars_bf16* v_stage,
                                 const int32_t* block_fill, int B_cache, float* o, int batch,
                                 int B, int hq, int hkv, int d, int page_size, float scale,
                                 void* workspace, size_t ws_bytes, int32_t* status,
                                 void* stream);

/* Gradient of mars_attn_dual_stream (the training step's backward of the attention under
 * M, [notes] Key design 1 and overall framework): for upstream gradient dO, per (batch,
 * query head) with P = softmax(scale Q K^T + M): dQ = scale dS K, and per kv head
 * dK = scale sum dS^T Q, dV = sum P^T dO over its query heads, where dS = P * (dP - D),
 * dP = dO V^T, D_i = sum_c dO_ic O_ic.
 *   q [b, 2L, hq, d], k, v [b, 2L, hkv, d] bf16   the forward's inputs
 *   o, d_o [b, 2L, hq, d] float                   the forward's output and its gradient
 *   dq [b, 2L, hq, d], dk, dv [b, 2L, hkv, d] float (written)
 *   workspace >= mars_workspace_bytes(MARS_OP_DUAL_GRAD, b, B, hq, hkv, d, 0, 0, L) bytes:
 *             dO in bf16 and, per query row, the softmax log-sum-exp and D (fp32)
 * The call recomputes the row statistics with the forward kernel, then runs a tcgen05
 * kernel per (batch, query head, key tile) for dK and dV and a row-parallel one for dQ;
 * no score block is stored. P and dS are rounded to bf16 before their products (fp32
 * accumulate). dK and dV are sums over the kv group's query heads in an order that
 * depends on scheduling (fp32 atomics), so they may differ in the last bits from run to
 * run. scale <= 0 means 1/sqrt(d). status: as for mars_attn_dual_stream (a pipeline wait
 * that ran out sets MARS_ST_TIMEOUT); may be NULL. */
int mars_attn_dual_stream_grad(const mars_bf16* q, const mars_bf16* k, const mars_bf16* v,
                               const float* o, const float* d_o, int batch, int L, int B,
                               int hq, int hkv, int d, float scale, float* dq, float* dk,
                               float* dv, void* workspace, size_t ws_bytes, int32_t* status,
                               void* stream);

/* mars_attn_dual_stream_grad from the forward's row statistics: lse as written by
 * mars_attn_dual_stream_lse with the same q, k, v, L, B and scale (read only), which
 * saves the forward pass the plain entry point runs to recompute it. Other arguments,
 * workspace, layouts and errors as mars_attn_dual_stream_grad. */
int mars_attn_dual_stream_grad_lse(const mars_bf16* q, const mars_bf16* k, const mars_bf16* v,
                                   const float* o, const float* d_o, const float* lse,
                                   int batch, int L, int B, int hq, int hkv, int d, float scale,
                                   float* dq, float* dk, float* dv, void* workspace,
                                   size_t ws_bytes, int32_t* status, void* stream);

/* Dual-stream training loss L = L_mask + L_AR ([notes] Key design 2: the masked-stream
 * cross-entropy plus the clean-stream next-token cross-entropy; [gist] 2.B "Combined
 * Loss") for the LM head over the 2L positions of z = [x; x~]. For every row r with a
 * target y_r: ce_r = log sum_v exp(l_rv) - l_{r y_r}, with l = h W^T computed in fp32 from
 * bf16 inputs (the logits are never written). L_AR = mean of ce_r over the clean rows
 * (stream position t < L) with a target, L_mask = mean over the masked rows (t >= L) with
 * a target; a stream without targets gives 0. The caller chooses which rows carry targets
 * (the masked set, the right shift of the next-token targets): -1 leaves a row out.
 *   h         [batch*2L, hidden] bf16   row s*2L + t = sequence s, stream position t
 *   w         [vocab, hidden] bf16      the LM head, vocabulary-major
 *   targets   [batch*2L] int32          target word per row, or -1
 *   loss      [3] float (written)       {L_mask, L_AR, L_mask + L_AR}
 *   row_ce    [batch*2L] float or NULL  ce_r per row (0 for rows without a target)
 *   row_lse   [batch*2L] float or NULL  log sum_v exp(l_rv) per row (every row), the input
 *                                       of mars_dual_stream_ce_loss_grad
 *   workspace >= mars_workspace_bytes(MARS_OP_CE_LOSS, batch, 1, 0, 0, 0, 0, vocab, L)
 * hidden % 8 == 0. A target outside [-1, vocab) leaves its row out and flags
 * MARS_ST_BADTARGET. The sums run in a fixed order (float64), so repeated calls agree
 * bit for bit. status may be NULL. The gradient is mars_dual_stream_ce_loss_grad. */
int mars_dual_stream_ce_loss(const mars_bf16* h, const mars_bf16* w, const int32_t* targets,
                             int batch, int L, int hidden, int vocab, float* loss,
                             float* row_ce, float* row_lse, void* workspace, size_t ws_bytes,
                             int32_t* status, void* stream);

/* Gradient of L = L_mask + L_AR (as defined for mars_dual_stream_ce_loss) with respect to
 * h and W: dL/dl_rv = (softmax(l_r)_v - [v = y_r]) / N_x for a row of stream x with a
 * target (N_x = the rows of that stream with a target) and 0 for the others;
 * dh = dlogits W, dW = dlogits^T h. The logits are recomputed by the LM-head GEMM, whose
 * epilogue writes dlogits in bf16 to the workspace using row_lse from the forward call;
 * the two products run on the library's tcgen05 GEMM, which reads dlogits, W and h in
 * place (bf16 inputs, fp32 accumulate and output).
 *   row_lse   [batch*2L] float          from mars_dual_stream_ce_loss
 *   dh        [batch*2L, hidden] float or NULL (written)
 *   dw        [vocab, hidden] float or NULL    (written)
 *   workspace >= mars_workspace_bytes(MARS_OP_CE_LOSS_GRAD, batch, 1, 0, 0, 0, 0, vocab, L)
 *             (about batch*2L*vocab*2 bytes: the bf16 dlogits)
 * hidden % 8 == 0 and vocab % 8 == 0. */
int mars_dual_stream_ce_loss_grad(const mars_bf16* h, const mars_bf16* w,
                                  const int32_t* targets, const float* row_lse, int batch,
                                  int L, int hidden, int vocab, float* dh, float* dw,
                                  void* workspace, size_t ws_bytes, int32_t* status,
                                  void* stream);

/* Self-check of the in-kernel wait limit every pipeline relies on: enqueues one small
 * kernel that waits on an mbarrier nothing completes. The wait gives up after its time
 * limit (about 2 s) and ORs MARS_ST_TIMEOUT into *status (device int32, zeroed by the
 * caller, required); the kernel then exits normally and the context stays usable.
 * Asynchronous like the other calls. */
int mars_check_wait_timeout(int32_t* status, void* stream);

/* Human-readable name of a return code. Never NULL. */
const char* mars_strerror(int code);

/* Library build string (architecture and kernel variants). Never NULL. */
const char* mars_version(void);

/* Number of kernels libmars has enqueued (all threads, all devices) since it was loaded.
 * Host-side counter, read it to count the launches of a timed region. */
uint64_t mars_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MARS_H */
