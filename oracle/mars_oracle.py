"""Plain, slow, fp64 CPU oracle for the MARS block-masked attention and decode epilogue.

TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the benchmark's
CPU-baseline leg may import or run this module. The CUDA library and its Python binding
never import it, and it imports nothing from them: the two share no code.

What it follows. The method is "MARS (Mask AutoRegreSsion)" from the paper
"MARS: Enabling Autoregressive Models Multi-Token Generation" (Jin, Wang, Luo, Sun,
arXiv 2604.07023). Citations name the web page and its section:

  [notes]  the papernotes.org NeurIPS 2026 reading notes of the paper (Chinese). The only
           page that prints formulas. Sections used:
             Key design 1 (关键设计 1): the 2L x 2L dual-stream mask M over z = [x; x~],
               with the block index beta(t) = ceil(t / B);
             Key design 2 (关键设计 2): the loss L_mask + L_AR and the AR-signal fractions;
             Key design 3 (关键设计 3): left-to-right threshold acceptance;
             Key design 4 (关键设计 4): the block-level KV cache.
  [gist]   the gist.science English explainer, "2. Methodology", part C (Inference
           Mechanism) and part D (Block-Level KV Caching).

Readings taken where the pages are silent:
  * indices: M is stated 1-indexed; mask_M keeps that form, arrays are 0-indexed;
  * softmax scale: not stated, 1/sqrt(D);
  * grouped-query attention: not on the pages, query head h uses KV head h // (Hq/Hkv);
  * decode form: B [MASK] queries appended after the committed prefix; query k sees the
    whole prefix and block keys 0..k (causal inside the block);
  * "maximum probability": full-vocabulary softmax at temperature 1, argmax ties go to the
    lowest vocabulary index;
  * acceptance starts at block position 0, ">=" is inclusive, at least one token, at most B;
    tau is a float32 value compared exactly in fp64;
  * commit: each sequence's own N rows are written every step (per-sequence commit);
    kv_commit_batch_sync gives the batch-synchronised alternative, every sequence
    committing the smallest N of the batch; kv_commit_block the block-level cache with a
    B_cache boundary (rows held in a per-sequence block buffer until every sequence has
    filled its block; the block is written at the start of the call after the one that
    filled the last block);
  * per-request threshold: one float32 tau per sequence (head_accept_per_request).

Every function takes float64 numpy arrays (callers pass bf16-rounded values converted to
float64) and returns float64 / int64 numpy arrays. Nothing is blocked, fused or reordered
beyond what the definitions state; matmul (BLAS) is the only library primitive used.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


# ---------------------------------------------------------------------------------------
# Key design 1 [notes]: block index and the dual-stream mask M.
# ---------------------------------------------------------------------------------------

def beta(t, B: int):
    """Block index beta(t) = ceil(t / B) of a 1-indexed stream position t ([notes], Key
    design 1, definition under eq. M). Works on ints and integer numpy arrays."""
    return -((-np.asarray(t)) // B) if isinstance(t, np.ndarray) else -((-t) // B)


def mask_M(L: int, B: int) -> np.ndarray:
    """The 2L x 2L visibility matrix of mask M ([notes], Key design 1, eq. M).

    Entry [i-1, j-1] is True where M_ij = 0 (key j visible to query i), for 1-indexed
    i, j in 1..2L. Rows/cols 1..L are the clean stream x, L+1..2L the masked stream x~:
      case 1: i, j <= L and j <= i                         (clean stream, causal)
      case 2: i, j > L, beta(i-L) = beta(j-L), j <= i      (masked stream, causal in block)
      case 3: i > L, j <= L, beta(j) < beta(i-L)           (masked -> strictly earlier
                                                            clean blocks)
      otherwise M_ij = -inf (not visible).
    The last block is shorter when B does not divide L; beta stays ceil(t/B).
    """
    if L < 1 or B < 1:
        raise ValueError("L and B must be >= 1")
    i = np.arange(1, 2 * L + 1)[:, None]
    j = np.arange(1, 2 * L + 1)[None, :]
    case1 = (i <= L) & (j <= L) & (j <= i)
    bi = beta(np.maximum(i - L, 1), B)   # clamp only keeps beta defined where it is unused
    bj = beta(np.maximum(j - L, 1), B)
    case2 = (i > L) & (j > L) & (bi == bj) & (j <= i)
    case3 = (i > L) & (j <= L) & (beta(j, B) < bi)
    return case1 | case2 | case3


def mask_rows(L: int, B: int, rows) -> np.ndarray:
    """Rows `rows` (0-indexed) of mask_M(L, B), built from the same three cases without
    materialising the whole 2L x 2L matrix (used for sampled rows at large L)."""
    i = (np.asarray(rows, dtype=np.int64) + 1)[:, None]
    j = np.arange(1, 2 * L + 1)[None, :]
    case1 = (i <= L) & (j <= L) & (j <= i)
    bi = beta(np.maximum(i - L, 1), B)
    bj = beta(np.maximum(j - L, 1), B)
    case2 = (i > L) & (j > L) & (bi == bj) & (j <= i)
    case3 = (i > L) & (j <= L) & (beta(j, B) < bi)
    return case1 | case2 | case3


# ---------------------------------------------------------------------------------------
# Key design 2 [notes]: the AR-signal fraction, counted from M.
# ---------------------------------------------------------------------------------------

def ar_signal_fraction(L: int, B: int, combined: bool) -> float:
    """Fraction of predicted positions whose context is the full clean history
    ([notes], Key design 2: r_AR = 1/B with L_mask only, (1 + 1/B)/2 with L_mask + L_AR).

    Counted directly from M: a masked-stream row i = L + t (t = 1..L) has a fully clean
    context when its visible set is exactly the clean keys 1..t-1 plus itself; a clean row
    i has one when its visible set is exactly clean keys 1..i. With L_mask only the L
    masked rows carry loss; with L_mask + L_AR all 2L rows do.
    """
    vis = mask_M(L, B)
    n = 2 * L
    cols = np.arange(1, n + 1)
    clean_ok = 0
    for i in range(1, L + 1):
        want = cols <= i
        clean_ok += int(np.array_equal(vis[i - 1], want))
    masked_ok = 0
    for t in range(1, L + 1):
        i = L + t
        want = (cols <= t - 1) | (cols == i)
        masked_ok += int(np.array_equal(vis[i - 1], want))
    if combined:
        return (clean_ok + masked_ok) / (2 * L)
    return masked_ok / L


# ---------------------------------------------------------------------------------------
# Attention under M (training form): softmax(scale * Q K^T + M) V per (batch, q head).
# ---------------------------------------------------------------------------------------

def _masked_softmax_rows(S: np.ndarray, vis: np.ndarray) -> np.ndarray:
    """Row softmax of S with entries where vis is False set to -inf first."""
    S = np.where(vis, S, NEG_INF)
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    return P / P.sum(axis=1, keepdims=True)


def attn_dual_stream(q, k, v, L: int, B: int, scale: float | None = None, rows=None,
                     heads=None, batches=None):
    """Dual-stream attention output O for z = [x; x~] under mask M.

    q: [b, 2L, Hq, D]; k, v: [b, 2L, Hkv, D] (float64). Returns O [b, 2L, Hq, D] float64,
    or, when `rows` is given, O[:, rows] only ([notes], overall framework: both streams in
    one forward; Key design 1, eq. M). `heads`/`batches` restrict the work to those query
    heads / batch items (others left as NaN) so large shapes can be sampled.
    """
    b, n, Hq, D = q.shape
    Hkv = k.shape[2]
    if n != 2 * L:
        raise ValueError("sequence length of q must be 2L")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rows = np.arange(n) if rows is None else np.asarray(rows)
    vis = mask_rows(L, B, rows)
    out = np.full((b, len(rows), Hq, D), np.nan)
    for bi in (range(b) if batches is None else batches):
        for h in (range(Hq) if heads is None else heads):
            hk = h // g
            S = scale * (q[bi, rows, h, :] @ k[bi, :, hk, :].T)
            P = _masked_softmax_rows(S, vis)
            out[bi, :, h, :] = P @ v[bi, :, hk, :]
    return out


def attn_dual_stream_lse(q, k, L: int, B: int, scale: float | None = None):
    """Per query row, log2 of the softmax denominator of attn_dual_stream: lse[b, h, i] =
    log2 sum over the keys j visible to row i under M of exp(scale * q_i . k_j)
    ([notes] Key design 1, eq. M; the statistic the backward pass of that softmax reuses).
    q: [b, 2L, Hq, D], k: [b, 2L, Hkv, D] (float64). Returns [b, Hq, 2L] float64."""
    b, n, Hq, D = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    vis = mask_rows(L, B, np.arange(n))
    out = np.empty((b, Hq, n))
    for bi in range(b):
        for h in range(Hq):
            S = np.where(vis, scale * (q[bi, :, h, :] @ k[bi, :, h // g, :].T), NEG_INF)
            m = S.max(axis=1)
            out[bi, h] = (m + np.log(np.exp(S - m[:, None]).sum(axis=1))) / math.log(2.0)
    return out


def attn_dual_stream_grad_parts(q, k, v, do, L: int, B: int, scale: float | None = None):
    """The per-(batch, query head) intermediates of the dual-stream attention gradient, in
    the order the chain rule forms them ([notes] Key design 1, eq. M: the softmax runs
    over the keys M leaves visible). For upstream gradient dO [b, 2L, Hq, D], yields
    (bi, h, hk, P, dP, D, dS) with kv head hk = h // (Hq/Hkv):
      P  = masked softmax of S = scale Q K^T (0 where M hides the key),
      dP = dO V^T,
      D  = rowsum(P * dP) (equal to rowsum(dO * O), O = P V),
      dS = P * (dP - D)."""
    b, n, Hq, Dh = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(Dh)
    vis = mask_M(L, B)
    for bi in range(b):
        for h in range(Hq):
            hk = h // g
            Q, K, V, dO = q[bi, :, h, :], k[bi, :, hk, :], v[bi, :, hk, :], do[bi, :, h, :]
            P = _masked_softmax_rows(scale * (Q @ K.T), vis)
            dP = dO @ V.T
            D = (P * dP).sum(axis=1, keepdims=True)
            dS = P * (dP - D)
            yield bi, h, hk, P, dP, D, dS


def attn_dual_stream_grad(q, k, v, do, L: int, B: int, scale: float | None = None):
    """Gradient of the dual-stream attention (attn_dual_stream) for an upstream gradient
    dO [b, 2L, Hq, D]: per (batch, query head h), with kv head h // (Hq/Hkv) and P, dS
    from attn_dual_stream_grad_parts: dQ = scale dS K, and summed over the query heads of
    a kv head dK = scale dS^T Q, dV = P^T dO. Returns (dq [b, 2L, Hq, D],
    dk [b, 2L, Hkv, D], dv [b, 2L, Hkv, D])."""
    Dh = q.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(Dh)
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for bi, h, hk, P, _, _, dS in attn_dual_stream_grad_parts(q, k, v, do, L, B, scale):
        dq[bi, :, h, :] = scale * (dS @ k[bi, :, hk, :])
        dk[bi, :, hk, :] += scale * (dS.T @ q[bi, :, h, :])
        dv[bi, :, hk, :] += P.T @ do[bi, :, h, :]
    return dq, dk, dv


# ---------------------------------------------------------------------------------------
# Decode form ([gist] 2.C, 2.D; [notes] Key design 3, Key design 4): B [MASK] queries per
# sequence over the committed prefix in a paged cache, causal inside the block.
# ---------------------------------------------------------------------------------------

def gather_prefix(pool, block_table_row, P: int, page_size: int):
    """Logical rows 0..P-1 of one sequence's cache: pool[page, hkv, slot, :] with
    page = block_table_row[t // page_size], slot = t % page_size. Returns [P, Hkv, D]."""
    Hkv, D = pool.shape[1], pool.shape[3]
    out = np.empty((P, Hkv, D))
    for t in range(P):
        page = int(block_table_row[t // page_size])
        out[t] = pool[page, :, t % page_size, :]
    return out


def decode_attn(q, k_blk, v_blk, k_pool, v_pool, block_table, seq_lens, page_size: int,
                scale: float | None = None, seqs=None):
    """Attention output of the B appended [MASK] queries of each sequence.

    q: [b, B, Hq, D]; k_blk, v_blk: [b, B, Hkv, D]; k_pool, v_pool: [pages, Hkv, page_size,
    D]; block_table: [b, max_pages] int; seq_lens: [b] committed prefix lengths P_s.
    Keys of sequence s: the P_s prefix rows, then the B block rows; query k sees every
    prefix row and block rows 0..k. Returns O [b, B, Hq, D] float64 (NaN for sequences
    not in `seqs`).
    """
    b, B, Hq, D = q.shape
    Hkv = k_blk.shape[2]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.full(q.shape, np.nan)
    for s in (range(b) if seqs is None else seqs):
        P = int(seq_lens[s])
        K = np.concatenate([gather_prefix(k_pool, block_table[s], P, page_size), k_blk[s]])
        V = np.concatenate([gather_prefix(v_pool, block_table[s], P, page_size), v_blk[s]])
        j = np.arange(P + B)[None, :]
        kq = np.arange(B)[:, None]
        vis = (j < P) | ((j - P) <= kq)
        for h in range(Hq):
            hk = h // g
            S = scale * (q[s, :, h, :] @ K[:, hk, :].T)
            out[s, :, h, :] = _masked_softmax_rows(S, vis) @ V[:, hk, :]
    return out


# ---------------------------------------------------------------------------------------
# Step epilogue: LM-head logits, max-prob and argmax, threshold acceptance
# ([notes] Key design 3; [gist] 2.C "Confidence Thresholding").
# ---------------------------------------------------------------------------------------

def head_logits(h, w_vocab_major, chunk: int = 16384):
    """logits[r, v] = sum_d h[r, d] * W[v, d] for h [R, H] and W stored [V, H]; computed
    in vocabulary chunks to bound memory."""
    R = h.shape[0]
    V = w_vocab_major.shape[0]
    out = np.empty((R, V))
    for c0 in range(0, V, chunk):
        out[:, c0:c0 + chunk] = h @ w_vocab_major[c0:c0 + chunk].T
    return out


def maxprob_argmax(logits):
    """Per row: token = lowest index attaining the max logit; maxprob = max_v softmax(l)_v
    = 1 / sum_v exp(l_v - max); gap = max minus the second-largest logit (0 on ties;
    infinite for a one-word vocabulary, which has no second logit).
    Returns (tokens int64 [R], maxprob float64 [R], gap float64 [R])."""
    m = logits.max(axis=1)
    tokens = np.argmax(logits, axis=1)          # first occurrence = lowest index
    maxprob = 1.0 / np.exp(logits - m[:, None]).sum(axis=1)
    if logits.shape[1] < 2:
        return tokens.astype(np.int64), maxprob, np.full(len(m), np.inf)
    part = np.partition(logits, -2, axis=1)
    gap = part[:, -1] - part[:, -2]
    return tokens.astype(np.int64), maxprob, gap


def accept_count(maxprob_row, tau) -> int:
    """Left-to-right acceptance for one sequence ([notes] Key design 3): walk positions
    0, 1, ... accepting while maxprob >= tau, stop at the first position below tau; at
    least one token is always accepted and at most B (the row length). tau is taken as
    the float32 value the caller passes, compared in float64."""
    t = float(np.float32(tau))
    n = 0
    for p in maxprob_row:
        if p >= t:
            n += 1
        else:
            break
    return max(1, n)


def head_accept(h, w_vocab_major, batch: int, B: int, tau):
    """The whole epilogue for a step: h [batch*B, H] (row s*B + k = sequence s, block
    position k), W [V, H]. Returns (tokens [batch, B], maxprob [batch, B], n_accept
    [batch], gap [batch, B])."""
    tokens, maxprob, gap = maxprob_argmax(head_logits(h, w_vocab_major))
    tokens = tokens.reshape(batch, B)
    maxprob = maxprob.reshape(batch, B)
    gap = gap.reshape(batch, B)
    n = np.array([accept_count(maxprob[s], tau) for s in range(batch)], dtype=np.int64)
    return tokens, maxprob, n, gap


def head_accept_per_request(h, w_vocab_major, batch: int, B: int, taus):
    """head_accept with a threshold per request: sequence s uses taus[s] ([gist] 2.C
    "Adaptive Throughput": the speed is adjusted per request in real time; [notes]
    highlights, third point: the confidence threshold of each request is tuned online).
    Each taus[s] is taken as a float32 value, as in accept_count."""
    tokens, maxprob, gap = maxprob_argmax(head_logits(h, w_vocab_major))
    tokens = tokens.reshape(batch, B)
    maxprob = maxprob.reshape(batch, B)
    gap = gap.reshape(batch, B)
    n = np.array([accept_count(maxprob[s], taus[s]) for s in range(batch)], dtype=np.int64)
    return tokens, maxprob, n, gap


# ---------------------------------------------------------------------------------------
# Commit into the block-level KV cache ([notes] Key design 4; [gist] 2.D), per sequence.
# ---------------------------------------------------------------------------------------

def kv_commit(k_blk, v_blk, n_accept, seq_lens, block_table, k_pool, v_pool,
              page_size: int):
    """Copy the first N_s block rows of sequence s into the paged cache and advance its
    length: for i < N_s, pos = seq_len_s + i, page = block_table[s, pos // page_size],
    slot = pos % page_size, pool[page, :, slot, :] = blk[s, i, :, :]. Returns (new k_pool,
    new v_pool, new seq_lens, commit_slots [b, B]) with commit_slots = page * page_size +
    slot for committed rows and -1 otherwise. Inputs are not modified."""
    k_pool = k_pool.copy()
    v_pool = v_pool.copy()
    b, B = k_blk.shape[0], k_blk.shape[1]
    slots = np.full((b, B), -1, dtype=np.int64)
    new_lens = np.array(seq_lens, dtype=np.int64).copy()
    for s in range(b):
        for i in range(int(n_accept[s])):
            pos = int(seq_lens[s]) + i
            page = int(block_table[s][pos // page_size])
            slot = pos % page_size
            k_pool[page, :, slot, :] = k_blk[s, i]
            v_pool[page, :, slot, :] = v_blk[s, i]
            slots[s, i] = page * page_size + slot
        new_lens[s] = int(seq_lens[s]) + int(n_accept[s])
    return k_pool, v_pool, new_lens, slots


def kv_commit_batch_sync(k_blk, v_blk, n_accept, seq_lens, block_table, k_pool, v_pool,
                         page_size: int):
    """Batch-synchronised commit ([notes] Key design 4, second paragraph: the batch
    advances by the smallest number of tokens any of its samples accepted in the step,
    the faster samples waiting; [gist] 2.D: the cache moves only with what every sample
    of the batch accepted). Every sequence commits N_min = min_s N_s rows, N_s clamped to
    [0, B] first; otherwise exactly kv_commit."""
    B = k_blk.shape[1]
    n = [min(max(int(x), 0), B) for x in n_accept]
    n_min = min(n) if n else 0
    return kv_commit(k_blk, v_blk, [n_min] * len(n), seq_lens, block_table, k_pool, v_pool,
                     page_size)


def kv_commit_block(k_blk, v_blk, n_accept, seq_lens, fill, k_stage, v_stage,
                    flush_pending: bool, block_table, k_pool, v_pool, page_size: int,
                    B_cache: int):
    """Block-level commit with a batch-wide B_cache boundary ([notes] Key design 4: the
    prefix cache is frozen in blocks of B_cache tokens; within a batch the samples that
    accept faster wait at the block boundary until every sample has filled the block,
    and then the whole block is written to the persistent prefix cache; [gist] 2.D: the
    cache is updated only when a full block has been accepted across all samples).

    State: seq_lens[s] = tokens of sequence s in the persistent cache (the paged pool);
    fill[s] = accepted tokens of s held in its block buffer stage[s, :fill[s]] (k_stage,
    v_stage [b, B_cache, Hkv, D]); flush_pending = every block was full after the
    previous call. One call, in this order:
      1. if flush_pending, every sequence writes its block, stage[s, 0:B_cache], to the
         pool at positions seq_lens[s] .. seq_lens[s] + B_cache - 1 (page =
         block_table[s, pos // page_size], slot = pos % page_size), then
         seq_lens[s] += B_cache and fill[s] = 0;
      2. every sequence appends n_s = min(clamp(N_s, 0, B), B_cache - fill[s]) accepted
         rows (block rows 0..n_s-1) to its block buffer: a sequence whose block is full
         waits (n_s = 0); commit_slots[s, i] = page * page_size + slot of position
         seq_lens[s] + fill[s] + i, where row i goes when its block is written, for
         i < n_s, and -1 otherwise; fill[s] += n_s;
      3. flush_pending = every fill[s] == B_cache.
    Pages are assumed mapped. Returns (k_pool, v_pool, seq_lens, fill, k_stage, v_stage,
    flush_pending, commit_slots); inputs are not modified."""
    k_pool, v_pool = k_pool.copy(), v_pool.copy()
    k_stage, v_stage = k_stage.copy(), v_stage.copy()
    lens = np.array(seq_lens, dtype=np.int64).copy()
    fill = np.array(fill, dtype=np.int64).copy()
    b, B = k_blk.shape[0], k_blk.shape[1]
    if flush_pending:
        for s in range(b):
            for i in range(B_cache):
                pos = int(lens[s]) + i
                page = int(block_table[s][pos // page_size])
                k_pool[page, :, pos % page_size, :] = k_stage[s, i]
                v_pool[page, :, pos % page_size, :] = v_stage[s, i]
            lens[s] += B_cache
            fill[s] = 0
    slots = np.full((b, B), -1, dtype=np.int64)
    for s in range(b):
        n = min(min(max(int(n_accept[s]), 0), B), B_cache - int(fill[s]))
        for i in range(n):
            pos = int(lens[s]) + int(fill[s]) + i
            page = int(block_table[s][pos // page_size])
            slots[s, i] = page * page_size + pos % page_size
            k_stage[s, int(fill[s]) + i] = k_blk[s, i]
            v_stage[s, int(fill[s]) + i] = v_blk[s, i]
        fill[s] += n
    flush = bool((fill == B_cache).all())
    return k_pool, v_pool, lens, fill, k_stage, v_stage, flush, slots


def decode_attn_staged(q, k_blk, v_blk, k_pool, v_pool, block_table, seq_lens, k_stage,
                       v_stage, fill, page_size: int, scale: float | None = None, seqs=None):
    """Decode-form attention over the block-level cache of kv_commit_block: the keys of
    sequence s are its P_s persistent prefix rows (paged pool), then the fill_s accepted
    rows of its block buffer (stage[s, :fill_s]), then the B block rows of this step;
    block query k sees the prefix, the buffered rows and block rows 0..k ([notes] Key
    design 3 and 4; [gist] 2.C, 2.D). Returns O [b, B, Hq, D] float64 (NaN for
    sequences not in `seqs`)."""
    b, B, Hq, D = q.shape
    Hkv = k_blk.shape[2]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.full(q.shape, np.nan)
    for s in (range(b) if seqs is None else seqs):
        P, F = int(seq_lens[s]), int(fill[s])
        K = np.concatenate([gather_prefix(k_pool, block_table[s], P, page_size),
                            k_stage[s, :F], k_blk[s]])
        V = np.concatenate([gather_prefix(v_pool, block_table[s], P, page_size),
                            v_stage[s, :F], v_blk[s]])
        j = np.arange(P + F + B)[None, :]
        kq = np.arange(B)[:, None]
        vis = (j < P + F) | ((j - P - F) <= kq)
        for h in range(Hq):
            hk = h // g
            S = scale * (q[s, :, h, :] @ K[:, hk, :].T)
            out[s, :, h, :] = _masked_softmax_rows(S, vis) @ V[:, hk, :]
    return out


# ---------------------------------------------------------------------------------------
# Training loss of the dual stream ([notes] Key design 2; [gist] 2.B "Combined Loss").
# ---------------------------------------------------------------------------------------

def ce_loss_dual(h, w_vocab_major, targets, batch: int, L: int):
    """L = L_mask + L_AR for hidden states h [batch*2L, H] (row s*2L + t; t < L the clean
    stream, t >= L the masked stream) and the head W [V, H]. For a row with target y:
    ce = log sum_v exp(l_v) - l_y, l = h W^T. L_AR is the mean ce over the clean rows with
    a target, L_mask over the masked rows with one; target -1 leaves a row out; a stream
    without targets gives 0. Returns (L_mask, L_AR, ce [batch*2L], 0 where no target)."""
    logits = head_logits(h, w_vocab_major)
    m = logits.max(axis=1)
    lse = m + np.log(np.exp(logits - m[:, None]).sum(axis=1))
    y = np.asarray(targets, dtype=np.int64)
    V = logits.shape[1]
    valid = (y >= 0) & (y < V)
    ce = np.zeros(len(y), dtype=np.float64)
    rows = np.flatnonzero(valid)
    ce[rows] = lse[rows] - logits[rows, y[rows]]
    pos = np.arange(len(y)) % (2 * L)
    clean = valid & (pos < L)
    masked = valid & (pos >= L)
    l_ar = ce[clean].mean() if clean.any() else 0.0
    l_mask = ce[masked].mean() if masked.any() else 0.0
    return float(l_mask), float(l_ar), ce


def ce_loss_dual_grad(h, w_vocab_major, targets, batch: int, L: int):
    """Gradient of L = L_mask + L_AR (ce_loss_dual) with respect to the logits, h and W:
    dL/dl_rv = (softmax(l_r)_v - [v = y_r]) / N_x for a row of stream x with a target
    (N_x = that stream's rows with a target), 0 for rows without one; dh = dlogits W and
    dW = dlogits^T h. Returns (dh [R, H], dW [V, H], dlogits [R, V])."""
    logits = head_logits(h, w_vocab_major)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p /= p.sum(axis=1, keepdims=True)
    y = np.asarray(targets, dtype=np.int64)
    V = logits.shape[1]
    valid = (y >= 0) & (y < V)
    pos = np.arange(len(y)) % (2 * L)
    n_clean = int((valid & (pos < L)).sum())
    n_masked = int((valid & (pos >= L)).sum())
    scale = np.where(pos < L, 1.0 / max(n_clean, 1), 1.0 / max(n_masked, 1))
    scale = np.where(valid, scale, 0.0)
    g = p.copy()
    rows = np.flatnonzero(valid)
    g[rows, y[rows]] -= 1.0
    g *= scale[:, None]
    return g @ w_vocab_major, g.T @ h, g
