"""Parity of the sustained decode workload with the oracle, step by step (needs a GB300).

The workload is the benchmark's: batch 128, committed prefixes uniform in 2048..8192,
block B = 16, 28 query / 4 KV heads, head_dim 128, LM head 3584 x 152064, 16-token bf16
KV pages, tau cycling 1.0 / 0.95 / 0.9 / 0.8 every 16 steps, the accepted tokens'
K/V committed after each step (papernotes.org notes of "MARS: Enabling Autoregressive
Models Multi-Token Generation", Key design 3 and 4; gist.science explainer, 2.C and 2.D).

Every step runs decode attention, the head with its acceptance at that step's tau, and
the commit on the GPU, through the C ABI, over all 128 sequences. The oracle follows
with teacher forcing: both sides commit the GPU's N, which must equal the oracle's
wherever the comparison rules (parity_util) do not exclude it, so an excluded position
cannot derail the later steps. Checked:
  - every step: tokens, max-probs and N of one sequence in each of the 16 row blocks of
    the 2048-row LM head (which sequence of the block rotates with the step); N of all
    128 sequences obeys the acceptance rule on the GPU's own max-probs (1 <= N <= B,
    the accepted positions reach tau, the next one does not);
  - every step: seq_lens and commit slots of all 128 sequences, bit-exact against the
    oracle's commit over the block table;
  - around every tau change: attention O of 16 sampled sequences (one per row block),
    against the oracle on the cache it grew with its own commits, so that a wrong commit
    shows in a later step's attention;
  - at the end: the GPU's KV pages of the sampled sequences equal the oracle's, bit for
    bit, and no device status bit was raised.
A second run over fewer steps at tau 0 and 0.3 drives multi-token commits (N = B, and
mixed N) into the later steps' attention.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from block_masked_token_gb300 import mars
from block_masked_token_gb300 import workloads as W
from parity_util import assert_attn_close, compare_head

pytestmark = pytest.mark.gpu

DEV = "cuda"
f64 = W.to_f64


def _ws(nbytes):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=DEV)


def _row_block_samples(batch, B, rows_per_block=128, offset=0):
    """One sequence in every 128-row block of the head's rows (sequence s owns rows
    s*B .. s*B + B - 1); `offset` picks which sequence of the block."""
    per = max(rows_per_block // B, 1)
    nblk = -(-batch // per)
    return [min(blk * per + (blk + offset) % per, batch - 1) for blk in range(nblk)]


def _compact(pool_dev, bt_row):
    """The pages of one sequence, in logical order, as a float64 host pool, and the local
    block-table row that maps logical page i to compact page i."""
    pages = [int(p) for p in bt_row if p >= 0]
    idx = torch.tensor(pages, dtype=torch.long, device=pool_dev.device)
    local = np.full(len(bt_row), -1, dtype=np.int64)
    local[:len(pages)] = np.arange(len(pages))
    return f64(pool_dev.index_select(0, idx)), local, pages


def _acceptance_rule_holds(n, p, tau, B):
    """N obeys the left-to-right rule on the given max-probs: 1 <= N <= B; for N >= 2 the
    positions 0..N-1 all reach tau; and when position 0 reaches tau and N < B, position
    N does not (when position 0 is below tau the scan stops there and N = 1)."""
    t = np.float32(tau)
    for s in range(len(n)):
        k = int(n[s])
        if not 1 <= k <= B:
            return False
        if k >= 2 and not (p[s, :k] >= t).all():
            return False
        if k < B and p[s, 0] >= t and p[s, k] >= t:
            return False
    return True


def _run_chain(cfg, attn_steps):
    inp = W.make_decode_inputs(cfg, seed=0, device=DEV)
    b, B = cfg.batch, cfg.B
    kp, vp = inp.k_pool, inp.v_pool
    bt_dev = inp.block_table.to(DEV)
    bt = inp.block_table.numpy()
    sl = inp.prefix_lens.to(DEV)
    hint = int(inp.prefix_lens.max()) + B * cfg.steps
    ws_a = _ws(mars.mars_workspace_bytes(mars.OP_DECODE_ATTN, b, B, cfg.hq, cfg.hkv, cfg.d,
                                         max_len=hint))
    ws_h = _ws(mars.mars_workspace_bytes(mars.OP_HEAD_ACCEPT, b, B, vocab=cfg.vocab))
    o = torch.empty(b, B, cfg.hq, cfg.d, dtype=torch.float32, device=DEV)
    tokens = torch.empty(b, B, dtype=torch.int32, device=DEV)
    maxprob = torch.empty(b, B, dtype=torch.float32, device=DEV)
    n_acc = torch.empty(b, dtype=torch.int32, device=DEV)
    slots = torch.empty(b, B, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    w64 = f64(inp.w)

    # oracle state: lengths of every sequence; the cache of the sampled sequences
    lens = inp.prefix_lens.numpy().astype(np.int64)
    attn_seqs = _row_block_samples(b, B)
    cache = {}
    for s in attn_seqs:
        pk, local, pages = _compact(kp, bt[s])
        pv, _, _ = _compact(vp, bt[s])
        cache[s] = [pk, pv, local, pages]
    # the commit slots of all sequences need only the block table: the oracle's commit on
    # a value-free (one-element) copy of the pool gives them
    z_blk = np.zeros((b, B, 1, 1))
    z_pool = np.zeros((inp.num_pages, 1, cfg.page_size, 1))
    excluded = {"tokens": 0, "seqs": 0, "head_rows": 0}

    for step in range(cfg.steps):
        tau = cfg.tau_at(step)
        q, kb, vb, h = inp.q[step], inp.k_blk[step], inp.v_blk[step], inp.h[step]
        mars.mars_decode_attn(q, kb, vb, kp, vp, bt_dev, sl, hint, o, ws_a, st)
        mars.mars_head_accept(h, inp.w, b, B, tau, tokens, maxprob, n_acc, ws_h, st)
        mars.mars_kv_commit(kb, vb, n_acc, sl, bt_dev, kp, vp, slots, st)
        torch.cuda.synchronize()
        n_gpu = n_acc.cpu().numpy().astype(np.int64)
        p_gpu = maxprob.cpu().numpy()
        assert _acceptance_rule_holds(n_gpu, p_gpu, tau, B), f"step {step}: acceptance rule"

        # LM head, max-prob, argmax and N on one sequence per row block
        hs = _row_block_samples(b, B, offset=step)
        rows = [s * B + k for s in hs for k in range(B)]
        rt, rp, rn, gap = oracle.head_accept(f64(h[rows]), w64, len(hs), B, tau)
        ex = compare_head(tokens.cpu().numpy()[hs], p_gpu[hs], n_gpu[hs], rt, rp, rn, gap, tau)
        excluded["tokens"] += ex["tokens_excluded"]
        excluded["seqs"] += ex["seqs_excluded"]
        excluded["head_rows"] += len(rows)

        # attention of the sampled sequences on the oracle's own cache (before this
        # step's commit)
        if step in attn_steps:
            qs, kbs, vbs = f64(q[attn_seqs]), f64(kb[attn_seqs]), f64(vb[attn_seqs])
            got = o[attn_seqs].cpu().numpy()
            for i, s in enumerate(attn_seqs):
                pk, pv, local, _ = cache[s]
                ref = oracle.decode_attn(qs[i:i + 1], kbs[i:i + 1], vbs[i:i + 1], pk, pv,
                                         local[None], lens[s:s + 1], cfg.page_size)
                assert_attn_close(got[i:i + 1], ref, f"step {step} seq {s} attention")

        # commit: slots and lengths of every sequence, and the sampled sequences' cache
        _, _, rl, rs = oracle.kv_commit(z_blk, z_blk, n_gpu, lens, bt, z_pool, z_pool,
                                        cfg.page_size)
        np.testing.assert_array_equal(sl.cpu().numpy(), rl, err_msg=f"step {step} seq_lens")
        np.testing.assert_array_equal(slots.cpu().numpy(), rs, err_msg=f"step {step} slots")
        kbs, vbs = f64(kb[attn_seqs]), f64(vb[attn_seqs])
        for i, s in enumerate(attn_seqs):
            pk, pv, local, pages = cache[s]
            pk, pv, _, _ = oracle.kv_commit(kbs[i:i + 1], vbs[i:i + 1], n_gpu[s:s + 1],
                                            lens[s:s + 1], local[None], pk, pv, cfg.page_size)
            cache[s] = [pk, pv, local, pages]
        lens = rl

    assert int(st.item()) == 0, f"device status {int(st.item())}"
    for s in attn_seqs:
        pk, pv, _, pages = cache[s]
        idx = torch.tensor(pages, dtype=torch.long, device=DEV)
        np.testing.assert_array_equal(f64(kp.index_select(0, idx)), pk, err_msg=f"K seq {s}")
        np.testing.assert_array_equal(f64(vp.index_select(0, idx)), pv, err_msg=f"V seq {s}")
    print(f"{cfg.name}: {cfg.steps} steps, head rows checked {excluded['head_rows']}, "
          f"tokens excluded {excluded['tokens']}, sequences excluded {excluded['seqs']}, "
          f"tokens committed {int(lens.sum() - inp.prefix_lens.numpy().sum())}")
    return excluded


def test_sustained_decode_every_step_matches_oracle():
    """All 64 steps of the benchmark's workload (each tau of the schedule, every phase
    boundary)."""
    cfg = W.SUSTAINED_DECODE_7B
    attn_steps = {0, 1, 15, 16, 17, 31, 32, 33, 47, 48, 49, 63}
    _run_chain(cfg, attn_steps)


def test_sustained_decode_multi_token_commits_feed_attention():
    """The same loop at tau 0 (every position accepted: N = B = 16) and tau 0.3 (mixed N),
    so that multi-token commits of one step are read by the next step's attention."""
    cfg = dataclasses.replace(W.SUSTAINED_DECODE_7B, name="sustained_decode_7b_tau0_0.3",
                              taus=(0.0, 0.3), tau_period=3, steps=6)
    _run_chain(cfg, set(range(cfg.steps)))
