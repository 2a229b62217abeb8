"""Parity of the block-level cache with a B_cache boundary (needs a GB300).

mars_kv_commit_block and mars_decode_attn_block_cache against the oracle
(kv_commit_block, decode_attn_staged) over chains of steps, through the C ABI: every step
the attention over prefix + block buffer + block keys, then the commit with the step's
accepted counts (chosen by the test, including out-of-range ones that the rule clamps).
After every commit the whole pool, the buffered rows, the lengths, the fills, the commit
slots and the pending-flush flag are compared bit for bit ([notes] Key design 4;
[gist] 2.D).
"""
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


class BlockCache:
    """Device state of the block-level cache for one batch, and the oracle's copy."""

    def __init__(self, inp, cfg, B_cache, seed):
        b = cfg.batch
        g = torch.Generator().manual_seed(seed)
        shape = (b, B_cache, cfg.hkv, cfg.d)
        stage0 = torch.randn(shape, generator=g).to(torch.bfloat16)   # no initialisation
        self.B_cache = B_cache
        self.kp, self.vp = inp.k_pool.to(DEV), inp.v_pool.to(DEV)
        self.bt = inp.block_table.to(DEV)
        self.sl = inp.prefix_lens.to(DEV)
        self.fill = torch.zeros(b, dtype=torch.int32, device=DEV)
        self.ks, self.vs = stage0.to(DEV), stage0.flip(0).contiguous().to(DEV)
        self.sync = torch.zeros(mars.BLOCK_SYNC_WORDS, dtype=torch.int32, device=DEV)
        self.status = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.r = [f64(inp.k_pool), f64(inp.v_pool), inp.prefix_lens.numpy().astype(np.int64),
                  np.zeros(b, dtype=np.int64), f64(self.ks), f64(self.vs), False]
        self.bt_np = inp.block_table.numpy()

    def attend(self, q, kb, vb, hint, cfg):
        o = torch.empty(q.shape, dtype=torch.float32, device=DEV)
        ws = _ws(mars.mars_workspace_bytes(mars.OP_DECODE_ATTN, cfg.batch, cfg.B, cfg.hq,
                                           cfg.hkv, cfg.d, max_len=hint))
        mars.mars_decode_attn_block_cache(q.to(DEV), kb.to(DEV), vb.to(DEV), self.kp, self.vp,
                                          self.bt, self.sl, hint, self.ks, self.vs, self.fill,
                                          o, ws, self.status)
        torch.cuda.synchronize()
        rk, rv, rl, rf, rks, rvs, _ = self.r
        ref = oracle.decode_attn_staged(f64(q), f64(kb), f64(vb), rk, rv, self.bt_np, rl, rks,
                                        rvs, rf, cfg.page_size)
        return o, ref

    def commit(self, kb, vb, n, cfg):
        slots = torch.full((cfg.batch, cfg.B), -7, dtype=torch.int32, device=DEV)
        nd = torch.as_tensor(np.asarray(n, dtype=np.int32)).to(DEV)
        mars.mars_kv_commit_block(kb.to(DEV), vb.to(DEV), nd, self.sl, self.fill, self.ks,
                                  self.vs, self.sync, self.bt, self.kp, self.vp, slots,
                                  self.status)
        torch.cuda.synchronize()
        rk, rv, rl, rf, rks, rvs, flush = self.r
        out = oracle.kv_commit_block(f64(kb), f64(vb), np.asarray(n), rl, rf, rks, rvs, flush,
                                     self.bt_np, rk, rv, cfg.page_size, self.B_cache)
        self.r = list(out[:7])
        rk, rv, rl, rf, rks, rvs, flush = self.r
        rs = out[7]
        assert int(self.status.item()) == 0
        np.testing.assert_array_equal(slots.cpu().numpy(), rs)
        np.testing.assert_array_equal(self.sl.cpu().numpy(), rl)
        np.testing.assert_array_equal(self.fill.cpu().numpy(), rf)
        assert bool(self.sync[0].item()) == flush
        np.testing.assert_array_equal(f64(self.kp.cpu()), rk)
        np.testing.assert_array_equal(f64(self.vp.cpu()), rv)
        ks, vs = f64(self.ks.cpu()), f64(self.vs.cpu())
        for s in range(cfg.batch):
            np.testing.assert_array_equal(ks[s, :rf[s]], rks[s, :rf[s]])
            np.testing.assert_array_equal(vs[s, :rf[s]], rvs[s, :rf[s]])
        return flush


@pytest.mark.parametrize("batch,B,hq,hkv,d,B_cache,steps", [
    (5, 8, 4, 2, 128, 16, 12),
    (3, 4, 8, 2, 64, 8, 14),
    (4, 16, 7, 1, 128, 32, 8),      # B_cache = 2B; G*B = 112 query rows per kv head
])
def test_block_cache_chain_matches_oracle(batch, B, hq, hkv, d, B_cache, steps):
    cfg = W.DecodeConfig("bc", batch=batch, prefix_lo=0, prefix_hi=300, B=B, hq=hq, hkv=hkv,
                         d=d, hidden=64, vocab=64)
    inp = W.make_decode_inputs(cfg, seed=batch * 10 + B, steps=steps, with_head=False,
                               extra_pages=2)
    bc = BlockCache(inp, cfg, B_cache, seed=5)
    rng = np.random.default_rng(B_cache)
    hint = int(inp.prefix_lens.max()) + B * steps
    flushes = 0
    for step in range(steps):
        o, ref = bc.attend(inp.q[step], inp.k_blk[step], inp.v_blk[step], hint, cfg)
        assert_attn_close(o.cpu().numpy(), ref, f"step {step} attention")
        n = rng.integers(-1, B + 3, batch)
        flushes += bc.commit(inp.k_blk[step], inp.v_blk[step], n, cfg)
    assert flushes >= 1, "the chain never filled every block"


def test_block_cache_decode_step_end_to_end():
    """The tiny decode workload's step with the block-level cache: attention over prefix +
    block buffer, the LM head with acceptance at tau = 0.3 and 0 (multi-token), and the
    block commit with the accepted counts, against the oracle for 10 steps."""
    cfg = W.DecodeConfig("tiny_bc", batch=2, prefix_lo=37, prefix_hi=50, prefixes=(37, 50),
                         B=4, hq=4, hkv=2, d=64, hidden=256, vocab=512, taus=(0.3, 0.0),
                         tau_period=2, steps=10)
    inp = W.make_decode_inputs(cfg, seed=0, extra_pages=2)
    bc = BlockCache(inp, cfg, 8, seed=1)
    w = inp.w.to(DEV)
    ws_h = _ws(mars.mars_workspace_bytes(mars.OP_HEAD_ACCEPT, cfg.batch, cfg.B, vocab=cfg.vocab))
    for step in range(cfg.steps):
        tau = cfg.tau_at(step)
        o, ref = bc.attend(inp.q[step], inp.k_blk[step], inp.v_blk[step], 128, cfg)
        assert_attn_close(o.cpu().numpy(), ref, f"step {step} attention")
        tok = torch.empty(cfg.batch, cfg.B, dtype=torch.int32, device=DEV)
        mp = torch.empty(cfg.batch, cfg.B, dtype=torch.float32, device=DEV)
        n = torch.empty(cfg.batch, dtype=torch.int32, device=DEV)
        mars.mars_head_accept(inp.h[step].to(DEV), w, cfg.batch, cfg.B, tau, tok, mp, n, ws_h)
        torch.cuda.synchronize()
        rt, rp, rn, gap = oracle.head_accept(f64(inp.h[step]), f64(inp.w), cfg.batch, cfg.B, tau)
        compare_head(tok.cpu().numpy(), mp.cpu().numpy(), n.cpu().numpy(), rt, rp, rn, gap, tau)
        bc.commit(inp.k_blk[step], inp.v_blk[step], n.cpu().numpy(), cfg)


def test_block_cache_unmapped_page_is_flagged_and_skipped():
    """A page the caller unmaps between the call that fills the blocks and the call that
    writes them: the write of that block stops before the unmapped row (the rows before it
    are written and counted, the rest is dropped), ST_NOPAGE is raised, and the rows the
    sequence would take next, also on that page, are not taken."""
    cfg = W.DecodeConfig("bcu", batch=2, prefix_lo=0, prefix_hi=0, prefixes=(12, 3), B=8,
                         hq=2, hkv=2, d=64, hidden=64, vocab=64)
    inp = W.make_decode_inputs(cfg, seed=7, steps=3, with_head=False, extra_pages=1)
    bc = BlockCache(inp, cfg, 8, seed=2)
    slots = torch.empty(2, 8, dtype=torch.int32, device=DEV)
    nd = torch.tensor([8, 8], dtype=torch.int32, device=DEV)
    for step in range(2):
        if step == 1:
            bc.bt[0, 1] = -1                   # positions 16..31 of sequence 0: no page
        kb, vb = inp.k_blk[step].to(DEV), inp.v_blk[step].to(DEV)
        mars.mars_kv_commit_block(kb, vb, nd, bc.sl, bc.fill, bc.ks, bc.vs, bc.sync, bc.bt,
                                  bc.kp, bc.vp, slots, bc.status)
        torch.cuda.synchronize()
        if step == 0:
            assert int(bc.status.item()) == 0 and bool(bc.sync[0].item())
    assert int(bc.status.item()) & mars.ST_NOPAGE
    assert bc.sl.cpu().tolist() == [16, 11]
    assert bc.fill.cpu().tolist() == [0, 8]
    assert (slots.cpu().numpy()[0] == -1).all()
    page0 = int(inp.block_table[0, 0])
    got = f64(bc.kp[page0, :, 12:16].cpu())                  # [hkv, 4, d]
    np.testing.assert_array_equal(got.transpose(1, 0, 2), f64(inp.k_blk[0][0, :4]))
