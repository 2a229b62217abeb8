"""GPU-vs-oracle parity of the four C-ABI entry points (needs a GB300).

Small cases run the oracle on every output; they span several tiles/splits and ragged
tails. The configuration-sized cases compare sampled outputs the oracle computes one by
one. Comparison rules are in parity_util.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_masked_token_gb300 import mars
from block_masked_token_gb300 import workloads as W
from parity_util import (UPSTREAM_REL, assert_attn_close, assert_within_bound, compare_head,
                         logit_rel_error, product_error_bound)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def f64(t):
    return W.to_f64(t)


def _ws(nbytes):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=DEV)


# --------------------------------------------------------------------------- helpers

def run_dual(q, k, v, L, B):
    o = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    mars.mars_attn_dual_stream(q, k, v, o, L=L, B=B)
    torch.cuda.synchronize()
    return o


def run_decode(inp, step, seq_lens, cfg, max_len_hint=None):
    q = inp.q[step].to(DEV)
    kb = inp.k_blk[step].to(DEV)
    vb = inp.v_blk[step].to(DEV)
    b = cfg.batch
    o = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    hint = int(seq_lens.max()) if max_len_hint is None else max_len_hint
    ws = _ws(mars.mars_workspace_bytes(mars.OP_DECODE_ATTN, b, cfg.B, cfg.hq, cfg.hkv, cfg.d,
                                       max_len=hint))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mars.mars_decode_attn(q, kb, vb, inp.k_pool_dev, inp.v_pool_dev, inp.bt_dev,
                          seq_lens.to(DEV), hint, o, ws, st)
    torch.cuda.synchronize()
    return o, int(st.item())


def run_head(h, w, batch, B, tau):
    tokens = torch.empty(batch, B, dtype=torch.int32, device=DEV)
    maxprob = torch.empty(batch, B, dtype=torch.float32, device=DEV)
    n = torch.empty(batch, dtype=torch.int32, device=DEV)
    ws = _ws(mars.mars_workspace_bytes(mars.OP_HEAD_ACCEPT, batch, B, vocab=w.shape[0]))
    mars.mars_head_accept(h, w, batch, B, tau, tokens, maxprob, n, ws)
    torch.cuda.synchronize()
    return tokens.cpu().numpy(), maxprob.cpu().numpy(), n.cpu().numpy()


def _to_dev(inp):
    inp.k_pool_dev = inp.k_pool.to(DEV)
    inp.v_pool_dev = inp.v_pool.to(DEV)
    inp.bt_dev = inp.block_table.to(DEV)
    return inp


# ------------------------------------------------------------------ dual-stream attention

@pytest.mark.parametrize("b,L,B,hq,hkv,d", [
    (1, 1, 1, 1, 1, 64),          # degenerate: one position per stream
    (2, 4, 2, 2, 1, 64),
    (1, 37, 4, 4, 2, 64),         # L not a multiple of B: short last block
    (2, 130, 16, 4, 4, 128),      # spans several 128-row tiles + ragged tail
    (1, 200, 3, 7, 1, 128),       # GQA 7, odd B
    (1, 64, 64, 2, 2, 64),        # B = L: masked stream sees no clean key
    (1, 50, 1, 2, 1, 64),         # B = 1
    (1, 33, 40, 2, 1, 128),       # B > L: one block
    (1, 300, 128, 2, 1, 128),     # B = tile: masked rows use one clean tile fewer
    (1, 300, 200, 2, 2, 64),      # B > tile, straddling tiles: key tiles only clean rows use
    (3, 257, 5, 3, 3, 128),       # no grouping (hq = hkv), one row past two full tiles
])
def test_dual_stream_small(b, L, B, hq, hkv, d):
    cfg = W.DualStreamConfig("t", b, L, B, hq, hkv, d)
    x = W.make_dual_stream_inputs(cfg, seed=L * 7 + B)
    o = run_dual(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), L, B)
    ref = oracle.attn_dual_stream(f64(x["q"]), f64(x["k"]), f64(x["v"]), L, B)
    assert_attn_close(o.cpu().numpy(), ref)


def test_dual_stream_config_0p5b_full():
    cfg = W.DUAL_STREAM_0P5B
    x = W.make_dual_stream_inputs(cfg, seed=0)
    o = run_dual(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), cfg.L, cfg.B)
    ref = oracle.attn_dual_stream(f64(x["q"]), f64(x["k"]), f64(x["v"]), cfg.L, cfg.B)
    assert_attn_close(o.cpu().numpy(), ref)


def test_dual_stream_config_7b_sampled():
    cfg = W.DUAL_STREAM_7B
    x = W.make_dual_stream_inputs(cfg, seed=0, device=DEV)
    o = run_dual(x["q"], x["k"], x["v"], cfg.L, cfg.B)
    L = cfg.L
    rows = sorted({0, 1, 127, 128, 4095, L, L + 1, L + 15, L + 16, L + 127, L + 128, 2 * L - 1,
                   *np.random.default_rng(0).integers(0, 2 * L, 24).tolist()})
    q, k, v = f64(x["q"]), f64(x["k"]), f64(x["v"])
    for bb, h in [(0, 0), (1, 13), (1, 27)]:
        ref = oracle.attn_dual_stream(q, k, v, L, cfg.B, rows=rows, heads=[h], batches=[bb])
        got = o[bb, rows, h].cpu().numpy()
        assert_attn_close(got, ref[bb, :, h], f"dual 7B b{bb} h{h}")
    # every one of the 2L = 8192 rows of one (batch, head)
    bb, h = 1, 20
    ref = oracle.attn_dual_stream(q, k, v, L, cfg.B, heads=[h], batches=[bb])
    assert_attn_close(o[bb, :, h].cpu().numpy(), ref[bb, :, h], f"dual 7B b{bb} h{h} all rows")


def test_dual_stream_many_items_per_cta():
    """More work items than SMs at d = 64 with a ragged last query tile and an odd block
    size: each persistent CTA runs several items, so the rings, S buffers, O staging and
    barrier phases carry over from item to item."""
    cfg = W.DualStreamConfig("t", 3, 700, 7, 12, 3, 64)
    x = W.make_dual_stream_inputs(cfg, seed=11)
    o = run_dual(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), cfg.L, cfg.B)
    ref = oracle.attn_dual_stream(f64(x["q"]), f64(x["k"]), f64(x["v"]), cfg.L, cfg.B)
    assert_attn_close(o.cpu().numpy(), ref)


def test_dual_stream_divergent_rescale():
    """One query row meets a key scoring far above its earlier maximum in a later key tile
    while the other rows of its warp do not: the per-row running maximum is raised for
    that row only (exercises the lazy rescale of O with rows that disagree)."""
    cfg = W.DualStreamConfig("t", 1, 300, 4, 2, 1, 64)
    x = W.make_dual_stream_inputs(cfg, seed=5)
    q, k = x["q"].clone(), x["k"].clone()
    qrow = q[0, 290, 0].float()
    k[0, 280, 0] = (4.0 * qrow).to(torch.bfloat16)      # clean key tile 2, row 290 only
    qm = q[0, 300 + 150, 1].float()
    k[0, 140, 0] = (4.0 * qm).to(torch.bfloat16)        # masked row t=150: clean key tile 1
    o = run_dual(q.to(DEV), k.to(DEV), x["v"].to(DEV), cfg.L, cfg.B)
    ref = oracle.attn_dual_stream(f64(q), f64(k), f64(x["v"]), cfg.L, cfg.B)
    assert_attn_close(o.cpu().numpy(), ref)


# Attention gradient. The kernels round P (for dV) and dS (for dQ, dK; formed from the
# rounded P) to bf16 before their tensor-core products; each output element is checked
# against the error bound of that
# arithmetic (parity_util.product_error_bound), computed from the oracle's own P, dP, D
# and dS. The cases give the kernels the oracle's forward output as O and an upstream
# gradient whose values bf16 represents exactly, so that neither the forward's error nor
# the kernels' bf16 copy of dO enters the comparison.

def bf16_exact_randn(shape, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(shape, generator=g, device=DEV).to(torch.bfloat16).to(torch.float32)


def gpu_dual_grad(x, o, d_o, L, B):
    q, k, v = x["q"], x["k"], x["v"]
    b, n, hq, d = q.shape
    hkv = k.shape[2]
    ws = _ws(mars.mars_workspace_bytes(mars.OP_DUAL_GRAD, b, B, hq, hkv, d, max_len=L))
    dq = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    dk = torch.empty(k.shape, dtype=torch.float32, device=DEV)
    dv = torch.empty(v.shape, dtype=torch.float32, device=DEV)
    mars.mars_attn_dual_stream_grad(q, k, v, o, d_o, L, B, dq, dk, dv, ws)
    torch.cuda.synchronize()
    return dq, dk, dv


def check_dual_grad(q, k, v, do, L, B, dq, dk, dv, what):
    """dq, dk, dv (GPU, any array-likes of the full shapes of q, k, v) against the oracle,
    element by element within the error bound; q, k, v, do are float64."""
    b, n, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    rq, rk, rv = (np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape))
    s1q, s2q, s3q = np.zeros(q.shape), np.zeros(q.shape), np.zeros(q.shape)
    s1k, s2k, s3k = np.zeros(k.shape), np.zeros(k.shape), np.zeros(k.shape)
    s1v, s2v = np.zeros(v.shape), np.zeros(v.shape)
    for bi, h, hk, P, dP, Dr, dS in oracle.attn_dual_stream_grad_parts(q, k, v, do, L, B):
        Ks, Qs, dO = scale * k[bi, :, hk], scale * q[bi, :, h], do[bi, :, h]
        rq[bi, :, h] = dS @ Ks
        rk[bi, :, hk] += dS.T @ Qs
        rv[bi, :, hk] += P.T @ dO
        adS, dS2, X = np.abs(dS), dS * dS, P * (np.abs(dP) + np.abs(Dr))
        aK, aQ = np.abs(Ks), np.abs(Qs)
        s1q[bi, :, h] = adS @ aK
        s2q[bi, :, h] = dS2 @ (Ks * Ks)
        s3q[bi, :, h] = X @ aK
        s1k[bi, :, hk] += adS.T @ aQ
        s2k[bi, :, hk] += dS2.T @ (Qs * Qs)
        s3k[bi, :, hk] += X.T @ aQ
        s1v[bi, :, hk] += P.T @ np.abs(dO)
        s2v[bi, :, hk] += (P * P).T @ (dO * dO)
        del P, dP, dS, adS, dS2, X
    worst = {}
    for got, ref, bnd, name in (
            (dq, rq, product_error_bound(s1q, s2q, n, UPSTREAM_REL * s3q, roundings=2), "dq"),
            (dk, rk, product_error_bound(s1k, s2k, n, UPSTREAM_REL * s3k, extra_roundings=G,
                                         roundings=2), "dk"),
            (dv, rv, product_error_bound(s1v, s2v, n, None, extra_roundings=G), "dv")):
        worst[name] = assert_within_bound(np.asarray(got), ref, bnd, f"{what} {name}")
    return worst


def grad_case(x, L, B, seed=17):
    """The GPU gradient of inputs x (bf16, on the host) with the oracle's O and a
    bf16-exact dO, checked against the oracle."""
    q64, k64, v64 = f64(x["q"]), f64(x["k"]), f64(x["v"])
    o = torch.from_numpy(oracle.attn_dual_stream(q64, k64, v64, L, B)).float().to(DEV)
    d_o = bf16_exact_randn(o.shape, seed)
    xd = {kk: vv.to(DEV) for kk, vv in x.items()}
    dq, dk, dv = gpu_dual_grad(xd, o, d_o, L, B)
    return check_dual_grad(q64, k64, v64, f64(d_o), L, B, dq.cpu().numpy(), dk.cpu().numpy(),
                           dv.cpu().numpy(), f"grad L={L} B={B}")


@pytest.mark.parametrize("b,L,B,hq,hkv,d", [
    (1, 8, 2, 2, 1, 64),
    (2, 37, 4, 4, 2, 64),          # L not a multiple of B
    (1, 130, 16, 7, 1, 128),       # GQA 7, ragged
    (1, 64, 64, 2, 2, 128),        # B = L
    (1, 20, 1, 2, 1, 64),          # B = 1: masked rows see only themselves among masked keys
    (1, 33, 40, 2, 2, 128),        # B > L: one block
    (1, 300, 48, 4, 2, 64),        # blocks straddle 128-key tiles; three key tiles a stream
])
def test_dual_stream_grad_small(b, L, B, hq, hkv, d):
    cfg = W.DualStreamConfig("g", b, L, B, hq, hkv, d)
    grad_case(W.make_dual_stream_inputs(cfg, seed=L + B), L, B)


def test_dual_stream_lse_matches_oracle():
    """The forward with row statistics writes the same O as the plain forward and, per row,
    the log2 softmax denominator of the oracle; the pad rows of the last tile are 0."""
    cfg = W.DualStreamConfig("lse", 2, 200, 16, 4, 2, 128)
    x = W.make_dual_stream_inputs(cfg, seed=21)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o = run_dual(q, k, v, cfg.L, cfg.B)
    o2 = torch.empty_like(o)
    lse = torch.full(mars.dual_lse_shape(2, 4, cfg.L), float("nan"), device=DEV)
    mars.mars_attn_dual_stream_lse(q, k, v, o2, lse, cfg.L, cfg.B)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    ref = oracle.attn_dual_stream_lse(f64(x["q"]), f64(x["k"]), cfg.L, cfg.B)
    got = lse.cpu().double().numpy()
    for s_ in range(2):
        err = np.abs(got[:, :, s_, :cfg.L] - ref[:, :, s_ * cfg.L:(s_ + 1) * cfg.L]).max()
        assert err < 1e-3, f"stream {s_}: lse max-abs error {err:.2e}"
    assert (got[:, :, :, cfg.L:] == 0).all()


def test_dual_stream_lse_7b_one_head():
    """The row statistics of the full 2L = 8192 workload (3584 items, several per CTA), for
    every row of one head, against the oracle; O as the plain forward's."""
    cfg = W.DUAL_STREAM_7B
    x = W.make_dual_stream_inputs(cfg, seed=0, device=DEV)
    q, k, v = x["q"], x["k"], x["v"]
    o = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    lse = torch.empty(mars.dual_lse_shape(cfg.batch, cfg.hq, cfg.L), device=DEV)
    mars.mars_attn_dual_stream_lse(q, k, v, o, lse, cfg.L, cfg.B)
    torch.cuda.synchronize()
    assert torch.equal(o, run_dual(q, k, v, cfg.L, cfg.B))
    bb, h = 1, 13
    kvh = h // (cfg.hq // cfg.hkv)
    ref = oracle.attn_dual_stream_lse(f64(q[bb:bb + 1, :, h:h + 1]),
                                      f64(k[bb:bb + 1, :, kvh:kvh + 1]), cfg.L, cfg.B)
    got = lse[bb, h].cpu().double().numpy()                 # [2, Lp]
    for s_ in range(2):
        err = np.abs(got[s_, :cfg.L] - ref[0, 0, s_ * cfg.L:(s_ + 1) * cfg.L]).max()
        assert err < 1e-3, f"stream {s_}: lse max-abs error {err:.2e}"


def test_dual_stream_grad_from_lse_matches_plain_grad():
    """The gradient from the forward's statistics equals the plain gradient (which
    recomputes them with the same kernel): dQ bit for bit, dK/dV up to the order of their
    fp32 atomic sums (G = 2 adds per element: a few fp32 ulps of the largest summand)."""
    cfg = W.DualStreamConfig("glse", 1, 300, 48, 4, 2, 64)
    x = W.make_dual_stream_inputs(cfg, seed=8)
    xd = {kk: vv.to(DEV) for kk, vv in x.items()}
    q, k, v = xd["q"], xd["k"], xd["v"]
    o = run_dual(q, k, v, cfg.L, cfg.B)
    d_o = bf16_exact_randn(o.shape, 17)
    dq, dk, dv = gpu_dual_grad(xd, o, d_o, cfg.L, cfg.B)
    o2 = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    lse = torch.empty(mars.dual_lse_shape(1, 4, cfg.L), device=DEV)
    mars.mars_attn_dual_stream_lse(q, k, v, o2, lse, cfg.L, cfg.B)
    ws = _ws(mars.mars_workspace_bytes(mars.OP_DUAL_GRAD, 1, cfg.B, 4, 2, 64, max_len=cfg.L))
    dq2, dk2, dv2 = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    mars.mars_attn_dual_stream_grad_lse(q, k, v, o2, d_o, lse, cfg.L, cfg.B, dq2, dk2, dv2, ws)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq2)
    for a_, b_, name in ((dk, dk2, "dk"), (dv, dv2, "dv")):
        a_, b_ = a_.cpu().double().numpy(), b_.cpu().double().numpy()
        tol = 8 * 2.0 ** -24 * np.maximum(np.abs(a_), np.abs(b_)).max(axis=-1, keepdims=True)
        assert (np.abs(a_ - b_) <= tol).all(), f"{name}: differs beyond the atomic-order bound"


def test_dual_stream_grad_many_items_per_cta():
    """More (batch, kv head, key tile) work items than SMs, so persistent CTAs carry the
    rings, TMEM accumulators and barrier phases from item to item; ragged L, odd-sized
    blocks that straddle key tiles."""
    cfg = W.DualStreamConfig("gm", 3, 1100, 24, 6, 3, 64)
    grad_case(W.make_dual_stream_inputs(cfg, seed=5), cfg.L, cfg.B)


def test_dual_stream_grad_many_items_per_cta_d128():
    """d = 128 with about three work items per persistent CTA in both gradient kernels
    (504 key-tile items, 504 query-tile items), so the two MMA issuer threads of each
    kernel hand the TMEM accumulators over from item to item; ragged L, blocks of 24 that
    straddle 128-row tiles."""
    cfg = W.DualStreamConfig("gm128", 2, 1100, 24, 14, 2, 128)
    grad_case(W.make_dual_stream_inputs(cfg, seed=6), cfg.L, cfg.B)


def test_dual_stream_grad_7b_full_size_one_kv_group():
    """The timed gradient workload itself (batch 2, 2L = 8192, 28/4 heads, d 128, B 16:
    3584 items in each kernel, run as the bench launches them), checked on one whole kv
    group: dQ of its 7 query heads and dK, dV of its kv head, every element. O is the GPU
    forward's except on the checked group, which gets the oracle's."""
    cfg = W.DUAL_STREAM_7B
    x = W.make_dual_stream_inputs(cfg, seed=0, device=DEV)
    G = cfg.hq // cfg.hkv
    bb, kvh = 1, 2
    hs, ks = slice(kvh * G, (kvh + 1) * G), slice(kvh, kvh + 1)
    q64, k64, v64 = (f64(x[n][bb:bb + 1, :, sl]) for n, sl in (("q", hs), ("k", ks), ("v", ks)))
    o = run_dual(x["q"], x["k"], x["v"], cfg.L, cfg.B)
    o[bb:bb + 1, :, hs] = torch.from_numpy(oracle.attn_dual_stream(q64, k64, v64, cfg.L,
                                                                   cfg.B)).float().to(DEV)
    d_o = bf16_exact_randn(o.shape, 17)
    dq, dk, dv = gpu_dual_grad(x, o, d_o, cfg.L, cfg.B)
    check_dual_grad(q64, k64, v64, f64(d_o[bb:bb + 1, :, hs]), cfg.L, cfg.B,
                    dq[bb:bb + 1, :, hs].cpu().numpy(), dk[bb:bb + 1, :, ks].cpu().numpy(),
                    dv[bb:bb + 1, :, ks].cpu().numpy(), "grad 7B full size")


def test_dual_stream_grad_7b_heads_2l2048():
    """7B head shapes (one kv group of 7 query heads, d 128), 2L = 2048, B = 16."""
    cfg = W.DualStreamConfig("g7", 1, 1024, 16, 7, 1, 128)
    grad_case(W.make_dual_stream_inputs(cfg, seed=3), 1024, 16)


# ------------------------------------------------------------------------ decode attention

def _decode_case(cfg, seed=0, steps=1, extra_pages=3):
    inp = W.make_decode_inputs(cfg, seed=seed, steps=steps, with_head=False,
                               extra_pages=extra_pages)
    return _to_dev(inp)


@pytest.mark.parametrize("cfg", [
    W.TINY_DECODE,
    W.DecodeConfig("d1", batch=3, prefix_lo=0, prefix_hi=40, prefixes=(0, 17, 300), B=1,
                   hq=2, hkv=2, d=64, hidden=64, vocab=64),
    W.DecodeConfig("d2", batch=4, prefix_lo=100, prefix_hi=1500, B=8, hq=28, hkv=4, d=128,
                   hidden=64, vocab=64),
    W.DecodeConfig("d3", batch=2, prefix_lo=1, prefix_hi=9, prefixes=(1, 9), B=16, hq=7,
                   hkv=1, d=128, hidden=64, vocab=64),
    W.DecodeConfig("d4", batch=5, prefix_lo=500, prefix_hi=3000, B=3, hq=8, hkv=2, d=64,
                   hidden=64, vocab=64),
    # the KV-cached AR step at 7B attention shapes: one query per sequence
    W.DecodeConfig("d5", batch=4, prefix_lo=2048, prefix_hi=8192, B=1, hq=28, hkv=4, d=128,
                   hidden=64, vocab=64),
    # the largest query tile: G * B = 4 * 32 = 128 rows per kv head
    W.DecodeConfig("d8", batch=2, prefix_lo=0, prefix_hi=0, prefixes=(129, 1000), B=32, hq=8,
                   hkv=2, d=128, hidden=64, vocab=64),
    # empty prefixes: only the block keys
    W.DecodeConfig("d9", batch=3, prefix_lo=0, prefix_hi=0, prefixes=(0, 0, 0), B=16, hq=4,
                   hkv=1, d=64, hidden=64, vocab=64),
    # 400 one-tile pairs: several waves of CTAs, ordered longest first
    W.DecodeConfig("d10", batch=200, prefix_lo=0, prefix_hi=0, prefixes=(0,) * 200, B=4,
                   hq=4, hkv=2, d=64, hidden=64, vocab=64),
    # very uneven prefixes, few pairs: the long ones split, some splits past a short end
    W.DecodeConfig("d11", batch=7, prefix_lo=0, prefix_hi=0,
                   prefixes=(3000, 5, 130, 0, 700, 4096, 1), B=8, hq=8, hkv=2, d=128,
                   hidden=64, vocab=64),
])
def test_decode_small(cfg):
    inp = _decode_case(cfg, seed=1)
    o, st = run_decode(inp, 0, inp.prefix_lens, cfg)
    assert st == 0
    ref = oracle.decode_attn(f64(inp.q[0]), f64(inp.k_blk[0]), f64(inp.v_blk[0]),
                             f64(inp.k_pool), f64(inp.v_pool), inp.block_table.numpy(),
                             inp.prefix_lens.numpy(), cfg.page_size)
    assert_attn_close(o.cpu().numpy(), ref)


def test_decode_divergent_rescale():
    """A prefix key far along the cache scores far above every earlier key for one query
    row only (block position 0, head 0), so that row alone raises its running maximum
    inside a warp of rows that do not."""
    cfg = W.DecodeConfig("dr", batch=2, prefix_lo=0, prefix_hi=0, prefixes=(700, 333), B=4,
                         hq=4, hkv=1, d=64, hidden=64, vocab=64)
    inp = W.make_decode_inputs(cfg, seed=6, steps=1, with_head=False, extra_pages=2)
    qrow = inp.q[0][0, 0, 0].float()
    pos = 660                   # second key tile of the split that holds it
    page = int(inp.block_table[0, pos // 16])
    inp.k_pool[page, 0, pos % 16] = (4.0 * qrow).to(torch.bfloat16)
    _to_dev(inp)
    o, st = run_decode(inp, 0, inp.prefix_lens, cfg)
    assert st == 0
    ref = oracle.decode_attn(f64(inp.q[0]), f64(inp.k_blk[0]), f64(inp.v_blk[0]),
                             f64(inp.k_pool), f64(inp.v_pool), inp.block_table.numpy(),
                             inp.prefix_lens.numpy(), cfg.page_size)
    assert_attn_close(o.cpu().numpy(), ref)


def test_decode_hint_smaller_than_length_is_still_correct():
    cfg = W.DecodeConfig("d5", batch=3, prefix_lo=600, prefix_hi=2000, B=4, hq=4, hkv=2,
                         d=64, hidden=64, vocab=64)
    inp = _decode_case(cfg, seed=2)
    o, st = run_decode(inp, 0, inp.prefix_lens, cfg, max_len_hint=100)
    ref = oracle.decode_attn(f64(inp.q[0]), f64(inp.k_blk[0]), f64(inp.v_blk[0]),
                             f64(inp.k_pool), f64(inp.v_pool), inp.block_table.numpy(),
                             inp.prefix_lens.numpy(), cfg.page_size)
    assert st == 0
    assert_attn_close(o.cpu().numpy(), ref)


def test_decode_hint_far_above_lengths():
    """A length hint far above the prefixes plans many splits per pair, most of them past
    the prefix ends (empty partials that the merge skips)."""
    cfg = W.DecodeConfig("dh", batch=2, prefix_lo=0, prefix_hi=0, prefixes=(3, 40), B=4,
                         hq=4, hkv=2, d=64, hidden=64, vocab=64)
    inp = _decode_case(cfg, seed=4)
    o, st = run_decode(inp, 0, inp.prefix_lens, cfg, max_len_hint=20000)
    assert st == 0
    ref = oracle.decode_attn(f64(inp.q[0]), f64(inp.k_blk[0]), f64(inp.v_blk[0]),
                             f64(inp.k_pool), f64(inp.v_pool), inp.block_table.numpy(),
                             inp.prefix_lens.numpy(), cfg.page_size)
    assert_attn_close(o.cpu().numpy(), ref)


def test_decode_unmapped_page_sets_status():
    cfg = W.TINY_DECODE
    inp = _decode_case(cfg)
    inp.block_table[1, 1] = -1
    inp.bt_dev = inp.block_table.to(DEV)
    _, st = run_decode(inp, 0, inp.prefix_lens, cfg)
    assert st & mars.ST_NOPAGE


@pytest.mark.parametrize("d", [64, 128])
def test_decode_empty_pool_leaves_only_block_keys(d):
    """No pool and no block table while the lengths say there is a prefix: every prefix key
    is unmapped (flagged), nothing is read for it, and each query attends to the block keys
    alone, i.e. the oracle's output for an empty prefix."""
    cfg = W.DecodeConfig("de", batch=3, prefix_lo=0, prefix_hi=0, prefixes=(5, 200, 31),
                         B=4, hq=8, hkv=2, d=d, hidden=64, vocab=64)
    inp = W.make_decode_inputs(cfg, seed=2, steps=1, with_head=False)
    q, kb, vb = inp.q[0].to(DEV), inp.k_blk[0].to(DEV), inp.v_blk[0].to(DEV)
    pool = torch.empty(0, cfg.hkv, cfg.page_size, d, dtype=torch.bfloat16, device=DEV)
    bt = torch.empty(cfg.batch, 0, dtype=torch.int32, device=DEV)
    o = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    hint = int(inp.prefix_lens.max())
    ws = _ws(mars.mars_workspace_bytes(mars.OP_DECODE_ATTN, cfg.batch, cfg.B, cfg.hq, cfg.hkv,
                                       d, max_len=hint))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mars.mars_decode_attn(q, kb, vb, pool, pool, bt, inp.prefix_lens.to(DEV), hint, o, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) & mars.ST_OVERFLOW
    none = np.zeros(cfg.batch, dtype=np.int64)
    ref = oracle.decode_attn(f64(inp.q[0]), f64(inp.k_blk[0]), f64(inp.v_blk[0]),
                             np.zeros((0, cfg.hkv, cfg.page_size, d)),
                             np.zeros((0, cfg.hkv, cfg.page_size, d)),
                             np.zeros((cfg.batch, 0), dtype=np.int64), none, cfg.page_size)
    assert_attn_close(o.cpu().numpy(), ref)


def test_decode_single_split_direct_output():
    """With at least as many (sequence, kv head) pairs as SMs the kernel runs one split
    per pair and writes the normalised output directly (no merge pass)."""
    cfg = W.DecodeConfig("d6", batch=160, prefix_lo=0, prefix_hi=300, B=4, hq=4, hkv=2, d=64,
                         hidden=64, vocab=64)
    inp = _decode_case(cfg, seed=8)
    o, st = run_decode(inp, 0, inp.prefix_lens, cfg)
    assert st == 0
    ref = oracle.decode_attn(f64(inp.q[0]), f64(inp.k_blk[0]), f64(inp.v_blk[0]),
                             f64(inp.k_pool), f64(inp.v_pool), inp.block_table.numpy(),
                             inp.prefix_lens.numpy(), cfg.page_size)
    assert_attn_close(o.cpu().numpy(), ref)


def test_decode_multi_split_merge():
    """Few pairs and long prefixes: the keys are split across CTAs (here 5 splits of 2048
    keys for the longest sequence, some splits past the shorter one's end) and merged."""
    cfg = W.DecodeConfig("d7", batch=2, prefix_lo=0, prefix_hi=0, prefixes=(9000, 4100), B=8,
                         hq=7, hkv=1, d=128, hidden=64, vocab=64)
    inp = _decode_case(cfg, seed=9)
    o, st = run_decode(inp, 0, inp.prefix_lens, cfg)
    assert st == 0
    ref = oracle.decode_attn(f64(inp.q[0]), f64(inp.k_blk[0]), f64(inp.v_blk[0]),
                             f64(inp.k_pool), f64(inp.v_pool), inp.block_table.numpy(),
                             inp.prefix_lens.numpy(), cfg.page_size)
    assert_attn_close(o.cpu().numpy(), ref)


def test_decode_sustained_config_sampled():
    """Batch 128, prefixes 2048..8192, B=16, 7B heads: sampled sequences (single-split
    path, the shape the decode step of the benchmark runs)."""
    cfg = W.SUSTAINED_DECODE_7B
    inp = _to_dev(W.make_decode_inputs(cfg, seed=0, device=DEV, steps=1, with_head=False))
    hint = int(inp.prefix_lens.max()) + cfg.B * cfg.steps
    o, st = run_decode(inp, 0, inp.prefix_lens, cfg, max_len_hint=hint)
    assert st == 0
    seqs = [0, 64, 127]
    ref = oracle.decode_attn(f64(inp.q[0]), f64(inp.k_blk[0]), f64(inp.v_blk[0]),
                             f64(inp.k_pool), f64(inp.v_pool), inp.block_table.cpu().numpy(),
                             inp.prefix_lens.numpy(), cfg.page_size, seqs=seqs)
    assert_attn_close(o.cpu().numpy()[seqs], ref[seqs], "decode sustained")


def test_decode_config_7b_sampled():
    cfg = W.DECODE_7B
    inp = _to_dev(W.make_decode_inputs(cfg, seed=0, device=DEV, with_head=False))
    o, st = run_decode(inp, 0, inp.prefix_lens, cfg)
    assert st == 0
    seqs = [0, 5, 17, 31]
    ref = oracle.decode_attn(f64(inp.q[0]), f64(inp.k_blk[0]), f64(inp.v_blk[0]),
                             f64(inp.k_pool), f64(inp.v_pool), inp.block_table.cpu().numpy(),
                             inp.prefix_lens.numpy(), cfg.page_size, seqs=seqs)
    assert_attn_close(o.cpu().numpy()[seqs], ref[seqs], "decode 7B")


# --------------------------------------------------------------------------------- head

@pytest.mark.parametrize("batch,B,hidden,vocab,tau", [
    (2, 4, 256, 512, 0.9),
    (3, 5, 64, 1000, 0.5),          # ragged vocabulary tile
    (1, 16, 128, 77, 0.0),          # tau 0: whole block
    (4, 8, 512, 3000, 1.0),         # tau 1: plain AR
    (2, 32, 96, 300, 0.3),
    (1, 4, 64, 1, 1.0),             # one-word vocabulary: p = 1 >= tau = 1, the whole block
    (20, 16, 128, 77, 0.5),         # 320 rows (paired form) over a vocabulary smaller than
                                    # one W half: the odd CTA's half is all past the end
    (17, 16, 64, 1, 1.0),           # paired form, one-word vocabulary
    (20, 16, 200, 1000, 0.3),       # paired form, hidden 200: a ragged last k-block
])
def test_head_small(batch, B, hidden, vocab, tau):
    cfg = W.DecodeConfig("h", batch=batch, prefix_lo=1, prefix_hi=1, B=B, hq=1, hkv=1, d=64,
                         hidden=hidden, vocab=vocab, taus=(tau,))
    inp = W.make_decode_inputs(cfg, seed=3)
    tok, p, n = run_head(inp.h[0].to(DEV), inp.w.to(DEV), batch, B, tau)
    rt, rp, rn, gap = oracle.head_accept(f64(inp.h[0]), f64(inp.w), batch, B, tau)
    compare_head(tok, p, n, rt, rp, rn, gap, tau)
    if tau == 1.0 and vocab > 1:
        assert (n == 1).all()
    if tau == 0.0:
        assert (n == B).all()


@pytest.mark.parametrize("batch,B,tau", [
    (60, 5, 0.3),          # 300 rows: sequences straddle the boundaries at rows 128 and 256
    (20, 24, 0.0),         # whole blocks accepted across two straddles (rows 128, 256)
    (37, 7, 0.2),          # two straddles and a ragged last row block
    (9, 32, 0.1),          # B = 32 divides 128: no straddle, several sequences per block
    (130, 1, 0.5),         # the AR step's head: one row per sequence, two row blocks
    (150, 16, 0.4),        # 19 row blocks: a second tile group of 3 (an odd pair count)
])
def test_head_sequences_across_row_blocks(batch, B, tau):
    """The acceptance scan runs where the last partial of a 128-row block is merged; a
    sequence whose B rows straddle two blocks is scanned once both are merged."""
    cfg = W.DecodeConfig("hs", batch=batch, prefix_lo=1, prefix_hi=1, B=B, hq=1, hkv=1, d=64,
                         hidden=128, vocab=1000, taus=(tau,))
    inp = W.make_decode_inputs(cfg, seed=batch + B)
    tok, p, n = run_head(inp.h[0].to(DEV), inp.w.to(DEV), batch, B, tau)
    rt, rp, rn, gap = oracle.head_accept(f64(inp.h[0]), f64(inp.w), batch, B, tau)
    compare_head(tok, p, n, rt, rp, rn, gap, tau)
    # the same call with one threshold per sequence (0 or tau, alternating)
    taus = [0.0 if s % 2 else tau for s in range(batch)]
    tok2, p2, n2 = run_head_per_request(inp.h[0].to(DEV), inp.w.to(DEV), batch, B, taus)
    rt2, rp2, rn2, gap2 = oracle.head_accept_per_request(f64(inp.h[0]), f64(inp.w), batch, B,
                                                         taus)
    compare_head(tok2, p2, n2, rt2, rp2, rn2, gap2, taus)
    assert (n2[1::2] == B).all()


def test_head_tie_goes_to_lowest_index():
    batch, B, H, V = 1, 2, 64, 700
    h = torch.zeros(batch * B, H, dtype=torch.bfloat16)
    h[:, 0] = 1.0
    w = torch.zeros(V, H, dtype=torch.bfloat16)
    w[[5, 300, 650], 0] = 2.0               # equal logits in different vocabulary tiles
    w[[7], 0] = -1.0
    tok, p, n = run_head(h.to(DEV), w.to(DEV), batch, B, 0.5)
    assert (tok == 5).all()
    rt, rp, rn, _ = oracle.head_accept(f64(h), f64(w), batch, B, 0.5)
    assert (rt == 5).all()
    np.testing.assert_allclose(p, rp, atol=1e-4)


def test_head_config_7b_sampled_rows():
    cfg = W.DECODE_7B
    g = torch.Generator(device=DEV).manual_seed(0)
    inp = W.make_decode_inputs(W.DecodeConfig(**{**cfg.__dict__, "batch": 32}), seed=0,
                               device=DEV, steps=1)
    h, w = inp.h[0], inp.w
    tok, p, n = run_head(h, w, cfg.batch, cfg.B, cfg.taus[0])
    seqs = [0, 9, 31]
    rows = [s * cfg.B + k for s in seqs for k in range(cfg.B)]
    rt, rp, rn, gap = oracle.head_accept(f64(h[rows]), f64(w), len(seqs), cfg.B, cfg.taus[0])
    compare_head(tok[seqs], p[seqs], n[seqs], rt, rp, rn, gap, cfg.taus[0])
    del g


def test_head_2048_rows_7b_every_row_block():
    """2048 rows (batch 256 x B 8) at the 7B head shape, the LM head's full tile group of
    16 row blocks: one sequence of every row block against the oracle."""
    cfg = W.DecodeConfig(**{**W.DECODE_7B.__dict__, "batch": 256})
    inp = W.make_decode_inputs(cfg, seed=4, device=DEV, steps=1)
    h, w = inp.h[0], inp.w
    tok, p, n = run_head(h, w, cfg.batch, cfg.B, cfg.taus[0])
    per = 128 // cfg.B
    seqs = [blk * per + blk % per for blk in range(cfg.batch // per)]
    rows = [s * cfg.B + k for s in seqs for k in range(cfg.B)]
    rt, rp, rn, gap = oracle.head_accept(f64(h[rows]), f64(w), len(seqs), cfg.B, cfg.taus[0])
    compare_head(tok[seqs], p[seqs], n[seqs], rt, rp, rn, gap, cfg.taus[0])
    assert ((n >= 1) & (n <= cfg.B)).all()


# ------------------------------------------------------------------------------ commit

def test_commit_matches_oracle_and_guards():
    cfg = W.DecodeConfig("c", batch=5, prefix_lo=0, prefix_hi=60, B=8, hq=4, hkv=2, d=128,
                         hidden=64, vocab=64)
    inp = W.make_decode_inputs(cfg, seed=4, steps=2, with_head=False, extra_pages=4)
    n = torch.tensor([1, 8, 3, 0, 5], dtype=torch.int32)
    kp, vp = inp.k_pool.to(DEV), inp.v_pool.to(DEV)
    sl = inp.prefix_lens.to(DEV)
    slots = torch.empty(cfg.batch, cfg.B, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mars.mars_kv_commit(inp.k_blk[0].to(DEV), inp.v_blk[0].to(DEV), n.to(DEV), sl,
                        inp.block_table.to(DEV), kp, vp, slots, st)
    torch.cuda.synchronize()
    rk, rv, rl, rs = oracle.kv_commit(f64(inp.k_blk[0]), f64(inp.v_blk[0]), n.numpy(),
                                      inp.prefix_lens.numpy(), inp.block_table.numpy(),
                                      f64(inp.k_pool), f64(inp.v_pool), cfg.page_size)
    assert int(st.item()) == 0
    np.testing.assert_array_equal(sl.cpu().numpy(), rl)
    np.testing.assert_array_equal(slots.cpu().numpy(), rs)
    # whole pools bit-exact, including the unmapped guard pages
    np.testing.assert_array_equal(f64(kp.cpu()), rk)
    np.testing.assert_array_equal(f64(vp.cpu()), rv)


def test_commit_unmapped_page_is_skipped_and_flagged():
    cfg = W.DecodeConfig("c2", batch=2, prefix_lo=0, prefix_hi=0, prefixes=(14, 3), B=4,
                         hq=2, hkv=2, d=64, hidden=64, vocab=64)
    inp = W.make_decode_inputs(cfg, seed=5, steps=1, with_head=False)
    bt = inp.block_table.clone()
    bt[0, 1] = -1                      # positions 16.. of sequence 0 have no page
    kp, vp = inp.k_pool.to(DEV), inp.v_pool.to(DEV)
    sl = inp.prefix_lens.to(DEV)
    slots = torch.empty(2, 4, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    n = torch.tensor([4, 4], dtype=torch.int32, device=DEV)
    mars.mars_kv_commit(inp.k_blk[0].to(DEV), inp.v_blk[0].to(DEV), n, sl, bt.to(DEV), kp, vp,
                        slots, st)
    torch.cuda.synchronize()
    assert int(st.item()) & mars.ST_NOPAGE
    s = slots.cpu().numpy()
    assert s[0, 0] >= 0 and s[0, 1] >= 0 and (s[0, 2:] == -1).all()
    assert sl.cpu().tolist() == [16, 7]


# ----------------------------------------------------- per-request thresholds (speed knob)

def run_head_per_request(h, w, batch, B, taus):
    tokens = torch.empty(batch, B, dtype=torch.int32, device=DEV)
    maxprob = torch.empty(batch, B, dtype=torch.float32, device=DEV)
    n = torch.empty(batch, dtype=torch.int32, device=DEV)
    ws = _ws(mars.mars_workspace_bytes(mars.OP_HEAD_ACCEPT, batch, B, vocab=w.shape[0]))
    t = torch.tensor(taus, dtype=torch.float32, device=DEV)
    mars.mars_head_accept_per_request(h, w, batch, B, t, tokens, maxprob, n, ws)
    torch.cuda.synchronize()
    return tokens.cpu().numpy(), maxprob.cpu().numpy(), n.cpu().numpy()


def test_head_per_request_small():
    """Eight sequences with eight different thresholds in one call, including 0 (the whole
    block), 1.0 (one token) and a NaN entry (compares false: one token)."""
    batch, B = 8, 6
    cfg = W.DecodeConfig("hr", batch=batch, prefix_lo=1, prefix_hi=1, B=B, hq=1, hkv=1, d=64,
                         hidden=256, vocab=1000, taus=(0.5,))
    inp = W.make_decode_inputs(cfg, seed=11)
    taus = [0.0, 0.05, 0.1, 0.2, 0.3, 0.5, 1.0, float("nan")]
    tok, p, n = run_head_per_request(inp.h[0].to(DEV), inp.w.to(DEV), batch, B, taus)
    ref_taus = [t if t == t else 2.0 for t in taus]     # NaN behaves as a threshold > 1
    rt, rp, rn, gap = oracle.head_accept_per_request(f64(inp.h[0]), f64(inp.w), batch, B,
                                                     ref_taus)
    compare_head(tok, p, n, rt, rp, rn, gap, ref_taus)
    assert n[0] == B and n[6] == 1 and n[7] == 1
    # the same call with each threshold alone reproduces its sequence
    for s in (1, 4):
        _, _, n1 = run_head(inp.h[0].to(DEV), inp.w.to(DEV), batch, B, taus[s])
        assert n1[s] == n[s]


def test_head_per_request_7b_sampled_rows():
    cfg = W.DECODE_7B
    inp = W.make_decode_inputs(W.DecodeConfig(**{**cfg.__dict__, "batch": 32}), seed=2,
                               device=DEV, steps=1)
    h, w = inp.h[0], inp.w
    taus = [(0.0, 0.3, 0.5, 0.9)[s % 4] for s in range(cfg.batch)]
    tok, p, n = run_head_per_request(h, w, cfg.batch, cfg.B, taus)
    seqs = [0, 1, 2, 3, 17, 30]
    rows = [s * cfg.B + k for s in seqs for k in range(cfg.B)]
    rt, rp, rn, gap = oracle.head_accept_per_request(f64(h[rows]), f64(w), len(seqs), cfg.B,
                                                     [taus[s] for s in seqs])
    compare_head(tok[seqs], p[seqs], n[seqs], rt, rp, rn, gap, [taus[s] for s in seqs])
    assert n[0] == cfg.B


# ------------------------------------------------------------- batch-synchronised commit

def test_commit_batch_sync_matches_oracle():
    cfg = W.DecodeConfig("cs", batch=6, prefix_lo=0, prefix_hi=70, B=8, hq=4, hkv=2, d=128,
                         hidden=64, vocab=64)
    inp = W.make_decode_inputs(cfg, seed=7, steps=1, with_head=False, extra_pages=4)
    for n_list in ([5, 8, 3, 7, 6, 4], [8, 8, 8, 8, 8, 8], [2, 9, -1, 4, 4, 4]):
        n = torch.tensor(n_list, dtype=torch.int32)
        kp, vp = inp.k_pool.to(DEV), inp.v_pool.to(DEV)
        sl = inp.prefix_lens.to(DEV)
        slots = torch.empty(cfg.batch, cfg.B, dtype=torch.int32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        mars.mars_kv_commit_batch_sync(inp.k_blk[0].to(DEV), inp.v_blk[0].to(DEV), n.to(DEV),
                                       sl, inp.block_table.to(DEV), kp, vp, slots, st)
        torch.cuda.synchronize()
        rk, rv, rl, rs = oracle.kv_commit_batch_sync(
            f64(inp.k_blk[0]), f64(inp.v_blk[0]), n.numpy(), inp.prefix_lens.numpy(),
            inp.block_table.numpy(), f64(inp.k_pool), f64(inp.v_pool), cfg.page_size)
        assert int(st.item()) == 0
        np.testing.assert_array_equal(sl.cpu().numpy(), rl)
        np.testing.assert_array_equal(slots.cpu().numpy(), rs)
        np.testing.assert_array_equal(f64(kp.cpu()), rk)
        np.testing.assert_array_equal(f64(vp.cpu()), rv)


# ------------------------------------------------------------- dual-stream training loss

LOSS_TOL = 2e-4      # fp32 logits of bf16 inputs: |error of lse - l_y| well below 1e-4


def run_ce(h, w, y, batch, L, row_ce=True):
    loss = torch.empty(3, dtype=torch.float32, device=DEV)
    ce = torch.empty(batch * 2 * L, dtype=torch.float32, device=DEV) if row_ce else None
    ws = _ws(mars.mars_workspace_bytes(mars.OP_CE_LOSS, batch, 1, vocab=w.shape[0], max_len=L))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mars.mars_dual_stream_ce_loss(h, w, y, batch, L, loss, ws, row_ce=ce, status=st)
    torch.cuda.synchronize()
    return loss.cpu().numpy(), (ce.cpu().numpy() if row_ce else None), int(st.item())


@pytest.mark.parametrize("batch,L,H,V", [(2, 96, 256, 1000), (1, 200, 64, 7), (3, 1, 128, 300)])
def test_ce_loss_small(batch, L, H, V):
    cfg = W.CELossConfig("t", batch, L, H, V)
    x = W.make_ce_inputs(cfg, seed=L + V)
    y = x["targets"].clone()
    y[::5] = -1                                   # rows left out of both streams
    loss, ce, st = run_ce(x["h"].to(DEV), x["w"].to(DEV), y.to(DEV), batch, L)
    assert st == 0
    l_mask, l_ar, rce = oracle.ce_loss_dual(f64(x["h"]), f64(x["w"]), y.numpy(), batch, L)
    np.testing.assert_allclose(ce, rce, rtol=0, atol=LOSS_TOL)
    assert abs(loss[0] - l_mask) <= LOSS_TOL and abs(loss[1] - l_ar) <= LOSS_TOL
    assert abs(loss[2] - (l_mask + l_ar)) <= 2 * LOSS_TOL
    # the loss without the per-row output is the same bits
    loss2, _, _ = run_ce(x["h"].to(DEV), x["w"].to(DEV), y.to(DEV), batch, L, row_ce=False)
    np.testing.assert_array_equal(loss, loss2)


def test_ce_loss_bad_target_is_flagged_and_left_out():
    cfg = W.CELossConfig("t", 1, 16, 64, 100)
    x = W.make_ce_inputs(cfg, seed=3)
    y = x["targets"].clone()
    y[20] = 100                                   # == vocab: out of range
    loss, ce, st = run_ce(x["h"].to(DEV), x["w"].to(DEV), y.to(DEV), 1, 16)
    assert st & mars.ST_BADTARGET
    y[20] = -1
    l_mask, l_ar, _ = oracle.ce_loss_dual(f64(x["h"]), f64(x["w"]), y.numpy(), 1, 16)
    assert ce[20] == 0.0 and abs(loss[0] - l_mask) <= LOSS_TOL and abs(loss[1] - l_ar) <= LOSS_TOL


def test_ce_loss_7b_shapes_sampled_rows():
    cfg = W.CELossConfig("t7", 1, 512, 3584, 152064)
    x = W.make_ce_inputs(cfg, seed=0, device=DEV)
    loss, ce, st = run_ce(x["h"], x["w"], x["targets"], 1, 512)
    assert st == 0
    rows = sorted({0, 1, 255, 510, 511, 512, 513, 700, 1023,
                   *np.random.default_rng(2).integers(0, 1024, 20).tolist()})
    y = x["targets"].cpu().numpy()
    h = f64(x["h"][rows])
    _, _, rce = oracle.ce_loss_dual(h, f64(x["w"]), y[rows], len(rows), 1)
    # rows were regrouped, so only the per-row values are compared here
    np.testing.assert_allclose(ce[rows], rce, rtol=0, atol=LOSS_TOL)
    # the means are those of the per-row values (in float64)
    pos = np.arange(1024) % 1024
    ok = y >= 0
    assert abs(loss[0] - ce[ok & (pos >= 512)].astype(np.float64).mean()) < 1e-5
    assert abs(loss[1] - ce[ok & (pos < 512)].astype(np.float64).mean()) < 1e-5


def run_ce_grad(h, w, y, batch, L):
    rows = batch * 2 * L
    loss = torch.empty(3, dtype=torch.float32, device=DEV)
    lse = torch.empty(rows, dtype=torch.float32, device=DEV)
    ws = _ws(mars.mars_workspace_bytes(mars.OP_CE_LOSS, batch, 1, vocab=w.shape[0], max_len=L))
    mars.mars_dual_stream_ce_loss(h, w, y, batch, L, loss, ws, row_lse=lse)
    wg = _ws(mars.mars_workspace_bytes(mars.OP_CE_LOSS_GRAD, batch, 1, vocab=w.shape[0],
                                       max_len=L))
    dh = torch.empty(rows, h.shape[1], dtype=torch.float32, device=DEV)
    dw = torch.empty(w.shape, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mars.mars_dual_stream_ce_loss_grad(h, w, y, lse, batch, L, wg, dh, dw, st)
    torch.cuda.synchronize()
    return dh.cpu().numpy(), dw.cpu().numpy(), lse.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("batch,L,H,V", [(2, 96, 256, 1000), (1, 130, 64, 264), (3, 1, 128, 296)])
def test_ce_loss_grad_small(batch, L, H, V):
    """dh and dW element by element within the error bound of bf16 dlogits (every row,
    every word), and the forward's per-row log-sum-exp."""
    cfg = W.CELossConfig("g", batch, L, H, V)
    x = W.make_ce_inputs(cfg, seed=L * 3 + V)
    y = x["targets"].clone()
    y[::7] = -1
    dh, dw, lse, st = run_ce_grad(x["h"].to(DEV), x["w"].to(DEV), y.to(DEV), batch, L)
    assert st == 0
    h, w = f64(x["h"]), f64(x["w"])
    yy = y.numpy()
    rdh, rdw, g = oracle.ce_loss_dual_grad(h, w, yy, batch, L)
    # |softmax| / N per entry: g plus the one-hot term of rows with a target
    ok = yy >= 0
    pos = np.arange(len(yy)) % (2 * L)
    inv_n = np.where(pos < L, 1.0 / max(int((ok & (pos < L)).sum()), 1),
                     1.0 / max(int((ok & (pos >= L)).sum()), 1)) * ok
    p = g.copy()
    p[np.flatnonzero(ok), yy[ok]] += inv_n[ok]
    up = logit_rel_error(h, w)[:, None] * np.abs(p)
    ag, g2 = np.abs(g), g * g
    assert_within_bound(dh, rdh, product_error_bound(ag @ np.abs(w), g2 @ (w * w), V,
                                                     up @ np.abs(w)), "dh")
    assert_within_bound(dw, rdw, product_error_bound(ag.T @ np.abs(h), g2.T @ (h * h),
                                                     len(yy), up.T @ np.abs(h)), "dW")
    logits = h @ w.T
    m = logits.max(axis=1)
    rlse = m + np.log(np.exp(logits - m[:, None]).sum(axis=1))
    np.testing.assert_allclose(lse, rlse, rtol=0, atol=LOSS_TOL)


def test_ce_loss_grad_7b_shapes_sampled():
    """Hidden 3584, vocabulary 152064, 512 rows: dh on sampled rows, dW on sampled words,
    element by element within the error bound (the reference still needs every row's
    log-sum-exp, computed here in chunks)."""
    cfg = W.CELossConfig("g7", 1, 256, 3584, 152064)
    x = W.make_ce_inputs(cfg, seed=1, device=DEV)
    dh, dw, lse, st = run_ce_grad(x["h"], x["w"], x["targets"], 1, 256)
    assert st == 0
    h, w = f64(x["h"]), f64(x["w"])
    y = x["targets"].cpu().numpy()
    rows = sorted({0, 1, 255, 256, 257, 511, *np.random.default_rng(5).integers(0, 512, 10).tolist()})
    words = sorted({0, 1, 152063, *y[y >= 0][:6].tolist(),
                    *np.random.default_rng(6).integers(0, 152064, 6).tolist()})
    # exact log-sum-exp of every row (chunked over the vocabulary), then the gradient
    lse_ref = np.empty(512)
    for r0 in range(0, 512, 64):
        lg = h[r0:r0 + 64] @ w.T
        m = lg.max(axis=1)
        lse_ref[r0:r0 + 64] = m + np.log(np.exp(lg - m[:, None]).sum(axis=1))
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=LOSS_TOL)
    valid = y >= 0
    pos = np.arange(512) % 512
    scale = np.where(pos < 256, 1.0 / (valid & (pos < 256)).sum(), 1.0 / (valid & (pos >= 256)).sum())
    scale = np.where(valid, scale, 0.0)
    rel = logit_rel_error(h, w)

    # dh on the sampled rows: dlogits of those rows over the whole vocabulary
    p = np.exp(h[rows] @ w.T - lse_ref[rows][:, None]) * scale[rows][:, None]
    g = p.copy()
    for i, r in enumerate(rows):
        if valid[r]:
            g[i, y[r]] -= scale[r]
    rdh = g @ w
    bnd = product_error_bound(np.abs(g) @ np.abs(w), (g * g) @ (w * w), w.shape[0],
                              (rel[rows][:, None] * p) @ np.abs(w))
    assert_within_bound(dh[rows], rdh, bnd, "dh 7B")
    del p, g
    # dW on the sampled words: dlogits of every row at those words
    p = np.exp(h @ w[words].T - lse_ref[:, None]) * scale[:, None]   # [512, words]
    g = p.copy()
    for j, v in enumerate(words):
        g[(y == v) & valid, j] -= scale[(y == v) & valid]
    rdw = g.T @ h
    bnd = product_error_bound(np.abs(g).T @ np.abs(h), (g * g).T @ (h * h), 512,
                              (rel[:, None] * p).T @ np.abs(h))
    assert_within_bound(dw[words], rdw, bnd, "dW 7B")


# -------------------------------------------------------------- whole decode step chain

def test_tiny_decode_step_end_to_end():
    """Config 1: attention, head + acceptance, commit, all against the oracle, for two
    steps (the second step runs on the committed cache of the first)."""
    cfg = W.TINY_DECODE
    inp = W.make_decode_inputs(cfg, seed=0, steps=2, extra_pages=2)
    kp, vp = inp.k_pool.to(DEV), inp.v_pool.to(DEV)
    bt = inp.block_table.to(DEV)
    sl = inp.prefix_lens.to(DEV)
    w = inp.w.to(DEV)
    rk, rv, rl = f64(inp.k_pool), f64(inp.v_pool), inp.prefix_lens.numpy().astype(np.int64)
    for step in range(2):
        tau = cfg.tau_at(step) if step == 0 else 0.0     # step 1 forces a multi-token commit
        o = torch.empty(cfg.batch, cfg.B, cfg.hq, cfg.d, dtype=torch.float32, device=DEV)
        ws = _ws(mars.mars_workspace_bytes(mars.OP_DECODE_ATTN, cfg.batch, cfg.B, cfg.hq,
                                           cfg.hkv, cfg.d, max_len=64))
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        mars.mars_decode_attn(inp.q[step].to(DEV), inp.k_blk[step].to(DEV),
                              inp.v_blk[step].to(DEV), kp, vp, bt, sl, 64, o, ws, st)
        ref_o = oracle.decode_attn(f64(inp.q[step]), f64(inp.k_blk[step]),
                                   f64(inp.v_blk[step]), rk, rv, inp.block_table.numpy(), rl,
                                   cfg.page_size)
        tok, p, n = run_head(inp.h[step].to(DEV), w, cfg.batch, cfg.B, tau)
        rt, rp, rn, gap = oracle.head_accept(f64(inp.h[step]), f64(inp.w), cfg.batch, cfg.B,
                                             tau)
        assert_attn_close(o.cpu().numpy(), ref_o)
        compare_head(tok, p, n, rt, rp, rn, gap, tau)
        slots = torch.empty(cfg.batch, cfg.B, dtype=torch.int32, device=DEV)
        mars.mars_kv_commit(inp.k_blk[step].to(DEV), inp.v_blk[step].to(DEV),
                            torch.from_numpy(n).to(DEV), sl, bt, kp, vp, slots, st)
        rk, rv, rl, rs = oracle.kv_commit(f64(inp.k_blk[step]), f64(inp.v_blk[step]), rn, rl,
                                          inp.block_table.numpy(), rk, rv, cfg.page_size)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        np.testing.assert_array_equal(slots.cpu().numpy(), rs)
        np.testing.assert_array_equal(sl.cpu().numpy(), rl)
    np.testing.assert_array_equal(f64(kp.cpu()), rk)


# ------------------------------------------------------------------ bounded waits

def test_wait_limit_reports_timeout_and_context_stays_usable():
    """A kernel waiting on an mbarrier that nothing completes gives up after the wait limit,
    reports ST_TIMEOUT in the status word and exits; the next call runs normally."""
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    mars.mars_check_wait_timeout(status)
    torch.cuda.synchronize()
    assert int(status.item()) == mars.ST_TIMEOUT
    cfg = W.DualStreamConfig("after", 1, 130, 16, 2, 1, 64)
    x = W.make_dual_stream_inputs(cfg, seed=2)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = torch.empty(x["q"].shape, dtype=torch.float32, device=DEV)
    mars.mars_attn_dual_stream(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), o, L=cfg.L,
                               B=cfg.B, status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    ref = oracle.attn_dual_stream(f64(x["q"]), f64(x["k"]), f64(x["v"]), cfg.L, cfg.B)
    assert_attn_close(o.cpu().numpy(), ref)
