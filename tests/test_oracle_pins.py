"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a hand enumeration of
eq. M, the AR-signal percentages printed on the pages, a library routine (torch SDPA,
softmax, argmax) in fp64, a brute-force scalar loop, or an identity between the two
attention forms. The last section plants plausible mistakes in the oracle and checks
that some pin catches each of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import mars_oracle
from block_masked_token_gb300 import workloads as W
from conftest import golden_lines


def _read_mask(name):
    lines = golden_lines(name)
    L = int(lines[0].split()[1])
    B = int(lines[1].split()[1])
    rows = [[c == "1" for c in ln.strip()] for ln in lines[2:]]
    return L, B, np.array(rows, dtype=bool)


# ------------------------------------------------------------------ mask M (Key design 1)

@pytest.mark.parametrize("name", ["mask_M_L4_B2.txt", "mask_M_L3_B2.txt",
                                  "mask_M_L4_B4.txt", "mask_M_L3_B1.txt"])
def test_mask_matches_hand_enumeration(name):
    L, B, want = _read_mask(name)
    assert want.shape == (2 * L, 2 * L)
    np.testing.assert_array_equal(oracle.mask_M(L, B), want)


def test_beta_is_ceil():
    for B in range(1, 9):
        for t in range(1, 40):
            assert oracle.beta(t, B) == math.ceil(t / B)


@pytest.mark.parametrize("L", list(range(1, 17)))
def test_mask_invariants(L):
    for B in range(1, L + 1):
        vis = oracle.mask_M(L, B)
        # every row sees itself, so no softmax row is empty
        assert vis.diagonal().all()
        # the clean stream never sees the masked stream, and is plainly causal
        assert not vis[:L, L:].any()
        np.testing.assert_array_equal(vis[:L, :L], np.tril(np.ones((L, L), bool)))
        # nothing sees a later position in its own stream
        assert not np.triu(vis[L:, L:], 1).any()
        # masked row t sees t keys: t - B*(beta(t)-1) in its block plus B*(beta(t)-1)
        # clean ones; the total is L(L+1)/2 (clean) + L(L+1)/2 (masked) = L(L+1)
        assert vis.sum() == L * (L + 1)
        if B == L:
            assert not vis[L:, :L].any()
        if B == 1:
            for t in range(1, L + 1):
                row = vis[L + t - 1]
                assert row[:t - 1].all() and not row[t - 1:L].any()
                assert row[L + t - 1] and row[L:].sum() == 1


def test_mask_rows_equals_full_matrix():
    for L, B in [(7, 3), (16, 4), (9, 9), (33, 5)]:
        rows = np.arange(2 * L)
        np.testing.assert_array_equal(oracle.mask_rows(L, B, rows), oracle.mask_M(L, B))


# --------------------------------------------------------- AR-signal fraction (Key design 2)

def test_ar_signal_fraction_printed_values():
    for line in golden_lines("r_ar_printed.txt"):
        B, mode, pct, dec = line.split()
        B, pct, dec = int(B), float(pct), int(dec)
        L = 64                                     # any L divisible by B
        got = 100.0 * oracle.ar_signal_fraction(L, B, combined=(mode == "combined"))
        assert abs(got - pct) <= 0.5 * 10.0 ** (-dec) + 1e-12, (B, mode, got, pct)


def test_ar_signal_fraction_closed_form():
    for B in (1, 2, 4, 8, 16):
        L = 4 * B
        assert oracle.ar_signal_fraction(L, B, False) == pytest.approx(1.0 / B)
        assert oracle.ar_signal_fraction(L, B, True) == pytest.approx((1 + 1.0 / B) / 2)
        assert oracle.ar_signal_fraction(L, B, True) > 0.5


# ------------------------------------------------------------- dual-stream attention

def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64).numpy()


def _sdpa(q, k, v, mask=None, causal=False):
    # q [n, D], k/v [n, D] for one head; fp64 library routine on CPU
    Q = torch.from_numpy(q)[None, None]
    K = torch.from_numpy(k)[None, None]
    V = torch.from_numpy(v)[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(
        Q, K, V, attn_mask=m, is_causal=causal)[0, 0].numpy()


@pytest.mark.parametrize("L,B,hq,hkv,D", [(5, 2, 2, 1, 8), (16, 4, 4, 2, 16),
                                          (13, 16, 3, 3, 8), (24, 3, 6, 2, 32)])
def test_dual_stream_against_sdpa(L, B, hq, hkv, D):
    b = 2
    q = _rand((b, 2 * L, hq, D), 1)
    k = _rand((b, 2 * L, hkv, D), 2)
    v = _rand((b, 2 * L, hkv, D), 3)
    out = oracle.attn_dual_stream(q, k, v, L, B)
    vis = oracle.mask_M(L, B)
    g = hq // hkv
    for bi in range(b):
        for h in range(hq):
            hk = h // g
            # clean half: plain causal attention over the clean stream
            ref_clean = _sdpa(q[bi, :L, h], k[bi, :L, hk], v[bi, :L, hk], causal=True)
            np.testing.assert_allclose(out[bi, :L, h], ref_clean, rtol=1e-12, atol=1e-12)
            ref = _sdpa(q[bi, :, h], k[bi, :, hk], v[bi, :, hk], mask=vis)
            np.testing.assert_allclose(out[bi, :, h], ref, rtol=1e-12, atol=1e-12)


def _brute_attention_row(qrow, K, V, visible, scale):
    scores = []
    for j in range(len(K)):
        if visible[j]:
            scores.append((j, scale * sum(a * b for a, b in zip(qrow, K[j]))))
    m = max(s for _, s in scores)
    w = [(j, math.exp(s - m)) for j, s in scores]
    tot = sum(x for _, x in w)
    D = len(V[0])
    return [sum(x * V[j][d] for j, x in w) / tot for d in range(D)]


def test_dual_stream_bruteforce_hand_mask():
    L, B, vis = _read_mask("mask_M_L4_B2.txt")
    D = 4
    q = _rand((1, 2 * L, 2, D), 4)
    k = _rand((1, 2 * L, 1, D), 5)
    v = _rand((1, 2 * L, 1, D), 6)
    out = oracle.attn_dual_stream(q, k, v, L, B, scale=0.7)
    for h in range(2):
        for i in range(2 * L):
            ref = _brute_attention_row(q[0, i, h].tolist(), k[0, :, 0].tolist(),
                                       v[0, :, 0].tolist(), vis[i], 0.7)
            np.testing.assert_allclose(out[0, i, h], ref, rtol=1e-12, atol=1e-13)


def test_dual_stream_row_sampling_matches_full():
    L, B = 20, 4
    q = _rand((2, 2 * L, 4, 8), 7)
    k = _rand((2, 2 * L, 2, 8), 8)
    v = _rand((2, 2 * L, 2, 8), 9)
    full = oracle.attn_dual_stream(q, k, v, L, B)
    rows = [0, 3, 19, 20, 27, 39]
    part = oracle.attn_dual_stream(q, k, v, L, B, rows=rows, heads=[1, 3], batches=[1])
    np.testing.assert_allclose(part[1][:, [1, 3]], full[1][rows][:, [1, 3]], rtol=0, atol=0)


def test_dual_stream_lse_zero_queries_counts_visible_keys():
    """With q = 0 every visible score is 0, so the denominator is the number of visible
    keys: t + 1 for row t of either stream (clean row t sees keys 0..t; masked row t sees
    the clean keys before its block start bs and its own block's keys bs..t)."""
    L, B = 23, 5
    q = np.zeros((1, 2 * L, 2, 8))
    k = _rand((1, 2 * L, 1, 8), 3)
    lse = oracle.attn_dual_stream_lse(q, k, L, B)
    t = np.arange(L)
    want = np.log2(np.concatenate([t + 1, t + 1]).astype(np.float64))
    np.testing.assert_allclose(lse[0, 0], want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 1], want, rtol=0, atol=1e-12)


def test_dual_stream_lse_reproduces_attention_probabilities():
    """The probabilities attn_dual_stream applies are exp2(scale log2(e) s - lse): with V
    the identity (one value column per key), O itself is the probability matrix."""
    L, B = 9, 2
    n = 2 * L
    q = _rand((1, n, 2, n), 11) * 0.5                # head dim 2L, the width of V = I
    k = _rand((1, n, 1, n), 12)
    v = np.eye(n)[None, :, None, :]                  # [1, 2L, 1, 2L]
    o = oracle.attn_dual_stream(q, k, v, L, B, scale=0.4)
    lse = oracle.attn_dual_stream_lse(q, k, L, B, scale=0.4)
    vis = oracle.mask_rows(L, B, np.arange(n))
    for h in range(2):
        s = 0.4 * q[0, :, h] @ k[0, :, 0].T
        p = np.where(vis, np.exp2(s / math.log(2.0) - lse[0, h][:, None]), 0.0)
        np.testing.assert_allclose(o[0, :, h], p, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------- decode form

def _paged_from_logical(logical, page_size, perm, Hkv, D):
    """Scatter logical rows [P, Hkv, D] into the pages listed in perm (test-side layout);
    unused slots keep random values. Returns (pool, block-table row)."""
    pool = _rand((max(perm) + 2, Hkv, page_size, D), 99)
    for t in range(len(logical)):
        pool[perm[t // page_size], :, t % page_size, :] = logical[t]
    return pool, np.array(list(perm) + [-1, -1])


@pytest.mark.parametrize("B,P,ps", [(4, 8, 4), (2, 6, 16), (8, 16, 16), (1, 5, 4), (3, 9, 2)])
def test_decode_equals_masked_stream_row(B, P, ps):
    """A decode query at a block-aligned prefix P equals the masked-stream row L + P + k
    of the dual-stream form, with the prefix as the clean stream and the block keys as the
    masked stream (Key design 1 vs Key design 3/4: same visibility)."""
    assert P % B == 0
    Hq, Hkv, D = 4, 2, 8
    L = P + B + 3                           # extra positions after the block are masked
    q2 = _rand((1, 2 * L, Hq, D), 10)
    k2 = _rand((1, 2 * L, Hkv, D), 11)
    v2 = _rand((1, 2 * L, Hkv, D), 12)
    dual = oracle.attn_dual_stream(q2, k2, v2, L, B)
    perm = list(np.random.default_rng(0).permutation(P // ps + 3))
    kpool, bt = _paged_from_logical(k2[0, :P], ps, perm, Hkv, D)
    vpool, _ = _paged_from_logical(v2[0, :P], ps, perm, Hkv, D)
    qd = q2[:, L + P:L + P + B]
    kb = k2[:, L + P:L + P + B]
    vb = v2[:, L + P:L + P + B]
    dec = oracle.decode_attn(qd, kb, vb, kpool, vpool, bt[None, :], np.array([P]), ps)
    np.testing.assert_allclose(dec[0], dual[0, L + P:L + P + B], rtol=1e-12, atol=1e-12)


def test_decode_bruteforce():
    B, Hq, Hkv, D, ps = 3, 2, 1, 4, 4
    lens = [5, 0, 9]
    b = len(lens)
    q = _rand((b, B, Hq, D), 20)
    kb = _rand((b, B, Hkv, D), 21)
    vb = _rand((b, B, Hkv, D), 22)
    kpool = _rand((12, Hkv, ps, D), 23)
    vpool = _rand((12, Hkv, ps, D), 24)
    bt = np.array([[3, 7, -1, -1], [1, -1, -1, -1], [11, 0, 5, -1]])
    out = oracle.decode_attn(q, kb, vb, kpool, vpool, bt, np.array(lens), ps, scale=0.5)
    for s in range(b):
        keys = [kpool[bt[s][t // ps], 0, t % ps].tolist() for t in range(lens[s])]
        vals = [vpool[bt[s][t // ps], 0, t % ps].tolist() for t in range(lens[s])]
        keys += kb[s, :, 0].tolist()
        vals += vb[s, :, 0].tolist()
        for kq in range(B):
            visible = [True] * lens[s] + [i <= kq for i in range(B)]
            for h in range(Hq):
                ref = _brute_attention_row(q[s, kq, h].tolist(), keys, vals, visible, 0.5)
                np.testing.assert_allclose(out[s, kq, h], ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------- head, max-prob, acceptance

def test_maxprob_argmax_against_torch():
    g = torch.Generator().manual_seed(3)
    logits = (torch.randn(64, 1000, generator=g, dtype=torch.float64) * 4).numpy()
    logits[5, 10] = logits[5, 900] = logits[5].max() + 1.0       # exact tie
    tok, p, gap = oracle.maxprob_argmax(logits)
    T = torch.from_numpy(logits)
    np.testing.assert_allclose(p, torch.softmax(T, dim=1).max(dim=1).values.numpy(),
                               rtol=1e-13)
    first_max = [int(np.flatnonzero(r == r.max())[0]) for r in logits]
    np.testing.assert_array_equal(tok, first_max)
    no_tie = np.arange(64) != 5
    np.testing.assert_array_equal(tok[no_tie], T.argmax(dim=1).numpy()[no_tie])
    assert tok[5] == 10 and gap[5] == 0.0
    assert (p > 1.0 / 1000).all() and (p <= 1.0).all() and (gap >= 0).all()


def test_one_word_vocabulary():
    """V = 1: softmax is 1, so p = 1 >= tau for any tau <= 1 and the whole block is
    accepted; there is no second logit, so no tie."""
    h = _rand((6, 8), 90)
    w = _rand((1, 8), 91)
    tok, p, n, gap = oracle.head_accept(h, w, 2, 3, 1.0)
    assert (tok == 0).all() and (p == 1.0).all() and (n == 3).all() and np.isinf(gap).all()


def test_head_logits_chunked_equals_matmul():
    h = _rand((6, 40), 30)
    w = _rand((1000, 40), 31)
    np.testing.assert_allclose(oracle.head_logits(h, w, chunk=97), h @ w.T, rtol=1e-11, atol=1e-12)


def test_acceptance_golden_cases():
    for line in golden_lines("acceptance_cases.txt"):
        tau, ps, n = [x.strip() for x in line.split("|")]
        probs = [float(x) for x in ps.split()]
        assert oracle.accept_count(probs, float(tau)) == int(n), line


def test_acceptance_properties_on_seeded_inputs():
    cfg = W.TINY_DECODE
    inp = W.make_decode_inputs(cfg, seed=0)
    h = W.to_f64(inp.h[0])
    w = W.to_f64(inp.w)
    tok, p, n1, gap = oracle.head_accept(h, w, cfg.batch, cfg.B, 1.0)
    assert (n1 == 1).all()                                  # tau = 1.0: plain AR
    assert (p < 1.0).all()
    _, _, n0, _ = oracle.head_accept(h, w, cfg.batch, cfg.B, 0.0)
    assert (n0 == cfg.B).all()                              # tau = 0: the whole block
    _, _, nbig, _ = oracle.head_accept(h, w, cfg.batch, cfg.B, 1.5)
    assert (nbig == 1).all()
    prev = None
    for tau in np.linspace(0.0, 1.0, 41):
        n = np.array([oracle.accept_count(p[s], tau) for s in range(cfg.batch)])
        assert ((n >= 1) & (n <= cfg.B)).all()
        if prev is not None:
            assert (n <= prev).all()                        # N non-increasing in tau
        prev = n


def test_tau_one_gives_one_token_at_7b_vocab():
    """tau = 1.0 accepts exactly one token per step at the 7B vocabulary size, with the
    synthetic h/W distribution (log-uniform scales up to 8)."""
    g = torch.Generator().manual_seed(1)
    H, V, R = 64, 152064, 16
    s = torch.exp(math.log(0.5) + (math.log(8) - math.log(0.5)) * torch.rand(R, 1, generator=g))
    h = (torch.randn(R, H, generator=g) * s).to(torch.bfloat16).double().numpy()
    w = (torch.randn(V, H, generator=g) / math.sqrt(H)).to(torch.bfloat16).double().numpy()
    _, p, n, _ = oracle.head_accept(h, w, 2, 8, 1.0)
    assert (n == 1).all() and (p < 1).all()


def test_per_request_thresholds_golden_batch():
    """One batch whose sequences carry different thresholds reproduces the hand-derived N
    of every row. The max-probs are produced through the head itself: vocabulary 2, hidden
    1, W = [[0], [1]] and h = logit(p), so that softmax gives exactly p for token 1."""
    rows = [[x.strip() for x in ln.split("|")] for ln in golden_lines("per_request_tau_cases.txt")]
    taus = np.array([float(r[0]) for r in rows])
    probs = np.array([[float(x) for x in r[1].split()] for r in rows])
    want = np.array([int(r[2]) for r in rows])
    batch, B = probs.shape
    h = np.log(probs / (1.0 - probs)).reshape(batch * B, 1)
    w = np.array([[0.0], [1.0]])
    tok, p, n, _ = oracle.head_accept_per_request(h, w, batch, B, taus)
    np.testing.assert_allclose(p, probs, rtol=0, atol=1e-12)
    assert (tok == 1).all()
    np.testing.assert_array_equal(n, want)
    # a single threshold for the whole batch would not give these counts
    assert any((oracle.head_accept(h, w, batch, B, t)[2] != want).any() for t in taus)


def test_per_request_equal_thresholds_reduce_to_per_call():
    cfg = W.TINY_DECODE
    inp = W.make_decode_inputs(cfg, seed=0)
    h, w = W.to_f64(inp.h[0]), W.to_f64(inp.w)
    for tau in (0.0, 0.3, 0.9, 1.0):
        a = oracle.head_accept(h, w, cfg.batch, cfg.B, tau)
        b = oracle.head_accept_per_request(h, w, cfg.batch, cfg.B, [tau] * cfg.batch)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


# ------------------------------------------------------------------------- commit

def test_commit_golden_case():
    kv = dict(ln.split(None, 1) for ln in golden_lines("commit_case.txt"))
    ps = int(kv["page_size"])
    bt = np.array([[int(x) for x in kv["block_table"].split()]])
    sl = np.array([int(kv["seq_len"])])
    B = int(kv["B"])
    n = np.array([int(kv["N"])])
    Hkv, D = 2, 3
    kb = _rand((1, B, Hkv, D), 40)
    vb = _rand((1, B, Hkv, D), 41)
    kp = _rand((8, Hkv, ps, D), 42)
    vp = _rand((8, Hkv, ps, D), 43)
    kp2, vp2, sl2, slots = oracle.kv_commit(kb, vb, n, sl, bt, kp, vp, ps)
    np.testing.assert_array_equal(slots[0], [int(x) for x in kv["slots"].split()])
    assert sl2[0] == int(kv["new_seq_len"])
    for i, sl_ in enumerate(slots[0]):
        if sl_ >= 0:
            np.testing.assert_array_equal(kp2[sl_ // ps, :, sl_ % ps], kb[0, i])
            np.testing.assert_array_equal(vp2[sl_ // ps, :, sl_ % ps], vb[0, i])


def test_commit_properties():
    ps, Hkv, D, B = 4, 2, 5, 6
    lens = np.array([0, 3, 7, 12])
    n = np.array([6, 1, 4, 2])
    b = len(lens)
    bt = np.array([[0, 1, -1, -1, -1], [2, 3, -1, -1, -1], [4, 5, 6, -1, -1],
                   [7, 8, 9, 10, 11]])
    kb = _rand((b, B, Hkv, D), 50)
    vb = _rand((b, B, Hkv, D), 51)
    kp = _rand((13, Hkv, ps, D), 52)
    vp = _rand((13, Hkv, ps, D), 53)
    kp2, vp2, sl2, slots = oracle.kv_commit(kb, vb, n, lens, bt, kp, vp, ps)
    np.testing.assert_array_equal(sl2, lens + n)
    # page 12 is mapped to no sequence: untouched
    np.testing.assert_array_equal(kp2[12], kp[12])
    for s in range(b):
        P2 = int(sl2[s])
        got = oracle.gather_prefix(kp2, bt[s], P2, ps)
        old = oracle.gather_prefix(kp, bt[s], int(lens[s]), ps)
        np.testing.assert_array_equal(got[:lens[s]], old)        # prefix unchanged
        np.testing.assert_array_equal(got[lens[s]:], kb[s, :n[s]])
        assert (slots[s, n[s]:] == -1).all()


def test_commit_batch_sync_golden_case():
    kv = dict(ln.split(None, 1) for ln in golden_lines("commit_sync_case.txt"))
    ps, B = int(kv["page_size"]), int(kv["B"])
    bt = np.array([[int(x) for x in kv["block_table_0"].split()],
                   [int(x) for x in kv["block_table_1"].split()]])
    sl = np.array([int(x) for x in kv["seq_len"].split()])
    n = np.array([int(x) for x in kv["N"].split()])
    Hkv, D = 2, 3
    kb = _rand((2, B, Hkv, D), 60)
    vb = _rand((2, B, Hkv, D), 61)
    kp = _rand((8, Hkv, ps, D), 62)
    vp = _rand((8, Hkv, ps, D), 63)
    kp2, vp2, sl2, slots = oracle.kv_commit_batch_sync(kb, vb, n, sl, bt, kp, vp, ps)
    np.testing.assert_array_equal(slots[0], [int(x) for x in kv["slots_0"].split()])
    np.testing.assert_array_equal(slots[1], [int(x) for x in kv["slots_1"].split()])
    np.testing.assert_array_equal(sl2, [int(x) for x in kv["new_seq_len"].split()])
    for s in range(2):
        for i, sl_ in enumerate(slots[s]):
            if sl_ >= 0:
                np.testing.assert_array_equal(kp2[sl_ // ps, :, sl_ % ps], kb[s, i])
                np.testing.assert_array_equal(vp2[sl_ // ps, :, sl_ % ps], vb[s, i])


def test_commit_batch_sync_properties():
    """Every sequence advances by the same amount, the batch minimum; with equal counts it
    is the per-sequence commit."""
    ps, Hkv, D, B = 4, 2, 5, 6
    lens = np.array([0, 3, 7, 12])
    bt = np.array([[0, 1, -1, -1, -1], [2, 3, -1, -1, -1], [4, 5, 6, -1, -1],
                   [7, 8, 9, 10, 11]])
    kb, vb = _rand((4, B, Hkv, D), 70), _rand((4, B, Hkv, D), 71)
    kp, vp = _rand((13, Hkv, ps, D), 72), _rand((13, Hkv, ps, D), 73)
    n = np.array([6, 2, 4, 3])
    _, _, sl2, slots = oracle.kv_commit_batch_sync(kb, vb, n, lens, bt, kp, vp, ps)
    np.testing.assert_array_equal(sl2, lens + 2)
    assert ((slots >= 0).sum(axis=1) == 2).all()
    eq = np.array([3, 3, 3, 3])
    a = oracle.kv_commit_batch_sync(kb, vb, eq, lens, bt, kp, vp, ps)
    b = oracle.kv_commit(kb, vb, eq, lens, bt, kp, vp, ps)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def _block_case():
    lines = golden_lines("commit_block_case.txt")
    kv = {}
    calls, written, staged = [], [], []
    for ln in lines:
        if ln.startswith("call"):
            f = [x.split() for x in ln.split("|")]
            calls.append({"N": [int(x) for x in f[1]],
                          "slots": [[int(x) for x in f[2]], [int(x) for x in f[3]]],
                          "fill": [int(x) for x in f[4]], "seq_len": [int(x) for x in f[5]],
                          "flush": bool(int(f[6][0]))})
        elif ln.startswith("written"):
            written.append([int(x) for x in ln.split()[1:]])
        elif ln.startswith("staged"):
            staged.append([int(x) for x in ln.split()[1:]])
        else:
            k, v = ln.split(None, 1)
            kv[k] = v
    return kv, calls, written, staged


def test_commit_block_golden_case():
    kv, calls, written, staged = _block_case()
    ps, B, Bc = int(kv["page_size"]), int(kv["B"]), int(kv["B_cache"])
    bt = np.array([[int(x) for x in kv["block_table_0"].split()],
                   [int(x) for x in kv["block_table_1"].split()]])
    lens = np.array([int(x) for x in kv["seq_len"].split()])
    Hkv, D = 2, 3
    kp, vp = _rand((10, Hkv, ps, D), 64), _rand((10, Hkv, ps, D), 65)
    kp0 = kp.copy()
    ks, vs = np.zeros((2, Bc, Hkv, D)), np.zeros((2, Bc, Hkv, D))
    fill, flush = np.zeros(2, dtype=np.int64), False
    blocks = []
    for c, call in enumerate(calls):
        kb, vb = _rand((2, B, Hkv, D), 80 + c), _rand((2, B, Hkv, D), 90 + c)
        blocks.append((kb, vb))
        kp, vp, lens, fill, ks, vs, flush, slots = oracle.kv_commit_block(
            kb, vb, np.array(call["N"]), lens, fill, ks, vs, flush, bt, kp, vp, ps, Bc)
        np.testing.assert_array_equal(slots, call["slots"], err_msg=f"call {c + 1}")
        np.testing.assert_array_equal(fill, call["fill"], err_msg=f"call {c + 1}")
        np.testing.assert_array_equal(lens, call["seq_len"], err_msg=f"call {c + 1}")
        assert flush == call["flush"], f"call {c + 1}"
        if c < 3:                      # nothing reaches the pool before the block is full
            np.testing.assert_array_equal(kp, kp0)
    touched = set()
    for slot, c, s, row in written:
        np.testing.assert_array_equal(kp[slot // ps, :, slot % ps], blocks[c - 1][0][s, row])
        np.testing.assert_array_equal(vp[slot // ps, :, slot % ps], blocks[c - 1][1][s, row])
        touched.add(slot)
    for slot in range(10 * ps):
        if slot not in touched:
            np.testing.assert_array_equal(kp[slot // ps, :, slot % ps],
                                          kp0[slot // ps, :, slot % ps])
    for s, r, c, row in staged:
        np.testing.assert_array_equal(ks[s, r], blocks[c - 1][0][s, row])
        np.testing.assert_array_equal(vs[s, r], blocks[c - 1][1][s, row])


def test_commit_block_properties():
    """Over random accepted counts: the persistent lengths of all sequences advance
    together in whole blocks; the persisted rows followed by the buffered ones are the
    rows the per-sequence commit writes when each call's count is the number of rows the
    block could still take; and with every block filled by each call, each call writes
    the previous call's block."""
    rng = np.random.default_rng(3)
    ps, Hkv, D, B, Bc, b = 4, 1, 2, 5, 8, 3
    lens0 = np.array([2, 9, 4])
    npg = 12
    bt = np.array([np.arange(npg) + s * npg for s in range(b)])
    kp, vp = _rand((b * npg, Hkv, ps, D), 66), _rand((b * npg, Hkv, ps, D), 67)
    ks, vs = np.zeros((b, Bc, Hkv, D)), np.zeros((b, Bc, Hkv, D))
    lens, fill, flush = lens0.copy(), np.zeros(b, dtype=np.int64), False
    rk, rv, rl = kp.copy(), vp.copy(), lens0.copy()       # per-sequence commit reference
    for c in range(12):
        kb, vb = _rand((b, B, Hkv, D), 200 + c), _rand((b, B, Hkv, D), 300 + c)
        n = rng.integers(-1, B + 2, b)
        took = np.minimum(np.clip(n, 0, B), Bc - np.where(flush, 0, fill))
        kp, vp, lens, fill, ks, vs, flush, slots = oracle.kv_commit_block(
            kb, vb, n, lens, fill, ks, vs, flush, bt, kp, vp, ps, Bc)
        rk, rv, rl, rslots = oracle.kv_commit(kb, vb, took, rl, bt, rk, rv, ps)
        np.testing.assert_array_equal(slots, rslots)
        assert ((lens - lens0) % Bc == 0).all() and len(set((lens - lens0).tolist())) == 1
        np.testing.assert_array_equal(lens + fill, rl)
        for s in range(b):
            got = oracle.gather_prefix(kp, bt[s], int(lens[s]), ps)
            want = oracle.gather_prefix(rk, bt[s], int(lens[s]), ps)
            np.testing.assert_array_equal(got, want)
            pending = oracle.gather_prefix(rk, bt[s], int(rl[s]), ps)[int(lens[s]):]
            np.testing.assert_array_equal(ks[s, :fill[s]], pending)
    # B = B_cache and every count B: each call fills every block
    kb, vb = _rand((b, Bc, Hkv, D), 400), _rand((b, Bc, Hkv, D), 401)
    st = (kp, vp, lens0.copy(), np.zeros(b, dtype=np.int64), ks, vs, False)
    for c in range(3):
        kp2, vp2, l2, f2, ks2, vs2, fl2, _ = oracle.kv_commit_block(
            kb, vb, np.full(b, Bc), st[2], st[3], st[4], st[5], st[6], bt, st[0], st[1], ps, Bc)
        assert fl2 and (f2 == Bc).all()
        np.testing.assert_array_equal(l2, lens0 + Bc * c)
        st = (kp2, vp2, l2, f2, ks2, vs2, fl2)


def test_decode_staged_equals_decode_on_the_extended_prefix():
    """Attention over prefix + buffered block rows + block keys equals the plain decode
    attention over a prefix that the buffered rows extend (committed into the pool)."""
    b, B, Hq, Hkv, D, ps, Bc = 3, 4, 4, 2, 8, 4, 8
    lens = np.array([5, 0, 13])
    fill = np.array([3, 8, 0])
    npg = 8
    bt = np.array([np.arange(npg) + s * npg for s in range(b)])
    q = _rand((b, B, Hq, D), 500)
    kb, vb = _rand((b, B, Hkv, D), 501), _rand((b, B, Hkv, D), 502)
    kp, vp = _rand((b * npg, Hkv, ps, D), 503), _rand((b * npg, Hkv, ps, D), 504)
    ks, vs = _rand((b, Bc, Hkv, D), 505), _rand((b, Bc, Hkv, D), 506)
    got = oracle.decode_attn_staged(q, kb, vb, kp, vp, bt, lens, ks, vs, fill, ps)
    kp2, vp2, lens2, _ = oracle.kv_commit(ks, vs, fill, lens, bt, kp, vp, ps)
    want = oracle.decode_attn(q, kb, vb, kp2, vp2, bt, lens2, ps)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)


# --------------------------------------------------------------- dual-stream loss

def test_ce_loss_hand_worked_case():
    rows = [[x.strip() for x in ln.split("|")] for ln in golden_lines("ce_loss_case.txt")]
    y = np.array([int(r[1]) for r in rows])
    h = np.full((4, 1), math.log(2.0))
    w = np.array([[0.0], [1.0], [2.0]])
    l_mask, l_ar, ce = oracle.ce_loss_dual(h, w, y, 1, 2)
    for (row, tgt, frac), c in zip(rows, ce):
        if tgt.strip() == "-1":
            assert c == 0.0
        else:
            a, b = (float(v) for v in frac.split("/"))
            assert abs(c - math.log(a / b)) < 1e-14, (row, c)
    assert abs(l_ar - math.log(7.0)) < 1e-14
    assert abs(l_mask - math.log(49.0 / 8.0) / 2) < 1e-14


def test_ce_loss_uniform_logits_give_log_vocab():
    """W = 0 makes every logit equal, so every target costs exactly ln V."""
    V, H, b, L = 37, 8, 2, 5
    h = _rand((b * 2 * L, H), 80)
    y = np.random.default_rng(0).integers(0, V, b * 2 * L)
    l_mask, l_ar, ce = oracle.ce_loss_dual(h, np.zeros((V, H)), y, b, L)
    assert np.allclose(ce, math.log(V), rtol=0, atol=1e-14)
    assert abs(l_mask - math.log(V)) < 1e-14 and abs(l_ar - math.log(V)) < 1e-14


def test_ce_loss_against_torch_cross_entropy():
    V, H, b, L = 300, 24, 3, 7
    h = _rand((b * 2 * L, H), 81)
    w = _rand((V, H), 82)
    y = np.random.default_rng(1).integers(-1, V, b * 2 * L)
    l_mask, l_ar, ce = oracle.ce_loss_dual(h, w, y, b, L)
    logits = torch.from_numpy(h @ w.T)
    yt = torch.from_numpy(y)
    per = torch.nn.functional.cross_entropy(logits, yt, ignore_index=-1, reduction="none")
    np.testing.assert_allclose(ce, per.numpy(), rtol=1e-12, atol=1e-12)
    pos = np.arange(b * 2 * L) % (2 * L)
    for sel, got in (((pos < L), l_ar), ((pos >= L), l_mask)):
        ref = torch.nn.functional.cross_entropy(logits[torch.from_numpy(sel)],
                                                yt[torch.from_numpy(sel)], ignore_index=-1)
        assert abs(got - float(ref)) < 1e-12


def test_ce_loss_grad_matches_finite_differences():
    """Central differences of the oracle's own loss (a property of the mathematics, not of
    the gradient formula) match dh and dW entry by entry."""
    V, H, b, L = 11, 5, 2, 3
    h = _rand((b * 2 * L, H), 83)
    w = _rand((V, H), 84)
    y = np.random.default_rng(3).integers(-1, V, b * 2 * L)
    dh, dw, _ = oracle.ce_loss_dual_grad(h, w, y, b, L)
    eps = 1e-6

    def total(hh, ww):
        lm, la, _ = oracle.ce_loss_dual(hh, ww, y, b, L)
        return lm + la

    for (r, k) in [(0, 0), (3, 4), (7, 2), (11, 1)]:
        hp, hm = h.copy(), h.copy()
        hp[r, k] += eps
        hm[r, k] -= eps
        assert abs((total(hp, w) - total(hm, w)) / (2 * eps) - dh[r, k]) < 1e-7
    for (v, k) in [(0, 0), (5, 3), (10, 4)]:
        wp, wm = w.copy(), w.copy()
        wp[v, k] += eps
        wm[v, k] -= eps
        assert abs((total(h, wp) - total(h, wm)) / (2 * eps) - dw[v, k]) < 1e-7


def test_ce_loss_grad_against_torch_autograd():
    V, H, b, L = 40, 6, 2, 4
    h = _rand((b * 2 * L, H), 85)
    w = _rand((V, H), 86)
    y = np.random.default_rng(4).integers(-1, V, b * 2 * L)
    dh, dw, _ = oracle.ce_loss_dual_grad(h, w, y, b, L)
    ht = torch.tensor(h, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    yt = torch.tensor(y)
    logits = ht @ wt.T
    pos = torch.arange(b * 2 * L) % (2 * L)
    loss = (torch.nn.functional.cross_entropy(logits[pos >= L], yt[pos >= L], ignore_index=-1) +
            torch.nn.functional.cross_entropy(logits[pos < L], yt[pos < L], ignore_index=-1))
    loss.backward()
    np.testing.assert_allclose(dh, ht.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_dual_stream_grad_matches_finite_differences():
    """Central differences of <O, dO> computed by the forward oracle match dQ, dK, dV."""
    b, L, B, Hq, Hkv, D = 1, 5, 2, 4, 2, 3
    q = _rand((b, 2 * L, Hq, D), 87)
    k = _rand((b, 2 * L, Hkv, D), 88)
    v = _rand((b, 2 * L, Hkv, D), 89)
    do = _rand((b, 2 * L, Hq, D), 90)
    dq, dk, dv = oracle.attn_dual_stream_grad(q, k, v, do, L, B)
    eps = 1e-6

    def f(qq, kk, vv):
        return float((oracle.attn_dual_stream(qq, kk, vv, L, B) * do).sum())

    for arr, grad, idx in ((q, dq, [(0, 0, 0, 0), (0, 7, 3, 2), (0, 9, 1, 1)]),
                           (k, dk, [(0, 1, 0, 0), (0, 6, 1, 2), (0, 9, 1, 1)]),
                           (v, dv, [(0, 0, 0, 1), (0, 5, 1, 0), (0, 8, 0, 2)])):
        for ix in idx:
            p_, m_ = arr.copy(), arr.copy()
            p_[ix] += eps
            m_[ix] -= eps
            args_p = [p_ if a is arr else a for a in (q, k, v)]
            args_m = [m_ if a is arr else a for a in (q, k, v)]
            fd = (f(*args_p) - f(*args_m)) / (2 * eps)
            assert abs(fd - grad[ix]) < 1e-7, (ix, fd, grad[ix])


def test_dual_stream_grad_against_torch_autograd():
    b, L, B, Hq, Hkv, D = 2, 6, 4, 4, 2, 8
    q = _rand((b, 2 * L, Hq, D), 91)
    k = _rand((b, 2 * L, Hkv, D), 92)
    v = _rand((b, 2 * L, Hkv, D), 93)
    do = _rand((b, 2 * L, Hq, D), 94)
    dq, dk, dv = oracle.attn_dual_stream_grad(q, k, v, do, L, B)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    mask = torch.tensor(oracle.mask_M(L, B))
    rep = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        qt.transpose(1, 2), kt.repeat_interleave(rep, dim=2).transpose(1, 2),
        vt.repeat_interleave(rep, dim=2).transpose(1, 2), attn_mask=mask).transpose(1, 2)
    (o * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_dual_stream_grad_parts_identities():
    """The gradient's intermediates obey what the mathematics fixes: P is the forward
    oracle's attention (rows sum to 1, zero wherever M hides the key, P V = O), D equals
    rowsum(dO * O) for that O, and every row of dS sums to 0."""
    b, L, B, Hq, Hkv, D = 2, 7, 3, 4, 2, 5
    q = _rand((b, 2 * L, Hq, D), 95)
    k = _rand((b, 2 * L, Hkv, D), 96)
    v = _rand((b, 2 * L, Hkv, D), 97)
    do = _rand((b, 2 * L, Hq, D), 98)
    o = oracle.attn_dual_stream(q, k, v, L, B)
    vis = oracle.mask_M(L, B)
    seen = 0
    for bi, h, hk, P, dP, Dr, dS in oracle.attn_dual_stream_grad_parts(q, k, v, do, L, B):
        assert hk == h // (Hq // Hkv)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-13)
        assert (P[~vis] == 0).all() and (P[vis] > 0).all()
        np.testing.assert_allclose(P @ v[bi, :, hk], o[bi, :, h], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dP, do[bi, :, h] @ v[bi, :, hk].T, rtol=0, atol=1e-12)
        np.testing.assert_allclose(Dr[:, 0], (do[bi, :, h] * o[bi, :, h]).sum(axis=1),
                                   rtol=0, atol=1e-12)
        np.testing.assert_allclose(dS.sum(axis=1), 0.0, rtol=0, atol=1e-12)
        seen += 1
    assert seen == b * Hq


# ------------------------------------------- planted mistakes: each must fail some pin

def test_planted_floor_block_index_is_caught(monkeypatch):
    monkeypatch.setattr(mars_oracle, "beta", lambda t, B: np.asarray(t) // B)
    L, B, want = _read_mask("mask_M_L4_B2.txt")
    assert not np.array_equal(mars_oracle.mask_M(L, B), want)


def test_planted_inclusive_cross_stream_is_caught(monkeypatch):
    real = mars_oracle.mask_M

    def wrong(L, B):          # case 3 with <= instead of <: a row sees its own clean block
        vis = real(L, B)
        i = np.arange(1, 2 * L + 1)[:, None]
        j = np.arange(1, 2 * L + 1)[None, :]
        bi = mars_oracle.beta(np.maximum(i - L, 1), B)
        return vis | ((i > L) & (j <= L) & (mars_oracle.beta(j, B) == bi))
    monkeypatch.setattr(mars_oracle, "mask_M", wrong)
    L, B, want = _read_mask("mask_M_L4_B2.txt")
    assert not np.array_equal(mars_oracle.mask_M(L, B), want)
    assert abs(100 * mars_oracle.ar_signal_fraction(64, 4, True) - 62.5) > 0.05


def test_planted_transposed_softmax_is_caught(monkeypatch):
    def wrong(S, vis):
        S = np.where(vis, S, -np.inf)
        P = np.exp(S - S.max(axis=0, keepdims=True))
        return P / P.sum(axis=0, keepdims=True)
    monkeypatch.setattr(mars_oracle, "_masked_softmax_rows", wrong)
    with pytest.raises(AssertionError):
        test_dual_stream_against_sdpa(5, 2, 2, 1, 8)


def test_planted_strict_threshold_is_caught(monkeypatch):
    def wrong(row, tau):
        t = float(np.float32(tau))
        n = 0
        for p in row:
            if p > t:
                n += 1
            else:
                break
        return max(1, n)
    monkeypatch.setattr(oracle, "accept_count", wrong)
    with pytest.raises(AssertionError):
        test_acceptance_golden_cases()


def test_planted_swapped_page_slot_is_caught(monkeypatch):
    # (a slot permutation inside a page would not be caught by attention, which is
    # order-invariant over the prefix; the commit pins cover slot order)
    def wrong(pool, row, P, ps):         # page and slot indices swapped
        out = np.empty((P, pool.shape[1], pool.shape[3]))
        for t in range(P):
            out[t] = pool[int(row[t % ps]), :, t // ps, :]
        return out
    monkeypatch.setattr(mars_oracle, "gather_prefix", wrong)
    with pytest.raises(AssertionError):
        test_decode_equals_masked_stream_row(4, 8, 4)


def _grad_with(mistake):
    """The oracle's dual-stream gradient with one planted mistake (the arithmetic of
    attn_dual_stream_grad otherwise)."""
    def grad(q, k, v, do, L, B, scale=None):
        b, n, Hq, D = q.shape
        g = Hq // k.shape[2]
        scale = 1.0 / math.sqrt(D) if scale is None else scale
        vis = mars_oracle.mask_M(L, B)
        dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
        for bi in range(b):
            for h in range(Hq):
                hk = h // g
                Q, K, V, dO = q[bi, :, h], k[bi, :, hk], v[bi, :, hk], do[bi, :, h]
                P = mars_oracle._masked_softmax_rows(scale * (Q @ K.T), vis)
                dP = dO @ V.T
                if mistake == "no_rowsum":
                    dS = P * dP
                else:
                    dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
                dq[bi, :, h] = scale * (dS @ K)
                dk[bi, :, hk] += scale * ((dS if mistake == "untransposed_dk" else dS.T) @ Q)
                dv[bi, :, hk] += P.T @ dO
        return dq, dk, dv
    return grad


@pytest.mark.parametrize("mistake", ["no_rowsum", "untransposed_dk"])
def test_planted_gradient_mistakes_are_caught(monkeypatch, mistake):
    monkeypatch.setattr(oracle, "attn_dual_stream_grad", _grad_with(mistake))
    with pytest.raises(AssertionError):
        test_dual_stream_grad_matches_finite_differences()


def test_planted_natural_log_statistics_are_caught(monkeypatch):
    real = oracle.attn_dual_stream_lse
    monkeypatch.setattr(oracle, "attn_dual_stream_lse",
                        lambda *a, **kw: real(*a, **kw) * math.log(2.0))
    with pytest.raises(AssertionError):
        test_dual_stream_lse_zero_queries_counts_visible_keys()


def test_planted_single_mean_over_both_streams_is_caught(monkeypatch):
    real = oracle.ce_loss_dual

    def wrong(h, w, targets, batch, L):
        _, _, ce = real(h, w, targets, batch, L)
        m = float(ce[np.asarray(targets) >= 0].mean())
        return m, m, ce
    monkeypatch.setattr(oracle, "ce_loss_dual", wrong)
    with pytest.raises(AssertionError):
        test_ce_loss_hand_worked_case()


def test_gradient_copy_without_a_mistake_passes(monkeypatch):
    """The copy the planted gradient mistakes are made in passes the same pin unchanged, so
    each failure above comes from its mistake."""
    monkeypatch.setattr(oracle, "attn_dual_stream_grad", _grad_with(None))
    test_dual_stream_grad_matches_finite_differences()


def test_planted_loss_gradient_of_the_sum_is_caught(monkeypatch):
    """dlogits = softmax - onehot without the 1/N of each stream's mean: the gradient of
    the summed cross-entropy, not of L_mask + L_AR."""
    def wrong(h, w, targets, batch, L):
        logits = h @ w.T
        p = np.exp(logits - logits.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        y = np.asarray(targets)
        ok = y >= 0
        g = np.where(ok[:, None], p, 0.0)
        g[np.flatnonzero(ok), y[ok]] -= 1.0
        return g @ w, g.T @ h, None
    monkeypatch.setattr(oracle, "ce_loss_dual_grad", wrong)
    with pytest.raises(AssertionError):
        test_ce_loss_grad_matches_finite_differences()


def test_planted_batch_sync_on_the_largest_n_is_caught(monkeypatch):
    def wrong(k_blk, v_blk, n_accept, seq_lens, block_table, k_pool, v_pool, page_size):
        n_max = max(int(x) for x in n_accept)
        return oracle.kv_commit(k_blk, v_blk, [n_max] * len(n_accept), seq_lens, block_table,
                                k_pool, v_pool, page_size)
    monkeypatch.setattr(oracle, "kv_commit_batch_sync", wrong)
    with pytest.raises(AssertionError):
        test_commit_batch_sync_golden_case()


def _block_commit_with(mistake):
    """The oracle's block-level commit with one planted mistake: "own_flush" writes a
    sequence's block as soon as that sequence has filled it (no wait for the batch);
    "no_wait" lets a full block keep taking rows past the boundary."""
    def commit(k_blk, v_blk, n_accept, seq_lens, fill, k_stage, v_stage, flush_pending,
               block_table, k_pool, v_pool, page_size, B_cache):
        k_pool, v_pool = k_pool.copy(), v_pool.copy()
        k_stage, v_stage = k_stage.copy(), v_stage.copy()
        lens = np.array(seq_lens, dtype=np.int64).copy()
        fill = np.array(fill, dtype=np.int64).copy()
        b, B = k_blk.shape[0], k_blk.shape[1]
        for s in range(b):
            if flush_pending or (mistake == "own_flush" and fill[s] == B_cache):
                for i in range(B_cache):
                    pos = int(lens[s]) + i
                    page = int(block_table[s][pos // page_size])
                    k_pool[page, :, pos % page_size] = k_stage[s, i]
                    v_pool[page, :, pos % page_size] = v_stage[s, i]
                lens[s] += B_cache
                fill[s] = 0
        slots = np.full((b, B), -1, dtype=np.int64)
        for s in range(b):
            room = B if mistake == "no_wait" else B_cache - int(fill[s])
            n = min(min(max(int(n_accept[s]), 0), B), room)
            for i in range(n):
                pos = int(lens[s]) + int(fill[s]) + i
                page = int(block_table[s][pos // page_size])
                slots[s, i] = page * page_size + pos % page_size
                if fill[s] + i < B_cache:
                    k_stage[s, int(fill[s]) + i] = k_blk[s, i]
                    v_stage[s, int(fill[s]) + i] = v_blk[s, i]
            fill[s] = min(int(fill[s]) + n, B_cache)
        flush = bool((fill == B_cache).all())
        return k_pool, v_pool, lens, fill, k_stage, v_stage, flush, slots
    return commit


@pytest.mark.parametrize("mistake", ["own_flush", "no_wait"])
def test_planted_block_commit_mistakes_are_caught(monkeypatch, mistake):
    monkeypatch.setattr(oracle, "kv_commit_block", _block_commit_with(mistake))
    with pytest.raises(AssertionError):
        test_commit_block_golden_case()


def test_block_commit_copy_without_a_mistake_passes(monkeypatch):
    monkeypatch.setattr(oracle, "kv_commit_block", _block_commit_with(None))
    test_commit_block_golden_case()
    test_commit_block_properties()


def test_planted_first_threshold_for_every_request_is_caught(monkeypatch):
    real = oracle.head_accept
    monkeypatch.setattr(oracle, "head_accept_per_request",
                        lambda h, w, batch, B, taus: real(h, w, batch, B, float(taus[0])))
    with pytest.raises(AssertionError):
        test_per_request_thresholds_golden_batch()
