"""mars_head_accept_noalloc against mars_head_accept (GPU).

The no-allocation entry point is for callers that cannot call cudaMalloc when they run a
decode step (memory reserved up front, a host framework that owns all device memory, a
real-time path). It keeps its scratch in a fixed library-owned device array, so it must
give the same tokens, max-probs and N as the workspace entry point, call after call, and
refuse sizes its scratch cannot hold. This file is collected last on purpose: a failure
here leaves every other test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_masked_token_gb300 import mars
from block_masked_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
SCRATCH_BYTES = 8 << 20          # MARS_NOALLOC_SCRATCH_BYTES


def _noalloc():
    L = mars.lib()
    fn = L.mars_head_accept_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = I
    fn.argtypes = [P, P, I, I, I, I, F, P, P, P, P, P]
    return fn


def _outputs(batch, B):
    return (torch.full((batch, B), -7, dtype=torch.int32, device=DEV),
            torch.full((batch, B), -7.0, dtype=torch.float32, device=DEV),
            torch.full((batch,), -7, dtype=torch.int32, device=DEV))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("batch,B,hidden,vocab,tau", [
    (2, 4, 256, 512, 0.9),           # the tiny decode step's head
    (32, 8, 3584, 152064, 0.9),      # the 7B-class head (2.4 MB of scratch)
    (3, 5, 64, 1000, 0.0),           # ragged vocabulary tile, whole block accepted
])
def test_noalloc_matches_workspace_entry_point(batch, B, hidden, vocab, tau):
    fn = _noalloc()
    cfg = W.DecodeConfig("n", batch=batch, prefix_lo=1, prefix_hi=1, B=B, hq=1, hkv=1, d=64,
                         hidden=hidden, vocab=vocab, taus=(tau,))
    inp = W.make_decode_inputs(cfg, seed=11, device=DEV, steps=2)
    w = inp.w
    stream = torch.cuda.current_stream()
    for step in range(2):                    # two calls in a row share the scratch
        h = inp.h[step]
        tok, mp, n = _outputs(batch, B)
        ws = torch.empty(mars.mars_workspace_bytes(mars.OP_HEAD_ACCEPT, batch, B, vocab=vocab),
                         dtype=torch.uint8, device=DEV)
        mars.mars_head_accept(h, w, batch, B, tau, tok, mp, n, ws)
        tok2, mp2, n2 = _outputs(batch, B)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = fn(_ptr(h), _ptr(w), batch, B, hidden, vocab, tau, _ptr(tok2), _ptr(mp2),
                _ptr(n2), _ptr(st), ctypes.c_void_p(stream.cuda_stream))
        torch.cuda.synchronize()
        assert rc == mars.OK, mars.mars_strerror(rc)
        assert int(st.item()) == 0
        np.testing.assert_array_equal(tok2.cpu().numpy(), tok.cpu().numpy())
        np.testing.assert_allclose(mp2.cpu().numpy(), mp.cpu().numpy(), rtol=0, atol=1e-4)
        np.testing.assert_array_equal(n2.cpu().numpy(), n.cpu().numpy())


def _call(fn, h, w, batch, B, hidden, vocab, tau, tok, mp, n, st):
    stream = torch.cuda.current_stream()
    return fn(_ptr(h), _ptr(w), batch, B, hidden, vocab, tau, _ptr(tok), _ptr(mp), _ptr(n),
              _ptr(st), ctypes.c_void_p(stream.cuda_stream))


def _largest_rows(vocab):
    """The most rows (a whole number of 128-row blocks) whose workspace fits the scratch,
    by the library's own workspace size."""
    rows = 128
    while mars.mars_workspace_bytes(mars.OP_HEAD_ACCEPT, rows + 128, 1, vocab=vocab) <= \
            SCRATCH_BYTES:
        rows += 128
    assert mars.mars_workspace_bytes(mars.OP_HEAD_ACCEPT, rows, 1, vocab=vocab) <= SCRATCH_BYTES
    return rows


def test_noalloc_at_its_exact_limit_allocates_nothing():
    """The largest call the scratch holds (a whole number of row blocks at vocabulary
    152064, B = 16) matches the workspace entry point on two calls in a row, and the second
    call changes neither the device's free memory nor the caching allocator's counters;
    one row more is refused with ENOSPACE before anything runs."""
    fn = _noalloc()
    hidden, vocab, tau, B = 3584, 152064, 0.5, 16
    rows = _largest_rows(vocab)
    batch = rows // B
    cfg = W.DecodeConfig("lim", batch=batch, prefix_lo=1, prefix_hi=1, B=B, hq=1, hkv=1, d=64,
                         hidden=hidden, vocab=vocab, taus=(tau,))
    inp = W.make_decode_inputs(cfg, seed=12, device=DEV, steps=2)
    ws = torch.empty(mars.mars_workspace_bytes(mars.OP_HEAD_ACCEPT, batch, B, vocab=vocab),
                     dtype=torch.uint8, device=DEV)
    tok2, mp2, n2 = _outputs(batch, B)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for step in range(2):
        tok, mp, n = _outputs(batch, B)
        mars.mars_head_accept(inp.h[step], inp.w, batch, B, tau, tok, mp, n, ws)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        stats0 = torch.cuda.memory_stats()
        rc = _call(fn, inp.h[step], inp.w, batch, B, hidden, vocab, tau, tok2, mp2, n2, st)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        stats1 = torch.cuda.memory_stats()
        assert rc == mars.OK, mars.mars_strerror(rc)
        assert int(st.item()) == 0
        if step == 1:                      # the first call may set the device up
            assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
            for key in ("allocation.all.allocated", "segment.all.allocated",
                        "allocated_bytes.all.allocated", "reserved_bytes.all.allocated"):
                assert stats1.get(key, 0) == stats0.get(key, 0), key
        np.testing.assert_array_equal(tok2.cpu().numpy(), tok.cpu().numpy())
        np.testing.assert_allclose(mp2.cpu().numpy(), mp.cpu().numpy(), rtol=0, atol=1e-4)
        np.testing.assert_array_equal(n2.cpu().numpy(), n.cpu().numpy())
    # one row more (batch rows + 1, B 1): one more row block than the scratch holds
    assert mars.mars_workspace_bytes(mars.OP_HEAD_ACCEPT, rows + 1, 1, vocab=vocab) > \
        SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.uint8, device=DEV)
    p = _ptr(dummy)
    rc = fn(p, p, rows + 1, 1, hidden, vocab, tau, p, p, p, None, None)
    assert rc == mars.ENOSPACE


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fn = _noalloc()
    batch, B, hidden, vocab = 512, 16, 3584, 152064     # 8192 rows: 64 row blocks
    assert mars.mars_workspace_bytes(mars.OP_HEAD_ACCEPT, batch, B, vocab=vocab) > SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.uint8, device=DEV)
    p = _ptr(dummy)
    rc = fn(p, p, batch, B, hidden, vocab, 0.9, p, p, p, None, None)
    assert rc == mars.ENOSPACE
