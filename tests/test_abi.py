"""The C ABI library loads and exports every entry point include/mars.h declares, and its
host-side argument checks reject bad calls before launching anything (CPU only: the
calls below return an error code before any CUDA call)."""
import ctypes
import os
import re

import pytest

from block_masked_token_gb300 import mars

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(mars_\w+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(mars._LIB_PATH):
        from block_masked_token_gb300.build import build_library
        build_library()
    return mars.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert {"mars_attn_dual_stream", "mars_decode_attn", "mars_head_accept",
            "mars_kv_commit"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
    for n in mars.EXPORTED:
        assert n in names


def test_strerror_and_version(L):
    for code in (0, -1, -2, -3, -4, -5, 7):
        assert mars.mars_strerror(code)
    assert "sm_103a" in mars.mars_version()


def test_ce_workspace_size(L):
    rows, nvt = 2 * 2 * 100, (1000 + 255) // 256
    want = rows * nvt * 16 + ((rows * 4 + 255) // 256) * 256
    assert mars.mars_workspace_bytes(mars.OP_CE_LOSS, 2, 1, vocab=1000, max_len=100) == want
    assert mars.mars_workspace_bytes(mars.OP_CE_LOSS, 2, 1, vocab=1000, max_len=0) == 0


def test_workspace_sizes(L):
    assert mars.mars_workspace_bytes(mars.OP_HEAD_ACCEPT, 2, 4, vocab=512) > 0
    ws = mars.mars_workspace_bytes(mars.OP_DECODE_ATTN, 32, 8, 28, 4, 128, max_len=2048)
    assert ws > 0 and ws % 16 == 0
    assert mars.mars_workspace_bytes(99, 1, 1) == 0
    assert mars.mars_workspace_bytes(mars.OP_DECODE_ATTN, 1, 4, 3, 2, 64) == 0   # hq % hkv
    assert mars.mars_workspace_bytes(mars.OP_DECODE_ATTN, 1, 33, 4, 2, 64) == 0  # B > 32


def _p(v=16):
    return ctypes.c_void_p(v)


def test_host_validation_codes(L):
    P = _p()
    # dual stream: unsupported head dim, bad group, misaligned pointer, null pointer
    assert L.mars_attn_dual_stream(P, P, P, P, 1, 8, 2, 4, 2, 96, 0.0, None, None) == mars.EUNSUPPORTED
    assert L.mars_attn_dual_stream(P, P, P, P, 1, 8, 2, 3, 2, 64, 0.0, None, None) == mars.EINVAL
    assert L.mars_attn_dual_stream(P, _p(18), P, P, 1, 8, 2, 4, 2, 64, 0.0, None, None) == mars.EALIGN
    assert L.mars_attn_dual_stream(None, P, P, P, 1, 8, 2, 4, 2, 64, 0.0, None, None) == mars.EINVAL
    assert L.mars_attn_dual_stream(P, P, P, P, 0, 8, 2, 4, 2, 64, 0.0, None, None) == mars.OK
    # head: NaN / inf tau, hidden not a multiple of 8, workspace too small
    nan = float("nan")
    assert L.mars_head_accept(P, P, 1, 4, 256, 512, nan, P, P, P, P, 1 << 20, None, None) == mars.EINVAL
    assert L.mars_head_accept(P, P, 1, 4, 256, 512, float("inf"), P, P, P, P, 1 << 20, None, None) == mars.EINVAL
    assert L.mars_head_accept(P, P, 1, 4, 252, 512, 0.9, P, P, P, P, 1 << 20, None, None) == mars.EUNSUPPORTED
    assert L.mars_head_accept(P, P, 1, 4, 256, 512, 0.9, P, P, P, P, 16, None, None) == mars.ENOSPACE
    assert L.mars_head_accept(P, P, 1, 0, 256, 512, 0.9, P, P, P, P, 1 << 20, None, None) == mars.EINVAL
    # decode: page size, B range, workspace too small
    args = [P, P, P, P, P, 10, P, 4, P, 64, P, 2, 4, 4, 2, 64]
    assert L.mars_decode_attn(*args, 8, 0.0, P, 1 << 30, None, None) == mars.EUNSUPPORTED
    assert L.mars_decode_attn(*args, 16, 0.0, P, 16, None, None) == mars.ENOSPACE
    too_many_rows = list(args)        # 28/4 heads: 7 query rows per kv head per position
    too_many_rows[13], too_many_rows[14], too_many_rows[12] = 28, 4, 19
    assert L.mars_decode_attn(*too_many_rows[:15], 128, 16, 0.0, P, 1 << 30, None, None) == mars.EUNSUPPORTED
    bad_b = list(args)
    bad_b[12] = 33
    assert L.mars_decode_attn(*bad_b, 16, 0.0, P, 1 << 30, None, None) == mars.EINVAL
    # head, per-request thresholds: null threshold array, then the checks of mars_head_accept
    assert L.mars_head_accept_per_request(P, P, 1, 4, 256, 512, None, P, P, P, P, 1 << 20, None, None) == mars.EINVAL
    assert L.mars_head_accept_per_request(P, P, 0, 4, 256, 512, None, P, P, P, P, 1 << 20, None, None) == mars.OK
    assert L.mars_head_accept_per_request(P, P, 1, 4, 252, 512, P, P, P, P, P, 1 << 20, None, None) == mars.EUNSUPPORTED
    assert L.mars_head_accept_per_request(P, P, 1, 4, 256, 512, P, P, P, P, P, 16, None, None) == mars.ENOSPACE
    assert L.mars_head_accept_per_request(P, _p(20), 1, 4, 256, 512, P, P, P, P, P, 1 << 20, None, None) == mars.EALIGN
    # loss: null loss pointer, hidden not a multiple of 8, workspace too small, L < 1
    assert L.mars_dual_stream_ce_loss(P, P, P, 1, 4, 64, 100, None, None, None, P, 1 << 30, None, None) == mars.EINVAL
    assert L.mars_dual_stream_ce_loss(P, P, P, 1, 4, 60, 100, P, None, None, P, 1 << 30, None, None) == mars.EUNSUPPORTED
    assert L.mars_dual_stream_ce_loss(P, P, P, 1, 4, 64, 100, P, None, None, P, 16, None, None) == mars.ENOSPACE
    assert L.mars_dual_stream_ce_loss(P, P, P, 1, 0, 64, 100, P, None, None, P, 1 << 30, None, None) == mars.EINVAL
    # attention gradient: unsupported head dim, null output, workspace too small
    ga = [P, P, P, P, P, 1, 8, 2, 4, 2]
    assert L.mars_attn_dual_stream_grad(*ga, 96, 0.0, P, P, P, P, 1 << 30, None, None) == mars.EUNSUPPORTED
    assert L.mars_attn_dual_stream_grad(*ga, 64, 0.0, None, P, P, P, 1 << 30, None, None) == mars.EINVAL
    assert L.mars_attn_dual_stream_grad(*ga, 64, 0.0, P, P, P, P, 16, None, None) == mars.ENOSPACE
    # wait-limit self-check: the status word is required
    assert L.mars_check_wait_timeout(None, None) == mars.EINVAL
    # forward with row statistics: null lse, misaligned lse, unsupported head dim
    assert L.mars_attn_dual_stream_lse(P, P, P, P, None, 1, 8, 2, 4, 2, 64, 0.0, None, None) == mars.EINVAL
    assert L.mars_attn_dual_stream_lse(P, P, P, P, _p(20), 1, 8, 2, 4, 2, 64, 0.0, None, None) == mars.EALIGN
    assert L.mars_attn_dual_stream_lse(P, P, P, P, P, 1, 8, 2, 4, 2, 96, 0.0, None, None) == mars.EUNSUPPORTED
    assert L.mars_attn_dual_stream_lse(P, P, P, P, None, 0, 8, 2, 4, 2, 64, 0.0, None, None) == mars.OK
    # gradient from those statistics: null lse, misaligned lse, workspace too small
    gl = [P, P, P, P, P]
    assert L.mars_attn_dual_stream_grad_lse(*gl, None, 1, 8, 2, 4, 2, 64, 0.0, P, P, P, P, 1 << 30, None, None) == mars.EINVAL
    assert L.mars_attn_dual_stream_grad_lse(*gl, _p(20), 1, 8, 2, 4, 2, 64, 0.0, P, P, P, P, 1 << 30, None, None) == mars.EALIGN
    assert L.mars_attn_dual_stream_grad_lse(*gl, P, 1, 8, 2, 4, 2, 64, 0.0, P, P, P, P, 16, None, None) == mars.ENOSPACE
    # loss gradient: vocabulary not a multiple of 8, null row_lse, workspace too small
    assert L.mars_dual_stream_ce_loss_grad(P, P, P, P, 1, 4, 64, 100, P, P, P, 1 << 30, None, None) == mars.EUNSUPPORTED
    assert L.mars_dual_stream_ce_loss_grad(P, P, P, None, 1, 4, 64, 96, P, P, P, 1 << 30, None, None) == mars.EINVAL
    assert L.mars_dual_stream_ce_loss_grad(P, P, P, P, 1, 4, 64, 96, P, P, P, 16, None, None) == mars.ENOSPACE
    assert L.mars_dual_stream_ce_loss_grad(P, P, P, P, 0, 4, 64, 96, P, P, P, 16, None, None) == mars.OK
    # commit (both policies): page size, null pool, B out of range
    for fn in (L.mars_kv_commit, L.mars_kv_commit_batch_sync):
        assert fn(P, P, P, P, P, 4, P, P, 10, None, 2, 4, 2, 64, 8, None, None) == mars.EUNSUPPORTED
        assert fn(P, P, P, P, P, 4, None, P, 10, None, 2, 4, 2, 64, 16, None, None) == mars.EINVAL
        assert fn(P, P, P, P, P, 4, P, P, 10, None, 2, 33, 2, 64, 16, None, None) == mars.EINVAL
        assert fn(P, P, P, P, P, 4, P, P, 10, None, 0, 4, 2, 64, 16, None, None) == mars.OK
    # block-level commit: B_cache range and alignment, null state, page size, misaligned stage
    cb = L.mars_kv_commit_block
    for bc in (4, 12, 72):
        assert cb(P, P, P, P, P, P, P, bc, P, P, 4, P, P, 10, None, 2, 4, 2, 64, 16, None, None) == mars.EUNSUPPORTED
    assert cb(P, P, P, P, P, P, P, 16, None, P, 4, P, P, 10, None, 2, 4, 2, 64, 16, None, None) == mars.EINVAL
    assert cb(P, P, P, P, None, P, P, 16, P, P, 4, P, P, 10, None, 2, 4, 2, 64, 16, None, None) == mars.EINVAL
    assert cb(P, P, P, P, P, P, P, 16, P, P, 4, P, P, 10, None, 2, 4, 2, 64, 8, None, None) == mars.EUNSUPPORTED
    assert cb(P, P, P, P, P, _p(24), P, 16, P, P, 4, P, P, 10, None, 2, 4, 2, 64, 16, None, None) == mars.EALIGN
    assert cb(P, P, P, P, P, P, P, 16, P, P, 4, P, P, 10, None, 0, 4, 2, 64, 16, None, None) == mars.OK
    # decode over the block-level cache: B_cache range, null block_fill, workspace too small
    da = [P, P, P, P, P, 10, P, 4, P, 64]
    tail = [P, 2, 4, 4, 2, 64, 16, 0.0, P]
    assert L.mars_decode_attn_block_cache(*da, P, P, P, 20, *tail, 1 << 30, None, None) == mars.EUNSUPPORTED
    assert L.mars_decode_attn_block_cache(*da, P, P, None, 16, *tail, 1 << 30, None, None) == mars.EINVAL
    assert L.mars_decode_attn_block_cache(*da, P, P, P, 16, *tail, 16, None, None) == mars.ENOSPACE
    assert L.mars_decode_attn_block_cache(*da, _p(20), P, P, 16, *tail, 1 << 30, None, None) == mars.EALIGN


def test_binding_rejects_cpu_tensors(L):
    import torch
    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    o = torch.zeros(1, 8, 2, 64)
    with pytest.raises(ValueError, match="CUDA"):
        mars.mars_attn_dual_stream(q, q[:, :, :1].contiguous(), q[:, :, :1].contiguous(), o, L=4, B=2)


def test_every_binding_rejects_cpu_tensors(L):
    """No entry point has a CPU path: each binding refuses host tensors before anything
    is launched, and every tensor-taking binding is covered here."""
    import inspect

    import torch

    def z(*shape, dt=torch.float32):
        return torch.zeros(*shape, dtype=dt)

    def bf(*shape):
        return z(*shape, dt=torch.bfloat16)

    def i32(*shape):
        return z(*shape, dt=torch.int32)

    ws = z(64, dt=torch.uint8)
    q, kv, o = bf(1, 8, 2, 64), bf(1, 8, 1, 64), z(1, 8, 2, 64)
    kvf = z(1, 8, 1, 64)
    lse = z(1, 2, 2, 128)
    pool = bf(4, 1, 16, 64)
    blk = bf(1, 4, 1, 64)
    calls = {
        "mars_attn_dual_stream": lambda: mars.mars_attn_dual_stream(q, kv, kv, o, 4, 2),
        "mars_attn_dual_stream_lse":
            lambda: mars.mars_attn_dual_stream_lse(q, kv, kv, o, lse, 4, 2),
        "mars_attn_dual_stream_grad":
            lambda: mars.mars_attn_dual_stream_grad(q, kv, kv, o, o, 4, 2, o, kvf, kvf, ws),
        "mars_attn_dual_stream_grad_lse":
            lambda: mars.mars_attn_dual_stream_grad_lse(q, kv, kv, o, o, lse, 4, 2, o, kvf, kvf,
                                                        ws),
        "mars_decode_attn":
            lambda: mars.mars_decode_attn(bf(1, 4, 2, 64), blk, blk, pool, pool, i32(1, 4),
                                          i32(1), 64, z(1, 4, 2, 64), ws),
        "mars_head_accept":
            lambda: mars.mars_head_accept(bf(4, 256), bf(512, 256), 1, 4, 0.9, i32(1, 4),
                                          z(1, 4), i32(1), ws),
        "mars_head_accept_per_request":
            lambda: mars.mars_head_accept_per_request(bf(4, 256), bf(512, 256), 1, 4, z(1),
                                                      i32(1, 4), z(1, 4), i32(1), ws),
        "mars_kv_commit":
            lambda: mars.mars_kv_commit(blk, blk, i32(1), i32(1), i32(1, 4), pool, pool),
        "mars_kv_commit_batch_sync":
            lambda: mars.mars_kv_commit_batch_sync(blk, blk, i32(1), i32(1), i32(1, 4), pool,
                                                   pool),
        "mars_kv_commit_block":
            lambda: mars.mars_kv_commit_block(blk, blk, i32(1), i32(1), i32(1), bf(1, 16, 1, 64),
                                              bf(1, 16, 1, 64), i32(4), i32(1, 4), pool, pool),
        "mars_decode_attn_block_cache":
            lambda: mars.mars_decode_attn_block_cache(bf(1, 4, 2, 64), blk, blk, pool, pool,
                                                      i32(1, 4), i32(1), 64, bf(1, 16, 1, 64),
                                                      bf(1, 16, 1, 64), i32(1), z(1, 4, 2, 64),
                                                      ws),
        "mars_dual_stream_ce_loss":
            lambda: mars.mars_dual_stream_ce_loss(bf(8, 64), bf(96, 64), i32(8), 1, 4, z(3), ws),
        "mars_dual_stream_ce_loss_grad":
            lambda: mars.mars_dual_stream_ce_loss_grad(bf(8, 64), bf(96, 64), i32(8), z(8), 1,
                                                       4, ws),
        "mars_check_wait_timeout": lambda: mars.mars_check_wait_timeout(i32(1)),
    }
    scalar_only = {"mars_strerror", "mars_version", "mars_launch_count", "mars_workspace_bytes"}
    bindings = {n for n, f in vars(mars).items()
                if n.startswith("mars_") and inspect.isfunction(f)} - scalar_only
    assert bindings == set(calls), bindings ^ set(calls)
    for name, call in calls.items():
        with pytest.raises(ValueError, match="CUDA"):
            call()

