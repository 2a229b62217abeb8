"""ctypes binding of libmars (include/mars.h) with the same entry-point names.

Argument marshalling only: shapes, dtypes and devices are checked, raw device pointers
and the current CUDA stream are passed through, and a non-zero return code raises
MarsError. Every step of the computation runs in the library's kernels; there is no
fallback: if libmars.so is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmars.so")
_lib = None

OK, EINVAL, EALIGN, EUNSUPPORTED, ECUDA, ENOSPACE = 0, -1, -2, -3, -4, -5
ST_NOPAGE, ST_OVERFLOW, ST_TIMEOUT, ST_BADTARGET = 1, 2, 4, 8
OP_DECODE_ATTN, OP_HEAD_ACCEPT, OP_CE_LOSS, OP_CE_LOSS_GRAD, OP_DUAL_GRAD = 1, 2, 3, 4, 5
PAGE_SIZE = 16
BLOCK_SYNC_WORDS = 4


class MarsError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {mars_strerror(code)} ({code})")


def lib() -> ctypes.CDLL:
    """Load libmars.so (built in-tree by block_masked_token_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libmars.so not built at {_LIB_PATH}; run "
                               "`python -m block_masked_token_gb300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.mars_workspace_bytes.restype = S
        L.mars_workspace_bytes.argtypes = [I] * 9
        L.mars_attn_dual_stream.restype = I
        L.mars_attn_dual_stream.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P]
        L.mars_decode_attn.restype = I
        L.mars_decode_attn.argtypes = [P, P, P, P, P, I, P, I, P, I, P, I, I, I, I, I, I, F,
                                       P, S, P, P]
        L.mars_head_accept.restype = I
        L.mars_head_accept.argtypes = [P, P, I, I, I, I, F, P, P, P, P, S, P, P]
        L.mars_head_accept_per_request.restype = I
        L.mars_head_accept_per_request.argtypes = [P, P, I, I, I, I, P, P, P, P, P, S, P, P]
        L.mars_kv_commit.restype = I
        L.mars_kv_commit.argtypes = [P, P, P, P, P, I, P, P, I, P, I, I, I, I, I, P, P]
        L.mars_kv_commit_batch_sync.restype = I
        L.mars_kv_commit_batch_sync.argtypes = L.mars_kv_commit.argtypes
        L.mars_kv_commit_block.restype = I
        L.mars_kv_commit_block.argtypes = [P, P, P, P, P, P, P, I, P, P, I, P, P, I, P, I, I, I,
                                           I, I, P, P]
        L.mars_decode_attn_block_cache.restype = I
        L.mars_decode_attn_block_cache.argtypes = [P, P, P, P, P, I, P, I, P, I, P, P, P, I, P,
                                                   I, I, I, I, I, I, F, P, S, P, P]
        L.mars_dual_stream_ce_loss.restype = I
        L.mars_dual_stream_ce_loss.argtypes = [P, P, P, I, I, I, I, P, P, P, P, S, P, P]
        L.mars_attn_dual_stream_grad.restype = I
        L.mars_attn_dual_stream_grad.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P, P, P, P,
                                                 S, P, P]
        L.mars_attn_dual_stream_lse.restype = I
        L.mars_attn_dual_stream_lse.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P, P]
        L.mars_attn_dual_stream_grad_lse.restype = I
        L.mars_attn_dual_stream_grad_lse.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, P, P,
                                                     P, P, S, P, P]
        L.mars_dual_stream_ce_loss_grad.restype = I
        L.mars_dual_stream_ce_loss_grad.argtypes = [P, P, P, P, I, I, I, I, P, P, P, S, P, P]
        L.mars_check_wait_timeout.restype = I
        L.mars_check_wait_timeout.argtypes = [P, P]
        L.mars_strerror.restype = ctypes.c_char_p
        L.mars_strerror.argtypes = [I]
        L.mars_version.restype = ctypes.c_char_p
        L.mars_version.argtypes = []
        L.mars_launch_count.restype = ctypes.c_uint64
        L.mars_launch_count.argtypes = []
        _lib = L
    return _lib


EXPORTED = ("mars_workspace_bytes", "mars_attn_dual_stream", "mars_decode_attn",
            "mars_head_accept", "mars_head_accept_per_request", "mars_kv_commit",
            "mars_kv_commit_batch_sync", "mars_kv_commit_block", "mars_decode_attn_block_cache",
            "mars_dual_stream_ce_loss",
            "mars_dual_stream_ce_loss_grad", "mars_attn_dual_stream_grad",
            "mars_attn_dual_stream_lse", "mars_attn_dual_stream_grad_lse",
            "mars_check_wait_timeout", "mars_strerror",
            "mars_version", "mars_launch_count")


def mars_check_wait_timeout(status, stream=None):
    """Enqueue the wait-limit self-check: sets ST_TIMEOUT in status after about 2 s."""
    _check(status, "status", torch.int32, (1,))
    _rc(lib().mars_check_wait_timeout(_ptr(status), _stream(stream)), "mars_check_wait_timeout")


def mars_strerror(code: int) -> str:
    return lib().mars_strerror(int(code)).decode()


def mars_version() -> str:
    return lib().mars_version().decode()


def mars_launch_count() -> int:
    return int(lib().mars_launch_count())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (libmars has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _rc(code, where):
    if code != OK:
        raise MarsError(code, where)


def mars_workspace_bytes(op, batch, B, hq=1, hkv=1, d=64, hidden=8, vocab=1, max_len=0):
    return int(lib().mars_workspace_bytes(op, batch, B, hq, hkv, d, hidden, vocab, max_len))


def mars_attn_dual_stream(q, k, v, o, L: int, B: int, scale: float = 0.0, status=None,
                          stream=None):
    """o[b, 2L, hq, d] (float32) = attention of q under mask M (see include/mars.h)."""
    b, n, hq, d = q.shape
    hkv = k.shape[2]
    _check(q, "q", torch.bfloat16, (b, 2 * L, hq, d))
    _check(k, "k", torch.bfloat16, (b, 2 * L, hkv, d))
    _check(v, "v", torch.bfloat16, (b, 2 * L, hkv, d))
    _check(o, "o", torch.float32, (b, 2 * L, hq, d))
    if status is not None:
        _check(status, "status", torch.int32, (1,))
    _rc(lib().mars_attn_dual_stream(_ptr(q), _ptr(k), _ptr(v), _ptr(o), b, L, B, hq, hkv, d,
                                    float(scale), _ptr(status), _stream(stream)),
        "mars_attn_dual_stream")


def mars_decode_attn(q, k_blk, v_blk, k_pool, v_pool, block_table, seq_lens,
                     max_len_hint: int, o, workspace, status=None, scale: float = 0.0,
                     stream=None):
    b, B, hq, d = q.shape
    hkv = k_blk.shape[2]
    num_pages = k_pool.shape[0]
    _check(q, "q", torch.bfloat16)
    _check(k_blk, "k_blk", torch.bfloat16, (b, B, hkv, d))
    _check(v_blk, "v_blk", torch.bfloat16, (b, B, hkv, d))
    _check(k_pool, "k_pool", torch.bfloat16, (num_pages, hkv, PAGE_SIZE, d))
    _check(v_pool, "v_pool", torch.bfloat16, (num_pages, hkv, PAGE_SIZE, d))
    _check(block_table, "block_table", torch.int32)
    _check(seq_lens, "seq_lens", torch.int32, (b,))
    _check(o, "o", torch.float32, (b, B, hq, d))
    _check(workspace, "workspace", torch.uint8)
    if status is not None:
        _check(status, "status", torch.int32, (1,))
    _rc(lib().mars_decode_attn(_ptr(q), _ptr(k_blk), _ptr(v_blk), _ptr(k_pool), _ptr(v_pool),
                               num_pages, _ptr(block_table), block_table.shape[1],
                               _ptr(seq_lens), int(max_len_hint), _ptr(o), b, B, hq, hkv, d,
                               PAGE_SIZE, float(scale), _ptr(workspace), workspace.numel(),
                               _ptr(status), _stream(stream)), "mars_decode_attn")


def _head_args(h, w, batch, B, tokens, maxprob, n_accept, workspace, status):
    rows, hidden = h.shape
    vocab = w.shape[0]
    _check(h, "h", torch.bfloat16, (batch * B, hidden))
    _check(w, "w", torch.bfloat16, (vocab, hidden))
    _check(tokens, "tokens", torch.int32, (batch, B))
    _check(maxprob, "maxprob", torch.float32, (batch, B))
    _check(n_accept, "n_accept", torch.int32, (batch,))
    _check(workspace, "workspace", torch.uint8)
    if status is not None:
        _check(status, "status", torch.int32, (1,))
    return hidden, vocab


def mars_head_accept(h, w, batch: int, B: int, tau: float, tokens, maxprob, n_accept,
                     workspace, status=None, stream=None):
    hidden, vocab = _head_args(h, w, batch, B, tokens, maxprob, n_accept, workspace, status)
    _rc(lib().mars_head_accept(_ptr(h), _ptr(w), batch, B, hidden, vocab, float(tau),
                               _ptr(tokens), _ptr(maxprob), _ptr(n_accept), _ptr(workspace),
                               workspace.numel(), _ptr(status), _stream(stream)),
        "mars_head_accept")


def mars_head_accept_per_request(h, w, batch: int, B: int, taus, tokens, maxprob, n_accept,
                                 workspace, status=None, stream=None):
    hidden, vocab = _head_args(h, w, batch, B, tokens, maxprob, n_accept, workspace, status)
    _check(taus, "taus", torch.float32, (batch,))
    _rc(lib().mars_head_accept_per_request(_ptr(h), _ptr(w), batch, B, hidden, vocab,
                                           _ptr(taus), _ptr(tokens), _ptr(maxprob),
                                           _ptr(n_accept), _ptr(workspace), workspace.numel(),
                                           _ptr(status), _stream(stream)),
        "mars_head_accept_per_request")


def _kv_commit(fn, name, k_blk, v_blk, n_accept, seq_lens, block_table, k_pool, v_pool,
               commit_slots, status, stream):
    b, B, hkv, d = k_blk.shape
    num_pages = k_pool.shape[0]
    _check(k_blk, "k_blk", torch.bfloat16)
    _check(v_blk, "v_blk", torch.bfloat16, (b, B, hkv, d))
    _check(n_accept, "n_accept", torch.int32, (b,))
    _check(seq_lens, "seq_lens", torch.int32, (b,))
    _check(block_table, "block_table", torch.int32)
    _check(k_pool, "k_pool", torch.bfloat16, (num_pages, hkv, PAGE_SIZE, d))
    _check(v_pool, "v_pool", torch.bfloat16, (num_pages, hkv, PAGE_SIZE, d))
    if commit_slots is not None:
        _check(commit_slots, "commit_slots", torch.int32, (b, B))
    if status is not None:
        _check(status, "status", torch.int32, (1,))
    _rc(fn(_ptr(k_blk), _ptr(v_blk), _ptr(n_accept), _ptr(seq_lens), _ptr(block_table),
           block_table.shape[1], _ptr(k_pool), _ptr(v_pool), num_pages, _ptr(commit_slots), b,
           B, hkv, d, PAGE_SIZE, _ptr(status), _stream(stream)), name)


def mars_kv_commit(k_blk, v_blk, n_accept, seq_lens, block_table, k_pool, v_pool,
                   commit_slots=None, status=None, stream=None):
    _kv_commit(lib().mars_kv_commit, "mars_kv_commit", k_blk, v_blk, n_accept, seq_lens,
               block_table, k_pool, v_pool, commit_slots, status, stream)


def mars_kv_commit_batch_sync(k_blk, v_blk, n_accept, seq_lens, block_table, k_pool, v_pool,
                              commit_slots=None, status=None, stream=None):
    _kv_commit(lib().mars_kv_commit_batch_sync, "mars_kv_commit_batch_sync", k_blk, v_blk,
               n_accept, seq_lens, block_table, k_pool, v_pool, commit_slots, status, stream)


def mars_kv_commit_block(k_blk, v_blk, n_accept, seq_lens, block_fill, k_stage, v_stage,
                         sync_state, block_table, k_pool, v_pool, commit_slots=None,
                         status=None, stream=None):
    """Block-level commit with a B_cache boundary (B_cache = k_stage.shape[1]); the state
    tensors seq_lens, block_fill, sync_state (and the stage) persist between calls."""
    b, B, hkv, d = k_blk.shape
    B_cache = k_stage.shape[1]
    num_pages = k_pool.shape[0]
    _check(k_blk, "k_blk", torch.bfloat16)
    _check(v_blk, "v_blk", torch.bfloat16, (b, B, hkv, d))
    _check(n_accept, "n_accept", torch.int32, (b,))
    _check(seq_lens, "seq_lens", torch.int32, (b,))
    _check(block_fill, "block_fill", torch.int32, (b,))
    _check(k_stage, "k_stage", torch.bfloat16, (b, B_cache, hkv, d))
    _check(v_stage, "v_stage", torch.bfloat16, (b, B_cache, hkv, d))
    _check(sync_state, "sync_state", torch.int32, (BLOCK_SYNC_WORDS,))
    _check(block_table, "block_table", torch.int32)
    _check(k_pool, "k_pool", torch.bfloat16, (num_pages, hkv, PAGE_SIZE, d))
    _check(v_pool, "v_pool", torch.bfloat16, (num_pages, hkv, PAGE_SIZE, d))
    if commit_slots is not None:
        _check(commit_slots, "commit_slots", torch.int32, (b, B))
    if status is not None:
        _check(status, "status", torch.int32, (1,))
    _rc(lib().mars_kv_commit_block(_ptr(k_blk), _ptr(v_blk), _ptr(n_accept), _ptr(seq_lens),
                                   _ptr(block_fill), _ptr(k_stage), _ptr(v_stage), B_cache,
                                   _ptr(sync_state), _ptr(block_table), block_table.shape[1],
                                   _ptr(k_pool), _ptr(v_pool), num_pages, _ptr(commit_slots),
                                   b, B, hkv, d, PAGE_SIZE, _ptr(status), _stream(stream)),
        "mars_kv_commit_block")


def mars_decode_attn_block_cache(q, k_blk, v_blk, k_pool, v_pool, block_table, seq_lens,
                                 max_len_hint: int, k_stage, v_stage, block_fill, o, workspace,
                                 status=None, scale: float = 0.0, stream=None):
    """mars_decode_attn with the block buffers of mars_kv_commit_block between the prefix
    and the block keys (B_cache = k_stage.shape[1])."""
    b, B, hq, d = q.shape
    hkv = k_blk.shape[2]
    num_pages = k_pool.shape[0]
    B_cache = k_stage.shape[1]
    _check(q, "q", torch.bfloat16)
    _check(k_blk, "k_blk", torch.bfloat16, (b, B, hkv, d))
    _check(v_blk, "v_blk", torch.bfloat16, (b, B, hkv, d))
    _check(k_pool, "k_pool", torch.bfloat16, (num_pages, hkv, PAGE_SIZE, d))
    _check(v_pool, "v_pool", torch.bfloat16, (num_pages, hkv, PAGE_SIZE, d))
    _check(block_table, "block_table", torch.int32)
    _check(seq_lens, "seq_lens", torch.int32, (b,))
    _check(k_stage, "k_stage", torch.bfloat16, (b, B_cache, hkv, d))
    _check(v_stage, "v_stage", torch.bfloat16, (b, B_cache, hkv, d))
    _check(block_fill, "block_fill", torch.int32, (b,))
    _check(o, "o", torch.float32, (b, B, hq, d))
    _check(workspace, "workspace", torch.uint8)
    if status is not None:
        _check(status, "status", torch.int32, (1,))
    _rc(lib().mars_decode_attn_block_cache(
        _ptr(q), _ptr(k_blk), _ptr(v_blk), _ptr(k_pool), _ptr(v_pool), num_pages,
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), int(max_len_hint),
        _ptr(k_stage), _ptr(v_stage), _ptr(block_fill), B_cache, _ptr(o), b, B, hq, hkv, d,
        PAGE_SIZE, float(scale), _ptr(workspace), workspace.numel(), _ptr(status),
        _stream(stream)), "mars_decode_attn_block_cache")


def mars_dual_stream_ce_loss(h, w, targets, batch: int, L: int, loss, workspace, row_ce=None,
                             row_lse=None, status=None, stream=None):
    rows, hidden = h.shape
    vocab = w.shape[0]
    _check(h, "h", torch.bfloat16, (batch * 2 * L, hidden))
    _check(w, "w", torch.bfloat16, (vocab, hidden))
    _check(targets, "targets", torch.int32, (batch * 2 * L,))
    _check(loss, "loss", torch.float32, (3,))
    _check(workspace, "workspace", torch.uint8)
    for t, name in ((row_ce, "row_ce"), (row_lse, "row_lse")):
        if t is not None:
            _check(t, name, torch.float32, (batch * 2 * L,))
    if status is not None:
        _check(status, "status", torch.int32, (1,))
    _rc(lib().mars_dual_stream_ce_loss(_ptr(h), _ptr(w), _ptr(targets), batch, L, hidden,
                                       vocab, _ptr(loss), _ptr(row_ce), _ptr(row_lse),
                                       _ptr(workspace), workspace.numel(), _ptr(status),
                                       _stream(stream)),
        "mars_dual_stream_ce_loss")


def mars_dual_stream_ce_loss_grad(h, w, targets, row_lse, batch: int, L: int, workspace,
                                  dh=None, dw=None, status=None, stream=None):
    rows, hidden = h.shape
    vocab = w.shape[0]
    _check(h, "h", torch.bfloat16, (batch * 2 * L, hidden))
    _check(w, "w", torch.bfloat16, (vocab, hidden))
    _check(targets, "targets", torch.int32, (batch * 2 * L,))
    _check(row_lse, "row_lse", torch.float32, (batch * 2 * L,))
    _check(workspace, "workspace", torch.uint8)
    if dh is not None:
        _check(dh, "dh", torch.float32, (batch * 2 * L, hidden))
    if dw is not None:
        _check(dw, "dw", torch.float32, (vocab, hidden))
    if status is not None:
        _check(status, "status", torch.int32, (1,))
    _rc(lib().mars_dual_stream_ce_loss_grad(_ptr(h), _ptr(w), _ptr(targets), _ptr(row_lse),
                                            batch, L, hidden, vocab, _ptr(dh), _ptr(dw),
                                            _ptr(workspace), workspace.numel(), _ptr(status),
                                            _stream(stream)),
        "mars_dual_stream_ce_loss_grad")


def dual_lse_shape(b: int, hq: int, L: int):
    """Shape of the row statistics mars_attn_dual_stream_lse writes: [b, hq, 2, Lp], Lp = L
    rounded up to a multiple of 128."""
    return (b, hq, 2, (L + 127) // 128 * 128)


def mars_attn_dual_stream_lse(q, k, v, o, lse, L: int, B: int, scale: float = 0.0, status=None,
                              stream=None):
    """mars_attn_dual_stream that also writes each row's softmax log-sum-exp (log2) into
    lse [b, hq, 2, Lp] float32 (see include/mars.h)."""
    b, n, hq, d = q.shape
    hkv = k.shape[2]
    _check(q, "q", torch.bfloat16, (b, 2 * L, hq, d))
    _check(k, "k", torch.bfloat16, (b, 2 * L, hkv, d))
    _check(v, "v", torch.bfloat16, (b, 2 * L, hkv, d))
    _check(o, "o", torch.float32, (b, 2 * L, hq, d))
    _check(lse, "lse", torch.float32, dual_lse_shape(b, hq, L))
    if status is not None:
        _check(status, "status", torch.int32, (1,))
    _rc(lib().mars_attn_dual_stream_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), b, L, B,
                                        hq, hkv, d, float(scale), _ptr(status), _stream(stream)),
        "mars_attn_dual_stream_lse")


def mars_attn_dual_stream_grad_lse(q, k, v, o, d_o, lse, L: int, B: int, dq, dk, dv, workspace,
                                   scale: float = 0.0, status=None, stream=None):
    """mars_attn_dual_stream_grad from the forward's lse (mars_attn_dual_stream_lse)."""
    b, n, hq, d = q.shape
    hkv = k.shape[2]
    _check(q, "q", torch.bfloat16, (b, 2 * L, hq, d))
    _check(k, "k", torch.bfloat16, (b, 2 * L, hkv, d))
    _check(v, "v", torch.bfloat16, (b, 2 * L, hkv, d))
    _check(o, "o", torch.float32, (b, 2 * L, hq, d))
    _check(d_o, "d_o", torch.float32, (b, 2 * L, hq, d))
    _check(lse, "lse", torch.float32, dual_lse_shape(b, hq, L))
    _check(dq, "dq", torch.float32, (b, 2 * L, hq, d))
    _check(dk, "dk", torch.float32, (b, 2 * L, hkv, d))
    _check(dv, "dv", torch.float32, (b, 2 * L, hkv, d))
    _check(workspace, "workspace", torch.uint8)
    _rc(lib().mars_attn_dual_stream_grad_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(d_o),
                                             _ptr(lse), b, L, B, hq, hkv, d, float(scale),
                                             _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                             workspace.numel(), _ptr(status), _stream(stream)),
        "mars_attn_dual_stream_grad_lse")


def mars_attn_dual_stream_grad(q, k, v, o, d_o, L: int, B: int, dq, dk, dv, workspace,
                               scale: float = 0.0, status=None, stream=None):
    b, n, hq, d = q.shape
    hkv = k.shape[2]
    _check(q, "q", torch.bfloat16, (b, 2 * L, hq, d))
    _check(k, "k", torch.bfloat16, (b, 2 * L, hkv, d))
    _check(v, "v", torch.bfloat16, (b, 2 * L, hkv, d))
    _check(o, "o", torch.float32, (b, 2 * L, hq, d))
    _check(d_o, "d_o", torch.float32, (b, 2 * L, hq, d))
    _check(dq, "dq", torch.float32, (b, 2 * L, hq, d))
    _check(dk, "dk", torch.float32, (b, 2 * L, hkv, d))
    _check(dv, "dv", torch.float32, (b, 2 * L, hkv, d))
    _check(workspace, "workspace", torch.uint8)
    _rc(lib().mars_attn_dual_stream_grad(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(d_o), b, L,
                                         B, hq, hkv, d, float(scale), _ptr(dq), _ptr(dk),
                                         _ptr(dv), _ptr(workspace), workspace.numel(),
                                         _ptr(status), _stream(stream)),
        "mars_attn_dual_stream_grad")
