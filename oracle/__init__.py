"""fp64 CPU oracle for the MARS hot path (test infrastructure only).

Only the test suite, the package smoke check and the benchmark's CPU-baseline leg may
import this package. The CUDA library never uses it.
"""
from .mars_oracle import (  # noqa: F401
    accept_count,
    ar_signal_fraction,
    attn_dual_stream,
    attn_dual_stream_grad,
    attn_dual_stream_grad_parts,
    attn_dual_stream_lse,
    beta,
    ce_loss_dual,
    ce_loss_dual_grad,
    decode_attn,
    decode_attn_staged,
    gather_prefix,
    head_accept,
    head_accept_per_request,
    head_logits,
    kv_commit,
    kv_commit_batch_sync,
    kv_commit_block,
    mask_M,
    mask_rows,
    maxprob_argmax,
)
