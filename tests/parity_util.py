"""Comparison rules between the CUDA path and the fp64 oracle.

Attention outputs: max-abs error <= 1e-2 against the oracle run on the same bf16-rounded
inputs. Max-probs: |delta| <= 1e-4. Argmax tokens, N and commit slots: bit-exact, except
positions whose top-2 logit gap (oracle, fp64) is below 1e-3 (token excluded) and
sequences where a position the acceptance scan examines has |p - tau| < 1e-4 (N and that
sequence's commit slots excluded). Exclusions are counted and returned.
"""
import numpy as np

ATTN_TOL = 1e-2
MAXPROB_TOL = 1e-4
GAP_EXCLUDE = 1e-3
TAU_EXCLUDE = 1e-4


def assert_attn_close(got, ref, what="attention"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref).max() if got.size else 0.0
    assert err <= ATTN_TOL, f"{what}: max-abs error {err:.3e} > {ATTN_TOL}"
    return err


def scanned_ambiguous(p_ref_row, tau):
    """True when a position the left-to-right scan examines lies within TAU_EXCLUDE of
    tau (the scan examines positions up to and including the first one below tau)."""
    t = float(np.float32(tau))
    for p in p_ref_row:
        if abs(p - t) < TAU_EXCLUDE:
            return True
        if p < t:
            return False
    return False


def compare_head(tok, p, n, tok_ref, p_ref, n_ref, gap_ref, tau):
    """tok/p: [b, B]; n: [b]; tau: one threshold, or one per sequence. Returns counts of
    excluded tokens and sequences."""
    tok, p, n = np.asarray(tok), np.asarray(p, np.float64), np.asarray(n)
    taus = np.broadcast_to(np.asarray(tau, dtype=np.float64), (len(n),))
    err = np.abs(p - p_ref).max()
    assert err <= MAXPROB_TOL, f"maxprob max-abs error {err:.3e} > {MAXPROB_TOL}"
    tie = gap_ref < GAP_EXCLUDE
    bad = (tok != tok_ref) & ~tie
    assert not bad.any(), f"argmax mismatch at {np.argwhere(bad)[:8].tolist()}"
    amb = np.array([scanned_ambiguous(p_ref[s], taus[s]) for s in range(len(n))], dtype=bool)
    badn = (n != n_ref) & ~amb
    assert not badn.any(), f"N mismatch at {np.flatnonzero(badn)[:8].tolist()}: " \
                           f"{n[badn][:8].tolist()} vs {n_ref[badn][:8].tolist()}"
    return {"tokens_excluded": int(tie.sum()), "seqs_excluded": int(amb.sum()),
            "maxprob_err": float(err)}
