"""Comparison rules between the CUDA path and the fp64 oracle.

Attention outputs: max-abs error <= 1e-2 against the oracle run on the same bf16-rounded
inputs. Max-probs: |delta| <= 1e-4. Argmax tokens, N and commit slots: bit-exact, except
positions whose top-2 logit gap (oracle, fp64) is below 1e-3 (token excluded) and
sequences where a position the acceptance scan examines has |p - tau| < 1e-4, for
0 < tau <= 1 (N and that sequence's commit slots excluded). Exclusions are counted and returned.

Gradients are compared element by element against a bound from an error model of the
kernels' arithmetic (product_error_bound below), not by a norm.
"""
import math

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
    tau (the scan examines positions up to and including the first one below tau). A
    max-prob lies in (0, 1], so with tau <= 0 every position is accepted and with tau > 1
    none is, on either side: no position is ambiguous then."""
    t = float(np.float32(tau))
    if t <= 0.0 or t > 1.0:
        return False
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


# ------------------------------------------------------------ gradient error model
#
# Every gradient output the kernels produce is a sum of products y_c = sum_j a_j b_jc in
# which one factor (a: P, dS or dlogits) is rounded to bf16 before a tensor-core product
# with fp32 accumulation; the other factor (b: K, Q, dO, W or h) is bf16 input data and
# exact. Per element, the error of y_c is bounded by three terms:
#   1. bf16 rounding of a_j: a_j (1 + d_j), |d_j| <= u = 2^-8 (8 significant bits, round
#      to nearest even: half the spacing 2^-7 of bf16 values in [1, 2)). With r such
#      roundings on the way to a_j (r = 2 for dS, which the kernels form from the already
#      rounded P and round again; r = 1 for P and dlogits), the worst case is
#      |error| <= r u S1, S1 = sum_j |a_j| |b_jc|. With the roundings independent and
#      zero-mean, Hoeffding's inequality over the r n bounded terms gives
#      |error| <= 7 sqrt(r) u S2, S2 = sqrt(sum_j a_j^2 b_jc^2), except with probability
#      2 exp(-49/2) = 4.6e-11 per element. The bound takes the smaller of the two.
#   2. fp32 accumulation: m = n/16 + 16 + extra roundings of partial sums no larger than
#      S1 (one per K = 16 MMA step, up to 16 inside a step, plus the atomic adds of the
#      query heads of a kv group); independent errors of at most 2^-24 relative give
#      7 * 2^-24 / sqrt(3) * sqrt(m) * S1 by the same argument.
#   3. upstream fp32 error of a_j before its rounding. Attention (P, dS): the fp32 scores
#      S = Q K^T (d = 128: about 2e-5 relative at the largest |q||k| scale of N(0,1)
#      inputs, 7 sigma), the row statistics and ex2.approx stay below 2^-14 |a_j| (a
#      margin of three), and dS = P (dP - D) also carries 2^-14 P (|dP| + |D|) for the
#      cancelling difference: 2^-14 * (S1 + S3), S3 = sum_j P_j (|dP_j| + |D|) |b_jc|.
#      LM head (dlogits = (p - onehot) / N): p = exp(l - lse) carries the relative error
#      of the fp32 logits, logit_rel_error below, applied to |p| / N.

U_BF16 = 2.0 ** -8
U_F32 = 2.0 ** -24
UPSTREAM_REL = 2.0 ** -14


def product_error_bound(a_abs_b, a2_b2, n, upstream=None, extra_roundings=0, roundings=1):
    """Element-wise bound of the model above from S1 = |a| @ |b| (a_abs_b), the sum of
    squares S2^2 = a^2 @ b^2 (a2_b2), the contraction length n and the number r of bf16
    roundings of a (`roundings`); `upstream` is the absolute upstream term beyond
    2^-14 * S1 (attention: 2^-14 * S3), or None."""
    s1 = np.asarray(a_abs_b, dtype=np.float64)
    s2 = np.sqrt(np.asarray(a2_b2, dtype=np.float64))
    m = n / 16.0 + 16.0 + extra_roundings
    bound = np.minimum(roundings * U_BF16 * s1, 7.0 * math.sqrt(roundings) * U_BF16 * s2)
    bound = bound + (7.0 * U_F32 / math.sqrt(3.0) * math.sqrt(m) + UPSTREAM_REL) * s1
    if upstream is not None:
        bound = bound + np.asarray(upstream, dtype=np.float64)
    return bound + 1e-12


def logit_rel_error(h_rows, w):
    """Upstream relative error of softmax(l)_v = exp(l_v - lse) for LM-head rows h_rows
    [R, H] and W [V, H]: the fp32 logits accumulate H bf16 products (m = H/16 + 16
    roundings, each at most 2^-24 of a partial sum bounded by sum_d |h_d||w_vd|, which
    Cauchy-Schwarz bounds by |h|_2 max_v |w_v|_2), 7 sigma as in term 2, once for l_v and
    once for lse. Returns [R]."""
    H = h_rows.shape[1]
    m = H / 16.0 + 16.0
    wmax = float(np.sqrt((w * w).sum(axis=1)).max())
    hn = np.sqrt((h_rows * h_rows).sum(axis=1))
    return 2.0 * 7.0 * U_F32 / math.sqrt(3.0) * math.sqrt(m) * hn * wmax


def assert_within_bound(got, ref, bound, what):
    """|got - ref| <= bound for every element; reports the worst ratio."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - np.asarray(ref, dtype=np.float64))
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    ratio = err / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    if worst > 1.0:
        idx = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
        raise AssertionError(f"{what}: error {err[idx]:.3e} > bound {bound[idx]:.3e} at "
                             f"{tuple(int(i) for i in idx)} ({int((ratio > 1).sum())} "
                             f"elements over)")
    return worst
