"""The work counts behind bench.py's roofline figures, checked on the CPU.

`achieved` in every roofline object is algorithmic work divided by measured time, so the
work formulas are part of the measurement. These tests tie each formula to something it
does not restate: the visible pairs of the oracle's explicit mask M (the dual-stream
flop count), and the sizes of the tensors a decode call actually reads and writes (the
decode-attention byte count and the LM-head flop count).
"""
import dataclasses
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from block_masked_token_gb300 import workloads as W  # noqa: E402


def _dual_configs():
    return [c for c in W.CONFIGS.values() if isinstance(c, W.DualStreamConfig)]


@pytest.mark.parametrize("L,B", [(8, 1), (8, 2), (8, 8), (12, 4), (32, 16), (64, 4)])
def test_dual_flops_count_the_visible_pairs_of_M(L, B):
    """4 d flop (QK^T and PV) per visible (query, key) pair of M, per (batch, head)."""
    base = _dual_configs()[0]
    cfg = dataclasses.replace(base, L=L, B=B)
    visible = int(oracle.mask_M(L, B).sum())
    assert bench.dual_flops(cfg) == 4.0 * cfg.d * visible * cfg.batch * cfg.hq


@pytest.mark.parametrize("L,B", [(10, 4), (10, 3), (9, 4), (7, 2), (16, 16), (13, 1)])
def test_every_row_of_M_sees_t_plus_one_keys(L, B):
    """Why the closed form L(L+1) needs no B | L: row t of either stream sees t + 1 keys
    (a masked row: the bs clean keys before its block start plus the t - bs + 1 masked keys
    of its block up to itself), also with a short last block."""
    rows = oracle.mask_M(L, B).sum(axis=1)
    t = list(range(L))
    assert [int(x) for x in rows[:L]] == [i + 1 for i in t]
    assert [int(x) for x in rows[L:]] == [i + 1 for i in t]
    cfg = dataclasses.replace(_dual_configs()[0], L=L, B=B)
    assert bench.dual_flops(cfg) == 4.0 * cfg.d * L * (L + 1) * cfg.batch * cfg.hq


def test_decode_bytes_and_head_flops_match_the_tensors():
    cfg = W.TINY_DECODE
    inp = W.make_decode_inputs(cfg, seed=0, device="cpu")
    q, kb, vb, h, w = inp.q[0], inp.k_blk[0], inp.v_blk[0], inp.h[0], inp.w
    lens = inp.prefix_lens.tolist()
    # one K and one V row of the pool per committed position and KV head
    row_bytes = inp.k_pool[0, :, 0, :].numel() * inp.k_pool.element_size()
    prefix = 2 * sum(lens) * row_bytes
    blocks = (kb.numel() + vb.numel()) * kb.element_size()
    o_bytes = q.numel() * 4                      # O is fp32 with Q's shape
    want = prefix + blocks + q.numel() * q.element_size() + o_bytes
    assert bench.decode_kv_bytes(lens, cfg) == want
    assert bench.head_flops(cfg) == 2.0 * h.shape[0] * h.shape[1] * w.shape[0]


def test_loss_flops_cover_both_streams():
    cfg = W.CE_LOSS_7B
    rows = cfg.batch * 2 * cfg.L
    assert bench.ce_flops(cfg) == 2.0 * rows * cfg.hidden * cfg.vocab


def test_gradient_work_is_two_and_a_half_forwards():
    """The gradient's algorithmic work: S again, dP, dV, dK, dQ (five products) against the
    forward's two, per visible pair."""
    cfg = W.DUAL_STREAM_7B
    assert torch.isclose(torch.tensor(2.5 * bench.dual_flops(cfg)),
                         torch.tensor(10.0 * cfg.d * cfg.L * (cfg.L + 1) * cfg.batch * cfg.hq))


def test_clock_summary_reads_reasons_and_median():
    """The clock record that decides whether a run is kept: median SM clock over the
    samples, the maximum clock, and every throttle reason seen Active at least once."""
    clk = bench.ClockSampler(0)
    clk.lines = [
        "2070, 2070, 900.1, Not Active, Not Active, Not Active, Not Active",
        "1980, 2070, 1390.0, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 1200.5, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "[N/A], 2070, 0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = clk.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    clk.lines = ["1400, 2070, 1000, Active, Not Active, Active, Not Active"]
    assert bench.ClockSampler.summary(clk)["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_peaks_come_from_the_measured_file_else_the_fallback(tmp_path, monkeypatch):
    """The roofline denominators: the measured copy bandwidth and bf16 rates when the
    measured-peaks file is present, else the fallback figures, labelled as such."""
    import json
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    fb = bench.load_peaks()
    assert fb["source"] == "fallback"
    assert (fb["hbm_gbs"], fb["bf16_tflops"], fb["bf16_tflops_sustained"]) == (6800.0, 1900.0, 1700.0)
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6795.1, "bf16_tflops": 1906.6, "bf16_tflops_sustained": 1687.3}))
    m = bench.load_peaks()
    assert m["source"] == "measured"
    assert (m["hbm_gbs"], m["bf16_tflops"], m["bf16_tflops_sustained"]) == (6795.1, 1906.6, 1687.3)
