"""Seeded synthetic inputs for the MARS hot path.

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic (no mask, softmax, acceptance or commit), so it can feed both the CUDA path
and the CPU oracle. The paper's own workloads (Qwen2.5-0.5B / 7B weights on six public
benchmarks, GSM8K for the wall-clock runs) are not available; these inputs stand in for
them with the models' attention and LM-head shapes.

Recipe (every draw from one torch.Generator seeded with `seed`, in this order):
  decode: prefix lengths (integer uniform, inclusive bounds); page permutation of the
  pool; then per step: Q, K_blk, V_blk ~ N(0,1); then prefix K pool, V pool ~ N(0,1);
  then per step: h-scales s = exp(U[ln 0.5, ln 8]) per (sequence, position) and
  h = s * N(0,1); last the LM head W ~ N(0, 1/H) stored vocabulary-major [V, H].
  dual-stream: Q, K, V ~ N(0,1).
All values are rounded to bf16 (round-to-nearest-even) before either side sees them.
On device='cuda' the same recipe runs on a CUDA generator (a different random stream
from the CPU one, same distributions); it is used where CPU generation of gigabytes of
input would dominate the run.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class DualStreamConfig:
    name: str
    batch: int
    L: int
    B: int
    hq: int
    hkv: int
    d: int


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    prefix_lo: int
    prefix_hi: int
    B: int
    hq: int
    hkv: int
    d: int
    hidden: int
    vocab: int
    taus: tuple = (0.9,)
    steps: int = 1
    page_size: int = 16
    prefixes: tuple | None = None      # explicit prefix lengths (overrides lo/hi)
    tau_period: int = 16               # steps per entry of `taus`

    def tau_at(self, step: int) -> float:
        return self.taus[(step // self.tau_period) % len(self.taus)]


TINY_DECODE = DecodeConfig("tiny_decode_b2_B4", batch=2, prefix_lo=37, prefix_hi=50,
                           prefixes=(37, 50), B=4, hq=4, hkv=2, d=64, hidden=256,
                           vocab=512, taus=(0.9,))
DUAL_STREAM_0P5B = DualStreamConfig("dual_stream_0.5b_b4_2L1024_B4", batch=4, L=512, B=4,
                                    hq=14, hkv=2, d=64)
DECODE_7B = DecodeConfig("decode_7b_b32_B8", batch=32, prefix_lo=512, prefix_hi=2048, B=8,
                         hq=28, hkv=4, d=128, hidden=3584, vocab=152064, taus=(0.9,))
DUAL_STREAM_7B = DualStreamConfig("dual_stream_7b_b2_2L8192_B16", batch=2, L=4096, B=16,
                                  hq=28, hkv=4, d=128)
SUSTAINED_DECODE_7B = DecodeConfig("sustained_decode_7b_b128_B16_64steps", batch=128,
                                   prefix_lo=2048, prefix_hi=8192, B=16, hq=28, hkv=4,
                                   d=128, hidden=3584, vocab=152064,
                                   taus=(1.0, 0.95, 0.9, 0.8), steps=64, tau_period=16)

@dataclass(frozen=True)
class CELossConfig:
    name: str
    batch: int
    L: int
    hidden: int
    vocab: int


# The training loss over the dual stream at the 7B head shape, with the stream length of
# the 7B dual-stream attention workload.
CE_LOSS_7B = CELossConfig("ce_loss_7b_b2_L4096", batch=2, L=4096, hidden=3584, vocab=152064)


def make_ce_inputs(cfg: CELossConfig, seed: int = 0, device=None):
    """Hidden states, head and targets for the dual-stream loss. Draw order: h = s * N(0,1)
    with s = exp(U[ln 0.5, ln 8]) per row; W ~ N(0, 1/H) [V, H]; targets uniform in
    [0, V) for every row, then -1 for the last clean row of each sequence (it has no next
    token). Every masked row carries a target (the masked set is the whole masked stream).
    Everything bf16 except the int32 targets."""
    dev = torch.device(device) if device is not None else torch.device("cpu")
    g = torch.Generator(device=dev).manual_seed(seed)
    rows = cfg.batch * 2 * cfg.L
    s = torch.exp(math.log(0.5) + (math.log(8.0) - math.log(0.5)) *
                  torch.rand(rows, 1, generator=g, device=dev))
    h = (torch.randn(rows, cfg.hidden, generator=g, device=dev) * s).to(torch.bfloat16)
    w = (torch.randn(cfg.vocab, cfg.hidden, generator=g, device=dev) /
         math.sqrt(cfg.hidden)).to(torch.bfloat16)
    y = torch.randint(0, cfg.vocab, (rows,), generator=g, device=dev, dtype=torch.int64)
    y = y.to(torch.int32)
    y.view(cfg.batch, 2 * cfg.L)[:, cfg.L - 1] = -1
    return {"h": h, "w": w, "targets": y}


# The KV-cached autoregressive step on the same sequences (one query per sequence, one
# token per step): the same kernels with B = 1 and tau = 1.0. The prefix lengths are the
# first draw of the generator, so with the same seed they equal the sustained workload's.
AR_DECODE_7B = DecodeConfig("ar_decode_7b_b128_B1_64steps", batch=128, prefix_lo=2048,
                            prefix_hi=8192, B=1, hq=28, hkv=4, d=128, hidden=3584,
                            vocab=152064, taus=(1.0,), steps=64, tau_period=16)

CONFIGS = {c.name: c for c in (TINY_DECODE, DUAL_STREAM_0P5B, DECODE_7B, DUAL_STREAM_7B,
                               SUSTAINED_DECODE_7B, AR_DECODE_7B, CE_LOSS_7B)}


def _gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev.type if dev.type == "cpu" else dev)
    g.manual_seed(seed)
    return g


def _randn(g, shape, device, scale: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def make_dual_stream_inputs(cfg: DualStreamConfig, seed: int = 0, device="cpu"):
    """Q [b, 2L, Hq, D], K and V [b, 2L, Hkv, D], bf16, contiguous."""
    g = _gen(seed, device)
    n = 2 * cfg.L
    q = _randn(g, (cfg.batch, n, cfg.hq, cfg.d), device)
    k = _randn(g, (cfg.batch, n, cfg.hkv, cfg.d), device)
    v = _randn(g, (cfg.batch, n, cfg.hkv, cfg.d), device)
    return {"q": q, "k": k, "v": v}


@dataclass
class DecodeInputs:
    prefix_lens: torch.Tensor          # int32 [b], the committed prefix before step 0
    block_table: torch.Tensor          # int32 [b, max_pages], -1 past the mapped pages
    num_pages: int
    k_pool: torch.Tensor               # bf16 [num_pages, Hkv, page_size, D]
    v_pool: torch.Tensor
    q: list = field(default_factory=list)       # per step bf16 [b, B, Hq, D]
    k_blk: list = field(default_factory=list)   # per step bf16 [b, B, Hkv, D]
    v_blk: list = field(default_factory=list)
    h: list = field(default_factory=list)       # per step bf16 [b*B, H]
    w: torch.Tensor | None = None               # bf16 [V, H]


def pages_needed(prefix: int, B: int, steps: int, page_size: int) -> int:
    """Pages a sequence must have mapped to commit up to B tokens on each of `steps`
    steps (allocation is the caller's job; this is the caller-side sizing)."""
    return -(-(prefix + B * steps) // page_size)


def make_decode_inputs(cfg: DecodeConfig, seed: int = 0, device="cpu", steps: int | None = None,
                       with_head: bool = True, extra_pages: int = 0) -> DecodeInputs:
    steps = cfg.steps if steps is None else steps
    g = _gen(seed, device)
    if cfg.prefixes is not None:
        prefix = torch.tensor(cfg.prefixes, dtype=torch.int32)
        if prefix.numel() != cfg.batch:
            raise ValueError("explicit prefixes must have one entry per sequence")
    else:
        prefix = torch.randint(cfg.prefix_lo, cfg.prefix_hi + 1, (cfg.batch,), generator=g,
                               device=device, dtype=torch.int64).to(torch.int32).cpu()
    need = [pages_needed(int(p), cfg.B, steps, cfg.page_size) for p in prefix.tolist()]
    max_pages = max(need)
    num_pages = sum(need) + extra_pages
    perm = torch.randperm(num_pages, generator=g, device=device).to(torch.int32).cpu()
    table = torch.full((cfg.batch, max_pages), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(need):
        table[s, :n] = perm[off:off + n]
        off += n
    inp = DecodeInputs(prefix_lens=prefix, block_table=table, num_pages=num_pages,
                       k_pool=None, v_pool=None)
    for _ in range(steps):
        inp.q.append(_randn(g, (cfg.batch, cfg.B, cfg.hq, cfg.d), device))
        inp.k_blk.append(_randn(g, (cfg.batch, cfg.B, cfg.hkv, cfg.d), device))
        inp.v_blk.append(_randn(g, (cfg.batch, cfg.B, cfg.hkv, cfg.d), device))
    pool_shape = (num_pages, cfg.hkv, cfg.page_size, cfg.d)
    inp.k_pool = _randn(g, pool_shape, device)
    inp.v_pool = _randn(g, pool_shape, device)
    if with_head:
        lo, hi = math.log(0.5), math.log(8.0)
        for _ in range(steps):
            u = torch.rand(cfg.batch * cfg.B, 1, generator=g, device=device)
            s = torch.exp(lo + (hi - lo) * u)
            x = torch.randn(cfg.batch * cfg.B, cfg.hidden, generator=g, device=device)
            inp.h.append((x * s).to(torch.bfloat16))
        inp.w = _randn(g, (cfg.vocab, cfg.hidden), device, scale=1.0 / math.sqrt(cfg.hidden))
    return inp


def to_f64(t: torch.Tensor):
    """bf16 (or any) tensor -> float64 numpy array on the host, exactly."""
    return t.detach().to("cpu", torch.float64).numpy()
