"""Seeded synthetic inputs for QUOKA chunk attention.

This module only draws random tensors; it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle can take their inputs
from it.  Every draw comes from ``numpy.random.default_rng`` (PCG64) with a
fixed seed sequence, so the same bits come out on every machine.

Two value recipes are used:

* ``iid_outliers`` (the tiny multi-head fp32 case): Q, K, V are i.i.d.
  N(0, 1).  Four query positions per head are outliers: a random unit
  vector scaled to norm 3*sqrt(d) is added (a shift of about 3 sigma per
  coordinate).  Eight history keys per head are planted needles: a copy of
  one of that head's outlier queries plus N(0, 0.1) noise (variance 0.1).
* ``massive_act`` (the Llama-shaped GQA cases): keys are N(0, 1) plus a bias
  on 4 random channels per KV head, each bias drawn from N(0, 4) (std 2) and
  constant over positions.  Queries are N(0, 1) plus 4 times a random unit
  direction per query head; 5% of the chunk positions (shared by all heads)
  replace that shared direction with a random unit direction of their own.
  Values are N(0, 1).  32 needles per KV head: the history key becomes a
  copy of an outlier query of one of the group's heads, plus N(0, 0.1)
  noise, plus the head's channel bias.

Tensors are returned as torch CPU tensors in the storage dtype (float32 or
bfloat16, rounded to nearest-even from the float32 draws).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class ChunkConfig:
    """One chunk of chunked prefill: C queries over T cached history keys."""
    name: str
    H_q: int
    H_kv: int
    d: int
    C: int
    T: int
    N_q: int
    B: int
    dtype: str            # "fp32" or "bf16"
    recipe: str           # "iid_outliers" or "massive_act"

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16


# The single-chunk workloads.
TINY_MHA_FP32 = ChunkConfig("mha4_d64_C128_T1024_fp32", 4, 4, 64, 128, 1024, 16, 256,
                            "fp32", "iid_outliers")
GQA_32K_BF16 = ChunkConfig("gqa32x8_d128_C2048_T32768_bf16", 32, 8, 128, 2048, 32768, 64, 2048,
                           "bf16", "massive_act")
GQA_128K_BF16 = ChunkConfig("gqa32x8_d128_C4096_T131072_bf16", 32, 8, 128, 4096, 131072, 128, 4096,
                            "bf16", "massive_act")
# Decode: one new token per step (C = 1), so the one query is the selected set.
DECODE_32K_BF16 = ChunkConfig("decode_gqa32x8_d128_C1_T32768_bf16", 32, 8, 128, 1, 32768, 1, 2048,
                              "bf16", "massive_act")


@dataclass(frozen=True)
class SweepConfig:
    """A whole prompt split into equal chunks processed in order."""
    name: str
    H_q: int
    H_kv: int
    d: int
    total: int
    C: int
    N_q: int
    B: int
    dtype: str = "bf16"

    @property
    def n_chunks(self) -> int:
        return self.total // self.C


SWEEP_64K_BF16 = SweepConfig("sweep_gqa32x8_d128_64k_C2048_bf16", 32, 8, 128, 65536, 2048, 64, 2048)


@dataclass(frozen=True)
class RaggedConfig:
    """A batch of sequences, one chunk each, over histories of different lengths."""
    name: str
    n_seq: int
    H_q: int
    H_kv: int
    d: int
    C: int
    T_min: int
    T_max: int
    N_q: int
    B: int
    dtype: str = "bf16"

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv


RAGGED_8x_BF16 = RaggedConfig("ragged8_gqa64x8_d128_C1024_T4k-64k_bf16", 8, 64, 8, 128, 1024,
                              4096, 65536, 64, 2048)


@dataclass
class ChunkInputs:
    """Tensors of one chunk plus the generator's bookkeeping (outliers, needles)."""
    Q: torch.Tensor          # [H_q, C, d]
    K_hist: torch.Tensor     # [H_kv, T, d]
    V_hist: torch.Tensor     # [H_kv, T, d]
    K_chunk: torch.Tensor    # [H_kv, C, d]
    V_chunk: torch.Tensor    # [H_kv, C, d]
    outliers: np.ndarray     # [H_q, n_out] chunk positions of outlier queries per head
    needles: list = field(default_factory=list)   # (g, t, h, c): key t of KV head g copies Q[h, c]


def _to_storage(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t if dtype == "fp32" else t.to(torch.bfloat16)


def _unit_rows(rng: np.random.Generator, shape) -> np.ndarray:
    v = rng.standard_normal(shape)
    return v / np.linalg.norm(v, axis=-1, keepdims=True)


def _iid_outliers(cfg: ChunkConfig, seed: int) -> ChunkInputs:
    rng = np.random.default_rng([seed, 0])
    H, C, T, d = cfg.H_q, cfg.C, cfg.T, cfg.d
    Q = rng.standard_normal((H, C, d), dtype=np.float32)
    K = rng.standard_normal((H, T, d), dtype=np.float32)
    V = rng.standard_normal((H, T, d), dtype=np.float32)
    Kc = rng.standard_normal((H, C, d), dtype=np.float32)
    Vc = rng.standard_normal((H, C, d), dtype=np.float32)
    n_out = min(4, C)
    outliers = np.stack([np.sort(rng.choice(C, n_out, replace=False)) for _ in range(H)])
    shift = 3.0 * math.sqrt(d) * _unit_rows(rng, (H, n_out, d))
    for h in range(H):
        Q[h, outliers[h]] += shift[h].astype(np.float32)
    needles = []
    n_needle = min(8, T)
    for h in range(H):
        pos = rng.choice(T, n_needle, replace=False) if T else []
        for j, t in enumerate(pos):
            c = int(outliers[h, j % n_out])
            K[h, t] = Q[h, c] + rng.normal(0.0, math.sqrt(0.1), d).astype(np.float32)
            needles.append((h, int(t), h, c))
    return ChunkInputs(_to_storage(Q, cfg.dtype), _to_storage(K, cfg.dtype), _to_storage(V, cfg.dtype),
                       _to_storage(Kc, cfg.dtype), _to_storage(Vc, cfg.dtype), outliers, needles)


def _massive_act_statics(rng: np.random.Generator, H_q: int, H_kv: int, d: int):
    """Per-KV-head channel bias (4 channels, N(0,4)) and per-query-head mean direction."""
    bias = np.zeros((H_kv, d), dtype=np.float32)
    for g in range(H_kv):
        ch = rng.choice(d, 4, replace=False)
        bias[g, ch] = rng.normal(0.0, 2.0, 4)
    m_hat = _unit_rows(rng, (H_q, d)).astype(np.float32)
    return bias, m_hat


def _massive_act_queries(rng: np.random.Generator, H_q: int, C: int, d: int, m_hat: np.ndarray):
    Q = rng.standard_normal((H_q, C, d), dtype=np.float32)
    n_out = int(round(0.05 * C))
    out_pos = np.sort(rng.choice(C, n_out, replace=False))
    direction = np.broadcast_to(m_hat[:, None, :], (H_q, C, d)).copy()
    direction[:, out_pos, :] = _unit_rows(rng, (H_q, n_out, d))
    Q += 4.0 * direction
    return Q, out_pos


def _plant_needles(rng, K, bias, Q, out_pos, H_q, H_kv, T_limit, count=32):
    """Overwrite `count` history keys per KV head (positions < T_limit) with noisy outlier queries."""
    G = H_q // H_kv
    d = K.shape[-1]
    needles = []
    n = min(count, T_limit)
    if n == 0 or len(out_pos) == 0:
        return needles
    for g in range(H_kv):
        pos = rng.choice(T_limit, n, replace=False)
        for t in pos:
            h = g * G + int(rng.integers(G))
            c = int(out_pos[int(rng.integers(len(out_pos)))])
            K[g, t] = Q[h, c] + rng.normal(0.0, math.sqrt(0.1), d).astype(np.float32) + bias[g]
            needles.append((g, int(t), h, c))
    return needles


def _massive_act(cfg: ChunkConfig, seed: int) -> ChunkInputs:
    rng = np.random.default_rng([seed, 1])
    H_q, H_kv, C, T, d = cfg.H_q, cfg.H_kv, cfg.C, cfg.T, cfg.d
    bias, m_hat = _massive_act_statics(rng, H_q, H_kv, d)
    Q, out_pos = _massive_act_queries(rng, H_q, C, d, m_hat)
    K = rng.standard_normal((H_kv, T, d), dtype=np.float32)
    K += bias[:, None, :]
    V = rng.standard_normal((H_kv, T, d), dtype=np.float32)
    Kc = rng.standard_normal((H_kv, C, d), dtype=np.float32) + bias[:, None, :]
    Vc = rng.standard_normal((H_kv, C, d), dtype=np.float32)
    needles = _plant_needles(rng, K, bias, Q, out_pos, H_q, H_kv, T)
    outliers = np.broadcast_to(out_pos, (H_q, len(out_pos))).copy()
    return ChunkInputs(_to_storage(Q, cfg.dtype), _to_storage(K, cfg.dtype), _to_storage(V, cfg.dtype),
                       _to_storage(Kc, cfg.dtype), _to_storage(Vc, cfg.dtype), outliers, needles)


def make_chunk(cfg: ChunkConfig, seed: int = 0) -> ChunkInputs:
    """Draw one chunk's tensors for `cfg` (see the module docstring for the recipes)."""
    if cfg.recipe == "iid_outliers":
        return _iid_outliers(cfg, seed)
    if cfg.recipe == "massive_act":
        return _massive_act(cfg, seed)
    raise ValueError(f"unknown recipe {cfg.recipe!r}")


@dataclass
class SweepInputs:
    """A whole prompt: per-chunk queries and the K/V of every position."""
    Q: list                 # n_chunks tensors [H_q, C, d]
    K_all: torch.Tensor     # [H_kv, total, d]
    V_all: torch.Tensor     # [H_kv, total, d]
    outliers: list          # per chunk: positions (within the chunk) of the outlier queries
    needles: list           # per chunk: (g, t, h, c) planted for that chunk's queries


def make_sweep(cfg: SweepConfig, seed: int = 0) -> SweepInputs:
    """Draw a whole prompt for chunked prefill with the ``massive_act`` recipe.

    Chunk i's keys and values are what chunk i appends to the cache; needles
    for chunk i's outlier queries are planted at positions earlier than
    i*C (a later chunk's needle may overwrite an earlier one's).
    """
    rng0 = np.random.default_rng([seed, 3])
    bias, m_hat = _massive_act_statics(rng0, cfg.H_q, cfg.H_kv, cfg.d)
    K = np.empty((cfg.H_kv, cfg.total, cfg.d), dtype=np.float32)
    V = np.empty((cfg.H_kv, cfg.total, cfg.d), dtype=np.float32)
    Qs, outs, needles = [], [], []
    for i in range(cfg.n_chunks):
        rng = np.random.default_rng([seed, 3, i])
        Q, out_pos = _massive_act_queries(rng, cfg.H_q, cfg.C, cfg.d, m_hat)
        sl = slice(i * cfg.C, (i + 1) * cfg.C)
        K[:, sl] = rng.standard_normal((cfg.H_kv, cfg.C, cfg.d), dtype=np.float32) + bias[:, None, :]
        V[:, sl] = rng.standard_normal((cfg.H_kv, cfg.C, cfg.d), dtype=np.float32)
        needles.append(_plant_needles(rng, K, bias, Q, out_pos, cfg.H_q, cfg.H_kv, i * cfg.C))
        Qs.append(_to_storage(Q, cfg.dtype))
        outs.append(out_pos)
    return SweepInputs(Qs, _to_storage(K, cfg.dtype), _to_storage(V, cfg.dtype), outs, needles)


def ragged_history_lengths(cfg: RaggedConfig, seed: int = 0) -> list:
    """History length per sequence, log-uniform in [T_min, T_max]."""
    rng = np.random.default_rng([seed, 4])
    u = rng.uniform(math.log(cfg.T_min), math.log(cfg.T_max), cfg.n_seq)
    return [int(math.floor(math.exp(x))) for x in u]


def make_ragged(cfg: RaggedConfig, seed: int = 0) -> list:
    """One ChunkInputs per sequence (``massive_act`` recipe, own history length each)."""
    out = []
    for s, T in enumerate(ragged_history_lengths(cfg, seed)):
        sub = ChunkConfig(f"{cfg.name}[{s}]", cfg.H_q, cfg.H_kv, cfg.d, cfg.C, T, cfg.N_q, cfg.B,
                          cfg.dtype, "massive_act")
        out.append(_massive_act(sub, seed * 1000 + 17 + s))
    return out


def small_chunk(H_q=4, H_kv=2, d=64, C=64, T=300, N_q=8, B=40, dtype="fp32",
                recipe="massive_act", seed=0) -> tuple:
    """A small case for tests: returns (cfg, inputs)."""
    cfg = ChunkConfig(f"small_{H_q}x{H_kv}_d{d}_C{C}_T{T}_{dtype}", H_q, H_kv, d, C, T, N_q, B, dtype, recipe)
    return cfg, make_chunk(cfg, seed)


def pack_varlen(seqs: list) -> dict:
    """Concatenate per-sequence ChunkInputs sequence-major, the layout of the
    ragged entry point: each sequence's tensors flattened in their own
    [heads, length, d] order, one after another.  Returns the host prefix sums
    cu_T, cu_C (lists of nseq + 1 ints) and the packed 1-D tensors."""
    cu_T, cu_C = [0], [0]
    for x in seqs:
        cu_T.append(cu_T[-1] + x.K_hist.shape[1])
        cu_C.append(cu_C[-1] + x.Q.shape[1])
    cat = lambda name: torch.cat([getattr(x, name).reshape(-1) for x in seqs])
    return dict(cu_T=cu_T, cu_C=cu_C, Q=cat("Q"), K_hist=cat("K_hist"), V_hist=cat("V_hist"),
                K_chunk=cat("K_chunk"), V_chunk=cat("V_chunk"))
