"""Seeded synthetic inputs for the gated-prefill path.

This module is the single source of input bytes for both the CUDA path and the
CPU oracle. It holds none of the method's arithmetic: it draws random numbers,
rounds them to bf16 storage and lays them out. Nothing here scores, selects,
gathers or attends.

Workload shapes follow the Qwen3-1.7B long-context prefill the TokenGate pages
describe (TokenGate deep dive, agientry.com, section 4 "Evidence across tasks
and architectures": Qwen3-1.7B, NIAH 16k-128k; section 4.2 "Length
extrapolation", Table 1). The datasets themselves (RepoBench-P,
2WikiMultihopQA, MultiNews, BioDEX, NIAH) are not used: seeded Gaussian hidden
states with a heavy-tailed fraction of rows stand in for them.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np


# ---------------------------------------------------------------------------
# bf16 storage helpers (storage format only, no method arithmetic)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return uint16 bits.
    A NaN stays a NaN (quiet, same sign): rounding its payload could carry into +-inf."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounding = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    out = ((u + rounding) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(f)
    out[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x0040)).astype(np.uint16)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns exactly to fp32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns exactly to fp64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------------------
# Workload descriptions
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one synthetic gated-prefill batch."""

    name: str
    doc_lens: tuple           # prunable document tokens per sequence
    instr_lens: tuple         # non-prunable instruction tokens per sequence
    d: int                    # gate-layer width (d_model)
    d_g: int                  # score-MLP hidden width
    H_q: int
    H_kv: int
    d_h: int
    K: int                    # default budget
    budgets: tuple = ()       # budget sweep (empty: just K)
    seed: int = 1234
    instr_where: str = "last"  # "last" | "first" | "scattered"
    fixed_tau_beta: Optional[float] = None  # tau = beta = this value; else U(0.8, 1.2) per head
    heavy_frac: float = 0.0   # fraction of hidden-state rows scaled by heavy_scale
    heavy_scale: float = 4.0
    score_levels: int = 0     # >0: scores for selection are quantised to this many levels
    rope_theta: float = 1.0e6

    @property
    def B(self) -> int:
        return len(self.doc_lens)

    @property
    def seq_lens(self) -> List[int]:
        return [a + b for a, b in zip(self.doc_lens, self.instr_lens)]

    @property
    def T_total(self) -> int:
        return int(sum(self.seq_lens))

    def budgets_or_k(self) -> tuple:
        return self.budgets if self.budgets else (self.K,)


def _ragged_lengths(seed: int):
    rng = np.random.default_rng([seed, 7])
    docs = rng.integers(4096, 16384, size=8, endpoint=True)
    instr = rng.integers(64, 512, size=8, endpoint=True)
    return tuple(int(x) for x in docs), tuple(int(x) for x in instr)


_RAGGED_DOCS, _RAGGED_INSTR = _ragged_lengths(1234 + 3)

WORKLOADS = {
    # tiny case the oracle finishes in well under a second
    "tiny": Workload("tiny", (480,), (32,), d=256, d_g=64, H_q=4, H_kv=2, d_h=64, K=64,
                     seed=1234 + 0, fixed_tau_beta=1.0),
    # Qwen3-1.7B-shaped gate layer at 8K context
    "qwen3_1p7b_8k": Workload("qwen3_1p7b_8k", (8192,), (128,), d=2048, d_g=512, H_q=16, H_kv=8,
                              d_h=128, K=1024, seed=1234 + 1),
    # budget sweep at N = 32K: one gate pass serves several budgets
    "sweep_32k": Workload("sweep_32k", (32768,), (256,), d=2048, d_g=512, H_q=16, H_kv=8, d_h=128,
                          K=4096, budgets=(256, 1024, 4096, 16384), seed=1234 + 2,
                          heavy_frac=0.02, heavy_scale=4.0),
    # ragged batch of 8 with tie-heavy (256-level) scores
    "ragged_b8": Workload("ragged_b8", _RAGGED_DOCS, _RAGGED_INSTR, d=2048, d_g=512, H_q=16, H_kv=8,
                          d_h=128, K=2048, seed=1234 + 3, score_levels=256),
    # long context, 128K
    "long_128k": Workload("long_128k", (131072,), (512,), d=2048, d_g=512, H_q=16, H_kv=8, d_h=128,
                          K=8192, seed=1234 + 4),
}


def with_changes(wl: Workload, **kw) -> Workload:
    return dataclasses.replace(wl, **kw)


# ---------------------------------------------------------------------------
# Generators
# ---------------------------------------------------------------------------

_TAG_H, _TAG_W1, _TAG_W2, _TAG_HEAVY, _TAG_MASK, _TAG_TAU, _TAG_BETA = 11, 12, 13, 14, 15, 16, 17
_TAG_S, _TAG_Q, _TAG_K, _TAG_V, _TAG_G = 21, 22, 23, 24, 25
_TAG_W2H, _TAG_B2H, _TAG_GH = 31, 32, 33


def _rng(seed: int, tag: int, extra: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, tag, extra])


def cu_seqlens_of(lens: Sequence[int]) -> np.ndarray:
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return cu


def make_instr_mask(wl: Workload) -> np.ndarray:
    """uint8 [T_total], 1 on non-prunable (instruction / question) tokens."""
    mask = np.zeros(wl.T_total, dtype=np.uint8)
    cu = cu_seqlens_of(wl.seq_lens)
    for b in range(wl.B):
        n_doc, n_ins = wl.doc_lens[b], wl.instr_lens[b]
        start, end = int(cu[b]), int(cu[b + 1])
        if wl.instr_where == "last":
            mask[end - n_ins:end] = 1
        elif wl.instr_where == "first":
            mask[start:start + n_ins] = 1
        elif wl.instr_where == "scattered":
            where = _rng(wl.seed, _TAG_MASK, b).choice(end - start, size=n_ins, replace=False)
            mask[start + where] = 1
        else:
            raise ValueError(wl.instr_where)
        assert n_doc + n_ins == end - start
    return mask


def make_positions(wl: Workload) -> np.ndarray:
    """Original position ids: 0..N_b-1 within each sequence (int32 [T_total])."""
    pos = np.empty(wl.T_total, dtype=np.int32)
    cu = cu_seqlens_of(wl.seq_lens)
    for b in range(wl.B):
        pos[cu[b]:cu[b + 1]] = np.arange(cu[b + 1] - cu[b], dtype=np.int32)
    return pos


def make_gate_inputs(wl: Workload) -> dict:
    """Hidden states at the gate layer plus the score-MLP weights.

    h ~ N(0, 1) (a seeded fraction ``heavy_frac`` of rows scaled by ``heavy_scale``),
    W1 ~ N(0, 1/d), w2 ~ N(0, 1/d_g), all rounded to bf16; no biases.
    """
    T, d, d_g = wl.T_total, wl.d, wl.d_g
    h32 = _rng(wl.seed, _TAG_H).standard_normal((T, d), dtype=np.float32)
    if wl.heavy_frac > 0 and T > 0:
        n_heavy = int(round(wl.heavy_frac * T))
        rows = _rng(wl.seed, _TAG_HEAVY).choice(T, size=n_heavy, replace=False)
        h32[rows] *= np.float32(wl.heavy_scale)
    W1 = _rng(wl.seed, _TAG_W1).standard_normal((d_g, d), dtype=np.float32) * np.float32(1.0 / np.sqrt(d))
    w2 = _rng(wl.seed, _TAG_W2).standard_normal((d_g,), dtype=np.float32) * np.float32(1.0 / np.sqrt(d_g))
    return {
        "h": f32_to_bf16_bits(h32),
        "W1": f32_to_bf16_bits(W1),
        "w2": f32_to_bf16_bits(w2),
        "b1": None,
        "b2": 0.0,
        "instr_mask": make_instr_mask(wl),
        "cu_seqlens": cu_seqlens_of(wl.seq_lens),
        "pos": make_positions(wl),
    }


def make_gate_head_weights(wl: Workload, H_g: int) -> dict:
    """Second score layer with one row per gate head: W2 [H_g, d_g] ~ N(0, 1/d_g) in bf16 and a
    per-head bias b2 [H_g] ~ N(0, 0.1^2) in fp32."""
    W2 = _rng(wl.seed, _TAG_W2H, H_g).standard_normal((H_g, wl.d_g), dtype=np.float32)
    W2 *= np.float32(1.0 / np.sqrt(wl.d_g))
    b2 = (_rng(wl.seed, _TAG_B2H, H_g).standard_normal(H_g, dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    return {"W2": f32_to_bf16_bits(W2), "b2": b2}


def make_head_gates(wl: Workload, M: int, H_g: int, tag_extra: int = 0) -> np.ndarray:
    """Per-head gate values of M kept rows, g ~ U(0.02, 1) fp32 [M, H_g]."""
    return _rng(wl.seed, _TAG_GH, 100 * H_g + tag_extra).uniform(0.02, 1.0, (M, H_g)).astype(np.float32)


def quantise_levels(s: np.ndarray, instr_mask: np.ndarray, cu_seqlens: np.ndarray,
                    levels: int) -> np.ndarray:
    """Snap each sequence's document scores onto ``levels`` equally spaced fp32 values.

    Used only to build tie-heavy selection inputs: per sequence, over its document
    rows, lo = min, hi = max, s_q = lo + rint((s - lo) / (hi - lo) * (levels-1)) * step.
    """
    out = np.array(s, dtype=np.float32, copy=True)
    for b in range(len(cu_seqlens) - 1):
        a, e = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        doc = np.nonzero(instr_mask[a:e] == 0)[0] + a
        if doc.size == 0:
            continue
        lo, hi = np.float32(out[doc].min()), np.float32(out[doc].max())
        if hi == lo:
            continue
        step = np.float32((hi - lo) / np.float32(levels - 1))
        q = np.rint((out[doc] - lo) / (hi - lo) * np.float32(levels - 1)).astype(np.float32)
        out[doc] = (lo + q * step).astype(np.float32)
    return out


def make_scores(wl: Workload, tag_extra: int = 0) -> np.ndarray:
    """A synthetic fp32 gate-score buffer (the pre-sigmoid logits) for selection tests.

    Heavy-tailed: N(0, 1) with ``heavy_frac`` (default 2%) of entries scaled by 4;
    quantised to ``score_levels`` levels when the workload asks for ties.
    """
    T = wl.T_total
    s = _rng(wl.seed, _TAG_S, tag_extra).standard_normal(T, dtype=np.float32)
    frac = wl.heavy_frac if wl.heavy_frac > 0 else 0.02
    n_heavy = int(round(frac * T))
    if n_heavy:
        rows = _rng(wl.seed, _TAG_HEAVY, 1000 + tag_extra).choice(T, size=n_heavy, replace=False)
        s[rows] *= np.float32(4.0)
    if wl.score_levels:
        s = quantise_levels(s, make_instr_mask(wl), cu_seqlens_of(wl.seq_lens), wl.score_levels)
    return s


def make_tau_beta(wl: Workload):
    """Per-head temperature tau_h and bias gain beta_h (fp32 [H_q])."""
    if wl.fixed_tau_beta is not None:
        v = np.full(wl.H_q, wl.fixed_tau_beta, dtype=np.float32)
        return v.copy(), v.copy()
    tau = _rng(wl.seed, _TAG_TAU).uniform(0.8, 1.2, wl.H_q).astype(np.float32)
    beta = _rng(wl.seed, _TAG_BETA).uniform(0.8, 1.2, wl.H_q).astype(np.float32)
    return tau, beta


def make_attention_inputs(wl: Workload, M_total: int, tag_extra: int = 0) -> dict:
    """Q/K/V for the kept rows (the projections sit outside the path), plus a gate buffer.

    Q ~ N(0,1) [M, H_q, d_h], K, V ~ N(0,1) [M, H_kv, d_h] in bf16; g ~ U(0.02, 1) fp32 [M].
    """
    M = int(M_total)
    q = _rng(wl.seed, _TAG_Q, tag_extra).standard_normal((M, wl.H_q, wl.d_h), dtype=np.float32)
    k = _rng(wl.seed, _TAG_K, tag_extra).standard_normal((M, wl.H_kv, wl.d_h), dtype=np.float32)
    v = _rng(wl.seed, _TAG_V, tag_extra).standard_normal((M, wl.H_kv, wl.d_h), dtype=np.float32)
    g = _rng(wl.seed, _TAG_G, tag_extra).uniform(0.02, 1.0, M).astype(np.float32)
    tau, beta = make_tau_beta(wl)
    return {"Q": f32_to_bf16_bits(q), "K": f32_to_bf16_bits(k), "V": f32_to_bf16_bits(v),
            "g": g, "tau": tau, "beta": beta}

