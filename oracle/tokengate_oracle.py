"""CPU oracle for the TokenGate gated-prefill path.

TEST INFRASTRUCTURE ONLY. This module is the plain, slow, obviously correct
definition that the CUDA path is checked against. Only the test suite, the
package's smoke check and the benchmark's CPU-baseline leg may import it; the
product path never calls it and shares no code with it.

Arithmetic is numpy float64 throughout. Inputs arrive as float arrays holding
the exact bf16 (or fp32) values the GPU reads; nothing here rounds to bf16.

Sources (the pages this follows, cited by page and equation):
  * "TokenGate: Learnable Token Pruning for Fast, Memory-Efficient LLM Prefill",
    paper deep dive (agientry.com), section 2 Eq. (2); section 3.1 Eqs. (3)-(4);
    section 3.2 Eqs. (5)-(8); section 3.4 "How the released code implements the
    paper" (the prune path: score, clamp the budget, select, keep indices, slice
    the hidden states, gather the original position ids).
  * "TokenGate" paper page (thelatestinai.com), Figure 1 (b)-(c): the gate keeps
    K tokens and forwards the kept hidden states with their importance scores;
    token-gated attention multiplies each attention weight by its key's gate
    value.

Readings where the pages leave a step open (each is listed in the design notes):
  * the score MLP is d -> d_g -> 1 with SiLU, and the gate value is
    g = sigmoid(s); instruction tokens get g = 1 (zero log-bias);
  * top-K ranks the fp32 pre-sigmoid score s, ties go to the lower index, -0.0
    ranks as +0.0 and NaN ranks below every number;
  * attention logit = tau_h * q.k / sqrt(d_h) + beta_h * ln g_j, with
    beta_h * ln g_j := 0 when beta_h == 0 (g^0 = 1); a query whose every key
    has zero weight outputs zeros;
  * GQA: query head h reads kv head floor(h / (H_q / H_kv));
  * RoPE (applied to Q/K at the gathered original positions) is the
    rotate-half form with inv_freq_i = theta^(-2i/d_h).

Parity status of each function: every function here is pinned by tests that do
not re-derive it from its own formula (library routines, closed forms, brute
force, invariants). None is "parity unpinned".

Readings for the exact gate form (normalize_scores, gated_attention_eq8): eps of
the RMS normalisation is a parameter (default 1e-6; the pages give none); m_i is
the number of retained keys query i sees (its index in the kept sequence + 1) and
p_i the number of positions it originally saw (its original position + 1).

Readings for per-head gate scores (the per-head bias and "uniform head aggregation for
selection" of the deep dive's section 3.4): the score MLP's second layer has H_g rows, one
score per gate head; selection ranks the row mean over heads, in fp32 as stored; query head h
reads gate head floor(h / (H_q / H_g)), with H_g dividing H_q. In the exact form each head's
scores are RMS-normalised on their own and selection ranks the mean of the normalised scores.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np


# ---------------------------------------------------------------------------
# Gate score: Eq. (3) of the deep dive, MLP part; gate value of Eq. (5) read as
# a sigmoid (see module docstring).
# ---------------------------------------------------------------------------

def rms_norm(a: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """LN_2 of Eq. (1) in the RMSNorm form of the Qwen3 family: a / sqrt(mean(a^2) + eps) * w."""
    a = np.asarray(a, dtype=np.float64)
    rms = np.sqrt(np.mean(a * a, axis=-1, keepdims=True) + eps)
    return a / rms * np.asarray(weight, dtype=np.float64)


def gate_score(h: np.ndarray, W1: np.ndarray, w2: np.ndarray, instr_mask: np.ndarray,
               b1: Optional[np.ndarray] = None, b2: float = 0.0,
               ln_weight: Optional[np.ndarray] = None, ln_eps: float = 1e-6):
    """Score every row: u = W1 h (+ b1), a = SiLU(u), s = w2 . a (+ b2), g = sigmoid(s).

    h [T, d], W1 [d_g, d], w2 [d_g], instr_mask [T] (1 = non-prunable).
    Returns (s [T], g [T]) in float64; g = 1 on non-prunable rows.
    Deep dive section 3.1, Eq. (3): b~_j = MLP(a~_j); the tokens in the
    non-prunable set carry no bias (read here as g_j = 1). With ln_weight given,
    h is the post-attention residual a^L and the MLP reads LN_2(a^L) (Eq. (1)).

    Per-head scores (deep dive section 3.4: a per-head bias): w2 [H_g, d_g] and b2 a
    scalar or [H_g] give one score per gate head, s and g [T, H_g].
    """
    if ln_weight is not None:
        h = rms_norm(h, ln_weight, ln_eps)
    h = np.asarray(h, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    u = h @ W1.T                                   # [T, d_g]
    if b1 is not None:
        u = u + np.asarray(b1, dtype=np.float64)[None, :]
    with np.errstate(over="ignore"):
        a = u / (1.0 + np.exp(-u))                 # SiLU(u) = u * sigmoid(u)
    if w2.ndim == 1:
        s = a @ w2 + float(b2)                     # [T]
    else:
        s = a @ w2.T + np.asarray(b2, dtype=np.float64)   # [T, H_g]
    with np.errstate(over="ignore"):
        g = 1.0 / (1.0 + np.exp(-s))
    keep = np.asarray(instr_mask) != 0
    g = np.where(keep if g.ndim == 1 else keep[:, None], 1.0, g)
    return s, g


def aggregate_heads(s: np.ndarray) -> np.ndarray:
    """Uniform head aggregation for selection (deep dive section 3.4): the mean of a row's
    per-head scores, s [T, H_g] -> [T]; a single-head score [T] is returned as it is."""
    s = np.asarray(s, dtype=np.float64)
    return s if s.ndim == 1 else s.mean(axis=1)


def gate_column(h: int, H_q: int, H_g: int) -> int:
    """The gate head that query head h reads: consecutive groups of H_q / H_g query heads
    share one gate head (H_g = 1: every head reads the same gate)."""
    return h // (H_q // H_g)


def _head_gate(g: Optional[np.ndarray], h: int, H_q: int, a: int, e: int) -> Optional[np.ndarray]:
    """Rows a..e-1 of the gate (or score bias) that query head h reads; None stays None."""
    if g is None:
        return None
    g = np.asarray(g)
    return g[a:e] if g.ndim == 1 else g[a:e, gate_column(h, H_q, g.shape[1])]


# ---------------------------------------------------------------------------
# Selection: Eq. (4), S = topK_{j in P}(b_j) U N, with the budget clamped to |P|
# and kept indices in original order (deep dive section 3.4).
# ---------------------------------------------------------------------------

def _rank_key(x: float):
    """Sort key for 'larger score first': NaN last, -0.0 equal to +0.0."""
    if math.isnan(x):
        return (1, 0.0)
    return (0, -(x + 0.0))


def topk_select(s: np.ndarray, instr_mask: np.ndarray, cu_seqlens: Sequence[int], K: int):
    """Keep set per sequence: the K_b = min(K, |P_b|) highest-scoring document rows plus
    every non-prunable row, listed in ascending row order.

    s [T] fp32 scores (compared exactly as stored), instr_mask [T], cu_seqlens [B+1].
    Returns (kept_idx int32 [M_total] of global rows, cu_kept int32 [B+1]).
    """
    if K < 0:
        raise ValueError("K must be >= 0")
    s = np.asarray(s, dtype=np.float32)
    B = len(cu_seqlens) - 1
    kept_all = []
    cu_kept = [0]
    for b in range(B):
        start, end = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        prunable = [j for j in range(start, end) if instr_mask[j] == 0]
        keep_always = [j for j in range(start, end) if instr_mask[j] != 0]
        K_b = min(K, len(prunable))
        ranked = sorted(prunable, key=lambda j: (_rank_key(float(s[j])), j))
        selected = ranked[:K_b]
        keep = sorted(selected + keep_always)
        kept_all.extend(keep)
        cu_kept.append(cu_kept[-1] + len(keep))
    return np.asarray(kept_all, dtype=np.int32), np.asarray(cu_kept, dtype=np.int32)


# ---------------------------------------------------------------------------
# Gather: deep dive section 3.4, hidden_states[:, keep] and position_ids[:, keep]
# (original ids), plus the kept gate values (Figure 1 (b)).
# ---------------------------------------------------------------------------

def gather_kept(h: np.ndarray, pos: Optional[np.ndarray], g: np.ndarray, kept_idx: np.ndarray,
                cu_seqlens: Sequence[int]):
    """Rows of h, pos and g at kept_idx. pos None means pos = row - start of its sequence."""
    kept_idx = np.asarray(kept_idx, dtype=np.int64)
    h_k = np.asarray(h)[kept_idx]
    if pos is None:
        seq_of = np.searchsorted(np.asarray(cu_seqlens), kept_idx, side="right") - 1
        p_k = (kept_idx - np.asarray(cu_seqlens, dtype=np.int64)[seq_of]).astype(np.int32)
    else:
        p_k = np.asarray(pos)[kept_idx]
    g_k = np.asarray(g)[kept_idx]
    return h_k, p_k, g_k


# ---------------------------------------------------------------------------
# Token-gated attention: Eq. (5) as the log-space bias form of Eq. (8) with a
# per-head temperature tau_h and gain beta_h (see module docstring).
# ---------------------------------------------------------------------------

def _log_bias(g: Optional[np.ndarray], beta: float, n: int) -> np.ndarray:
    if g is None or beta == 0.0:
        return np.zeros(n, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return beta * np.log(np.asarray(g, dtype=np.float64))


def gated_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, g: Optional[np.ndarray],
                    cu_kept: Sequence[int], tau: Sequence[float], beta: Sequence[float],
                    rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """o_i = sum_{j<=i, same sequence} softmax_j(tau_h q_i.k_j / sqrt(d_h) + beta_h ln g_j) v_j.

    Q [M, H_q, d_h], K/V [M, H_kv, d_h], g [M] or [M, H_g] (per-head gates, query head h
    reads column gate_column(h)) or None (no bias), cu_kept [B+1], tau/beta [H_q]. ``rows`` restricts the output to those global query rows
    (each row is an independent softmax); the result is [len(rows), H_q, d_h]
    (or [M, H_q, d_h] when rows is None). Two passes per row: max, then the
    normalised sum.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    M, H_q, d_h = Q.shape
    H_kv = K.shape[1]
    group = H_q // H_kv
    cu = np.asarray(cu_kept, dtype=np.int64)
    if rows is None:
        rows = np.arange(M)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), H_q, d_h), dtype=np.float64)
    seq_of = np.searchsorted(cu, rows, side="right") - 1
    inv_sqrt = 1.0 / math.sqrt(d_h)
    for h in range(H_q):
        kv = h // group
        for b in np.unique(seq_of):
            start = int(cu[b])
            sel = np.nonzero(seq_of == b)[0]
            r = rows[sel]
            end = int(r.max()) + 1
            keys = K[start:end, kv, :]
            vals = V[start:end, kv, :]
            bias = _log_bias(_head_gate(g, h, H_q, start, end), float(beta[h]), end - start)
            z = (Q[r, h, :] @ keys.T) * inv_sqrt              # [rows, keys]
            logits = float(tau[h]) * z + bias[None, :]
            causal = (np.arange(start, end)[None, :] <= r[:, None])
            logits = np.where(causal, logits, -np.inf)
            m = logits.max(axis=1, keepdims=True)
            m_safe = np.where(np.isfinite(m), m, 0.0)
            p = np.exp(logits - m_safe)                      # exp(-inf) = 0 outside the mask
            l = p.sum(axis=1, keepdims=True)
            o = (p @ vals) / np.where(l > 0, l, 1.0)
            out[sel, h, :] = np.where(l > 0, o, 0.0)
    return out


def gated_attention_weights_eq5(Q: np.ndarray, K: np.ndarray, g: Optional[np.ndarray],
                                tau: float, beta: float, i: int, h: int = 0,
                                kv: int = 0) -> np.ndarray:
    """Eq. (5) product form for one query row of a single sequence:
    alpha_ij = exp(tau z_ij) g_j^beta / sum_{j'<=i} exp(tau z_ij') g_j'^beta.

    A self-check of the log-bias form used by ``gated_attention``: ln of the
    product form is the logit plus beta ln g, so the two must agree.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    d_h = Q.shape[-1]
    z = (K[: i + 1, kv, :] @ Q[i, h, :]) / math.sqrt(d_h)
    w = np.exp(tau * z)
    if g is not None and beta != 0.0:
        w = w * np.power(np.asarray(g[: i + 1], dtype=np.float64), beta)
    total = w.sum()
    return w / total if total > 0 else np.zeros_like(w)


# ---------------------------------------------------------------------------
# The paper's exact gate form (deep dive section 3.1 Eq. (3); section 3.2 Eqs. (6)-(8)):
# sequence-RMS-normalised scores, a per-head softplus gain on the score bias and a per-query
# temperature from the pruning ratio.
# ---------------------------------------------------------------------------

def normalize_scores(s: np.ndarray, instr_mask: np.ndarray, cu_seqlens: Sequence[int],
                     eps: float = 1e-6) -> np.ndarray:
    """Eq. (3): b_j = b~_j / sqrt(mean over the sequence's prunable rows of b~^2 + eps), and
    b_j = 0 on the non-prunable rows. A sequence with no prunable row has b = 0 throughout.
    Per-head scores s [T, H_g] are normalised column by column."""
    s = np.asarray(s, dtype=np.float64)
    if s.ndim == 2:  # per-head scores: each head is normalised over the sequence on its own
        return np.stack([normalize_scores(s[:, c], instr_mask, cu_seqlens, eps) for c in range(s.shape[1])],
                        axis=1)
    b = np.zeros_like(s)
    for i in range(len(cu_seqlens) - 1):
        a, e = int(cu_seqlens[i]), int(cu_seqlens[i + 1])
        doc = [j for j in range(a, e) if instr_mask[j] == 0]
        if not doc:
            continue
        ms = sum(s[j] * s[j] for j in doc) / len(doc)
        for j in doc:
            b[j] = s[j] / math.sqrt(ms + eps)
    return b


def query_temperature(temp: float, m: int, p: int) -> float:
    """Eq. (7): tau_i = softplus(sigma) * log m_i / log max(2, p_i), with softplus(sigma)
    passed in as `temp`; m_i = retained keys query i sees, p_i = positions it originally saw."""
    return float(temp) * math.log(m) / math.log(max(2, p))


def gated_attention_eq8(Q: np.ndarray, K: np.ndarray, V: np.ndarray, b: Optional[np.ndarray],
                        pos: np.ndarray, cu_kept: Sequence[int], gain: Sequence[float],
                        temp: Sequence[float], rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Eq. (8): o_i = sum_{j<=i} softmax_j[tau_i (q_i.k_j / sqrt(d_h) + gain_h b_j)] v_j.

    gain_h = softplus(gamma_h) (>= 0), tau_i from Eq. (7) with temp_h = softplus(sigma_h).
    Query i of a sequence starting at kept row `start` sees m_i = i - start + 1 retained keys
    and originally saw p_i = pos_i + 1 positions (pos holds the original position ids).
    b None means no score bias; b [M, H_g] holds per-head biases (query head h reads column
    gate_column(h)). Layouts and `rows` as in gated_attention; two passes per row.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    M, H_q, d_h = Q.shape
    group = H_q // K.shape[1]
    cu = np.asarray(cu_kept, dtype=np.int64)
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), H_q, d_h), dtype=np.float64)
    bias = np.zeros(M) if b is None else np.asarray(b, dtype=np.float64)
    if bias.ndim == 1:
        bias = bias[:, None]
    for n, i in enumerate(rows):
        seq = int(np.searchsorted(cu, i, side="right") - 1)
        start = int(cu[seq])
        keys = np.arange(start, i + 1)
        for h in range(H_q):
            kv = h // group
            tau = query_temperature(temp[h], i - start + 1, int(pos[i]) + 1)
            z = (K[keys, kv, :] @ Q[i, h, :]) / math.sqrt(d_h)
            logits = tau * (z + float(gain[h]) * bias[keys, gate_column(h, H_q, bias.shape[1])])
            w = np.exp(logits - logits.max())
            out[n, h, :] = (w / w.sum()) @ V[keys, kv, :]
    return out


# ---------------------------------------------------------------------------
# RoPE at the gathered original positions (deep dive section 3.4 keeps the
# original position ids; the rotary form is the rotate-half convention).
# ---------------------------------------------------------------------------

def apply_rope(X: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate each head vector of X [M, H, d_h] by its row's position pos [M].

    Pairs (x_i, x_{i + d_h/2}) rotate by angle pos * theta^(-2i/d_h).
    """
    X = np.asarray(X, dtype=np.float64)
    M, H, d_h = X.shape
    half = d_h // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d_h)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]   # [M, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1 = X[..., :half]
    x2 = X[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---------------------------------------------------------------------------
# The whole prune path (deep dive section 3.4): score -> select -> gather.
# ---------------------------------------------------------------------------

def gate_prune_layer(h, pos, W1, w2, instr_mask, cu_seqlens, K, b1=None, b2=0.0):
    """Score, select on the (head-aggregated) score, gather (deep dive section 3.4)."""
    s, g = gate_score(h, W1, w2, instr_mask, b1, b2)
    kept_idx, cu_kept = topk_select(aggregate_heads(s).astype(np.float32), instr_mask, cu_seqlens, K)
    h_k, p_k, g_k = gather_kept(h, pos, g, kept_idx, cu_seqlens)
    return {"s": s, "g": g, "kept_idx": kept_idx, "cu_kept": cu_kept,
            "h_kept": h_k, "pos_kept": p_k, "g_kept": g_k}


def two_budget_prune_layer(h, pos, W1, w2, instr_mask, cu_seqlens, K_prune, b1=None, b2=0.0):
    """The packed two-budget forward (deep dive section 3.3, Eq. (9)): K_full = |P| keeps every
    row, K_prune keeps the pruned set; both lists over the same scores (phase 1 evaluated
    once), packed as 2B sequences: the B full ones first, then the B pruned ones."""
    full = gate_prune_layer(h, pos, W1, w2, instr_mask, cu_seqlens, len(instr_mask), b1, b2)
    prune = gate_prune_layer(h, pos, W1, w2, instr_mask, cu_seqlens, K_prune, b1, b2)
    T = len(instr_mask)
    cu = np.concatenate([full["cu_kept"], T + prune["cu_kept"][1:]]).astype(np.int32)
    cat = lambda k: np.concatenate([full[k], prune[k]])
    return {"s": full["s"], "g": full["g"], "kept_idx": cat("kept_idx"), "cu_packed": cu,
            "h_kept": cat("h_kept"), "pos_kept": cat("pos_kept"), "g_kept": cat("g_kept")}


# ---------------------------------------------------------------------------
# Backward of token-gated attention (deep dive section 3.2: the gate score reaches the loss
# only through the attention bias; section 3.1: no gradient crosses the top-K choice itself).
# ---------------------------------------------------------------------------

def gated_attention_bwd(Q, K, V, g, dO, cu_kept, tau, beta):
    """Gradients of L = sum(dO * o) for o = gated_attention(Q, K, V, g, cu_kept, tau, beta).

    With x_ij = tau_h q_i.k_j / sqrt(d_h) + beta_h ln g_j over j <= i in the sequence,
    P = softmax_j(x), o_i = sum_j P_ij v_j:
      dV_j += P_ij dO_i;  dP_ij = dO_i.v_j;  D_i = dO_i.o_i;  dX_ij = P_ij (dP_ij - D_i);
      dQ_i = tau_h / sqrt(d_h) sum_j dX_ij k_j;  dK_j += tau_h / sqrt(d_h) dX_ij q_i;
      dbias[j, h] = sum_i dX_ij  (the gradient w.r.t. the head-h bias beta_h ln g_j).
    Query heads of a GQA group add into their kv head's dK, dV. Returns float64
    (dQ [M,H_q,d], dK [M,H_kv,d], dV [M,H_kv,d], dbias [M,H_q]).
    """
    Q, K, V, dO = (np.asarray(a, dtype=np.float64) for a in (Q, K, V, dO))
    M, H_q, d_h = Q.shape
    H_kv = K.shape[1]
    group = H_q // H_kv
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    dbias = np.zeros((M, H_q))
    cu = np.asarray(cu_kept, dtype=np.int64)
    c = 1.0 / math.sqrt(d_h)
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        n = e - a
        if n == 0:
            continue
        causal = np.tril(np.ones((n, n), dtype=bool))
        for h in range(H_q):
            kv = h // group
            q, k, v, do = Q[a:e, h], K[a:e, kv], V[a:e, kv], dO[a:e, h]
            bias = _log_bias(_head_gate(g, h, H_q, a, e), float(beta[h]), n)
            x = np.where(causal, float(tau[h]) * c * (q @ k.T) + bias[None, :], -np.inf)
            mx = x.max(axis=1, keepdims=True)
            mx = np.where(np.isfinite(mx), mx, 0.0)
            p = np.exp(x - mx)
            l = p.sum(axis=1, keepdims=True)
            P = np.where(l > 0, p / np.where(l > 0, l, 1.0), 0.0)
            o = P @ v
            dP = do @ v.T
            D = np.sum(do * o, axis=1, keepdims=True)
            dX = P * (dP - D)
            dV[a:e, kv] += P.T @ do
            dQ[a:e, h] = float(tau[h]) * c * (dX @ k)
            dK[a:e, kv] += float(tau[h]) * c * (dX.T @ q)
            dbias[a:e, h] = dX.sum(axis=0)
    return dQ, dK, dV, dbias


def gated_attention_lse(Q, K, g, cu_kept, tau, beta):
    """ln sum_{j <= i} exp(x_ij) for every kept row i and query head h ([M, H_q]; -inf when
    every key has zero weight), the normaliser the backward rebuilds P with."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    M, H_q, d_h = Q.shape
    group = H_q // K.shape[1]
    cu = np.asarray(cu_kept, dtype=np.int64)
    out = np.full((M, H_q), -np.inf)
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        n = e - a
        if n == 0:
            continue
        causal = np.tril(np.ones((n, n), dtype=bool))
        for h in range(H_q):
            bias = _log_bias(_head_gate(g, h, H_q, a, e), float(beta[h]), n)
            x = np.where(causal, float(tau[h]) / math.sqrt(d_h) * (Q[a:e, h] @ K[a:e, h // group].T) + bias[None, :],
                         -np.inf)
            mx = x.max(axis=1)
            fin = np.isfinite(mx)
            out[a:e, h][fin] = mx[fin] + np.log(np.exp(x[fin] - mx[fin, None]).sum(axis=1))
    return out


def gate_score_grad(dbias, beta, g_kept, kept_idx, T):
    """dL/ds for every input row: the kept row j carries dL/d(ln g_j) = sum_h beta_h dbias[j, h]
    and d ln g / ds = 1 - g for g = sigmoid(s); non-prunable rows have the constant g = 1 and
    rows that were not kept get no gradient (the top-K choice itself has none).
    Per-head gates g_kept [M, H_g]: gate head c collects the query heads that read it,
    ds[:, c] = (1 - g[:, c]) sum_{h : gate_column(h) = c} beta_h dbias[:, h]; ds is [T, H_g]."""
    dbias = np.asarray(dbias, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    g_kept = np.asarray(g_kept, dtype=np.float64)
    kept_idx = np.asarray(kept_idx, dtype=np.int64)
    if g_kept.ndim == 1:
        ds = np.zeros(T)
        ds[kept_idx] = (dbias @ beta) * (1.0 - g_kept)
        return ds
    H_q, H_g = dbias.shape[1], g_kept.shape[1]
    ds = np.zeros((T, H_g))
    for c in range(H_g):
        heads = [h for h in range(H_q) if gate_column(h, H_q, H_g) == c]
        ds[kept_idx, c] = (dbias[:, heads] @ beta[heads]) * (1.0 - g_kept[:, c])
    return ds
