"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties an oracle function to a library routine (torch CPU fp64), a
closed form worked by hand (tests/golden/), a brute-force count, or an
invariant the TokenGate pages fix. The planted-mistake tests at the end show
that a dropped term, a flipped sign or a wrong head index fails a pin.
"""
import inspect
import json
import math
import os
import textwrap

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import tokengate_oracle as O
from learned_token_pruning_07_b300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.cpu


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Gate score (Eq. 3 MLP, sigmoid gate)
# ---------------------------------------------------------------------------

def test_gate_score_closed_form():
    fx = _golden("gate_score_closed_form.json")
    s, g = O.gate_score(np.array(fx["h"]), np.array(fx["W1"]), np.array(fx["w2"]),
                        np.array(fx["instr_mask"]))
    np.testing.assert_allclose(s, fx["s"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(g, fx["g"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("name,with_bias", [("tiny", False), ("tiny", True), ("qwen3_1p7b_8k", True)])
def test_gate_score_matches_torch_mlp(name, with_bias):
    wl = I.WORKLOADS[name]
    gi = I.make_gate_inputs(wl)
    h = I.bf16_bits_to_f64(gi["h"])
    W1 = I.bf16_bits_to_f64(gi["W1"])
    w2 = I.bf16_bits_to_f64(gi["w2"])
    rng = np.random.default_rng(5)
    b1 = rng.standard_normal(wl.d_g) if with_bias else None
    b2 = 0.3 if with_bias else 0.0
    s, g = O.gate_score(h, W1, w2, gi["instr_mask"], b1, b2)
    th = torch.from_numpy(h)
    lin1 = F.linear(th, torch.from_numpy(W1), None if b1 is None else torch.from_numpy(b1))
    ref_s = F.linear(F.silu(lin1), torch.from_numpy(w2)[None, :]).squeeze(1) + b2
    ref_g = torch.sigmoid(ref_s)
    ref_g[torch.from_numpy(gi["instr_mask"].astype(bool))] = 1.0
    np.testing.assert_allclose(s, ref_s.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g, ref_g.numpy(), rtol=1e-12, atol=1e-12)


def test_gate_score_with_rmsnorm_matches_torch():
    # LN_2 (Eq. (1)) as RMSNorm, then the score MLP: torch CPU fp64 F.rms_norm + F.linear / F.silu
    wl = I.WORKLOADS["tiny"]
    gi = I.make_gate_inputs(wl)
    h = I.bf16_bits_to_f64(gi["h"]) * 3.0 + 0.5
    W1, w2 = I.bf16_bits_to_f64(gi["W1"]), I.bf16_bits_to_f64(gi["w2"])
    ln_w = np.random.default_rng(9).uniform(0.5, 1.5, wl.d)
    s, g = O.gate_score(h, W1, w2, gi["instr_mask"], ln_weight=ln_w, ln_eps=1e-6)
    x = F.rms_norm(torch.from_numpy(h), (wl.d,), torch.from_numpy(ln_w), 1e-6)
    ref_s = F.linear(F.silu(F.linear(x, torch.from_numpy(W1))), torch.from_numpy(w2)[None, :]).squeeze(1)
    np.testing.assert_allclose(s, ref_s.numpy(), rtol=1e-12, atol=1e-12)
    # a row scaled by any c > 0 normalises to the same vector, so its score does not change
    s2, _ = O.gate_score(h * 7.0, W1, w2, gi["instr_mask"], ln_weight=ln_w, ln_eps=0.0)
    s3, _ = O.gate_score(h, W1, w2, gi["instr_mask"], ln_weight=ln_w, ln_eps=0.0)
    np.testing.assert_allclose(s2, s3, rtol=1e-12, atol=1e-12)


def test_gate_score_zero_initialised_mlp():
    # The score MLP starts at zero (deep dive section 3.1): every document token scores 0,
    # so g = sigmoid(0) = 1/2; instruction tokens carry g = 1.
    wl = I.WORKLOADS["tiny"]
    gi = I.make_gate_inputs(wl)
    h = I.bf16_bits_to_f64(gi["h"])
    s, g = O.gate_score(h, np.zeros((wl.d_g, wl.d)), I.bf16_bits_to_f64(gi["w2"]), gi["instr_mask"])
    assert np.all(s == 0.0)
    assert np.all(g[gi["instr_mask"] == 0] == 0.5)
    assert np.all(g[gi["instr_mask"] == 1] == 1.0)


# ---------------------------------------------------------------------------
# Selection (Eq. 4, clamped budget, original order)
# ---------------------------------------------------------------------------

def _better(a, b):
    """a ranks above b (larger first, NaN below everything, -0 == +0)."""
    if math.isnan(a):
        return False
    if math.isnan(b):
        return True
    return a > b


def _brute_force_keep(s, mask, cu, K):
    """Pairwise counting: doc row j is selected iff fewer than K_b doc rows beat it."""
    keep = []
    cu_out = [0]
    for b in range(len(cu) - 1):
        rows = list(range(cu[b], cu[b + 1]))
        doc = [j for j in rows if mask[j] == 0]
        K_b = min(K, len(doc))
        for j in rows:
            if mask[j]:
                keep.append(j)
                continue
            beaten_by = 0
            for jj in doc:
                sj, sjj = float(s[j]), float(s[jj])
                tie = (sj == sjj) or (math.isnan(sj) and math.isnan(sjj))
                if _better(sjj, sj) or (tie and jj < j):
                    beaten_by += 1
            if beaten_by < K_b:
                keep.append(j)
        cu_out.append(len(keep))
    return np.array(keep, dtype=np.int32), np.array(cu_out, dtype=np.int32)


def test_select_worked_example():
    fx = _golden("select_worked_example.json")
    for k, want in fx["expected"].items():
        kept, cu = O.topk_select(np.array(fx["s"], np.float32), np.array(fx["instr_mask"]),
                                 fx["cu_seqlens"], int(k))
        assert kept.tolist() == want
        assert cu.tolist() == [0, len(want)]


def _tiny_select_cases():
    rng = np.random.default_rng(17)
    cases = []
    # ties galore: small integer scores
    for where in ("last", "first", "scattered"):
        wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(23, 0, 9, 31), instr_lens=(5, 3, 0, 7),
                            instr_where=where)
        mask = I.make_instr_mask(wl)
        s = rng.integers(-3, 4, size=wl.T_total).astype(np.float32)
        cases.append((s, mask, I.cu_seqlens_of(wl.seq_lens)))
    # signed zeros, infinities and NaN
    s = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1.0, -0.0, np.nan, 0.0, -1.0], np.float32)
    cases.append((s, np.zeros(10, np.uint8), np.array([0, 10], np.int32)))
    # continuous scores
    s = rng.standard_normal(40).astype(np.float32)
    mask = (rng.random(40) < 0.2).astype(np.uint8)
    cases.append((s, mask, np.array([0, 13, 40], np.int32)))
    return cases


@pytest.mark.parametrize("case", range(5))
def test_select_matches_brute_force_for_every_budget(case):
    s, mask, cu = _tiny_select_cases()[case]
    max_doc = max(int(np.sum(mask[cu[b]:cu[b + 1]] == 0)) for b in range(len(cu) - 1))
    for K in range(0, max_doc + 2):
        kept, cu_k = O.topk_select(s, mask, cu, K)
        ref, ref_cu = _brute_force_keep(s, mask, cu, K)
        assert kept.tolist() == ref.tolist(), K
        assert cu_k.tolist() == ref_cu.tolist(), K


def test_select_invariants_on_tiny_workload():
    wl = I.WORKLOADS["tiny"]
    s = I.make_scores(wl)
    mask = I.make_instr_mask(wl)
    cu = I.cu_seqlens_of(wl.seq_lens)
    n_doc = int(np.sum(mask == 0))
    for K in (0, 1, 64, n_doc - 1, n_doc, n_doc + 5):
        kept, cu_k = O.topk_select(s, mask, cu, K)
        assert np.all(np.diff(kept) > 0)                             # original order, no repeats
        assert set(np.nonzero(mask)[0]) <= set(kept.tolist())        # N always survives
        assert len(kept) == min(K, n_doc) + int(mask.sum())          # |S| = K_b + |N|
        if K >= n_doc:
            assert kept.tolist() == list(range(wl.T_total))          # full budget keeps all
        sel = [j for j in kept if mask[j] == 0]
        rest = [j for j in range(wl.T_total) if mask[j] == 0 and j not in set(sel)]
        if sel and rest:
            assert s[sel].min() >= s[rest].max()


def test_select_all_equal_scores_keeps_first_k_documents():
    wl = I.with_changes(I.WORKLOADS["tiny"], instr_where="first")
    mask = I.make_instr_mask(wl)
    s = np.full(wl.T_total, 0.25, np.float32)
    kept, _ = O.topk_select(s, mask, I.cu_seqlens_of(wl.seq_lens), 10)
    assert kept.tolist() == list(range(32)) + list(range(32, 42))


def test_select_on_quantised_ragged_scores_matches_brute_force():
    wl = I.with_changes(I.WORKLOADS["ragged_b8"], doc_lens=(60, 41, 75), instr_lens=(7, 3, 12),
                        score_levels=16)
    s = I.make_scores(wl)
    assert len(np.unique(s)) < 0.8 * wl.T_total
    mask = I.make_instr_mask(wl)
    cu = I.cu_seqlens_of(wl.seq_lens)
    for K in (0, 5, 20, 40, 80):
        kept, cu_k = O.topk_select(s, mask, cu, K)
        ref, ref_cu = _brute_force_keep(s, mask, cu, K)
        assert kept.tolist() == ref.tolist()
        assert cu_k.tolist() == ref_cu.tolist()


def test_select_rejects_negative_budget():
    with pytest.raises(ValueError):
        O.topk_select(np.zeros(4, np.float32), np.zeros(4, np.uint8), [0, 4], -1)


# ---------------------------------------------------------------------------
# Gather (original position ids)
# ---------------------------------------------------------------------------

def test_gather_default_positions_are_original_ids():
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(20, 30), instr_lens=(4, 6))
    cu = I.cu_seqlens_of(wl.seq_lens)
    pos = I.make_positions(wl)
    rng = np.random.default_rng(3)
    kept = np.sort(rng.choice(wl.T_total, size=25, replace=False)).astype(np.int32)
    h = rng.standard_normal((wl.T_total, 8))
    g = rng.random(wl.T_total)
    hk, pk, gk = O.gather_kept(h, None, g, kept, cu)
    hk2, pk2, gk2 = O.gather_kept(h, pos, g, kept, cu)
    assert pk.tolist() == pk2.tolist()
    for m, j in enumerate(kept):
        assert np.array_equal(hk[m], h[j]) and gk[m] == g[j]
        assert pk[m] == (j if j < cu[1] else j - cu[1])


def test_gather_full_keep_is_identity():
    h = np.arange(12.0).reshape(6, 2)
    g = np.linspace(0, 1, 6)
    hk, pk, gk = O.gather_kept(h, None, g, np.arange(6), [0, 6])
    assert np.array_equal(hk, h) and np.array_equal(gk, g) and pk.tolist() == list(range(6))


# ---------------------------------------------------------------------------
# Token-gated attention (Eq. 5 / Eq. 8)
# ---------------------------------------------------------------------------

def _sdpa_reference(Q, K, V, g, cu, tau, beta):
    """torch CPU fp64 scaled_dot_product_attention with an additive float mask
    (causal -inf plus beta_h ln g_j), scale tau_h / sqrt(d_h), GQA by repeat_interleave."""
    M, H_q, d_h = Q.shape
    H_kv = K.shape[1]
    out = torch.zeros(M, H_q, d_h, dtype=torch.float64)
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        if e == a:
            continue
        q = torch.from_numpy(Q[a:e]).permute(1, 0, 2)                       # [H_q, n, d]
        k = torch.from_numpy(K[a:e]).permute(1, 0, 2).repeat_interleave(H_q // H_kv, dim=0)
        v = torch.from_numpy(V[a:e]).permute(1, 0, 2).repeat_interleave(H_q // H_kv, dim=0)
        n = e - a
        causal = torch.full((n, n), float("-inf"), dtype=torch.float64).triu(1)
        for h in range(H_q):
            bias = torch.zeros(n, dtype=torch.float64)
            if g is not None and beta[h] != 0:
                bias = float(beta[h]) * torch.log(torch.from_numpy(np.asarray(g[a:e], np.float64)))
            mask = causal + bias[None, :]
            o = F.scaled_dot_product_attention(q[h:h + 1], k[h:h + 1], v[h:h + 1], attn_mask=mask,
                                               scale=float(tau[h]) / math.sqrt(d_h))
            out[a:e, h] = o[0]
    return out.numpy()


def _rand_attn(seed, lens, H_q=4, H_kv=2, d_h=16):
    rng = np.random.default_rng(seed)
    M = sum(lens)
    Q = rng.standard_normal((M, H_q, d_h))
    K = rng.standard_normal((M, H_kv, d_h))
    V = rng.standard_normal((M, H_kv, d_h))
    g = rng.uniform(0.02, 1.0, M)
    tau = rng.uniform(0.5, 1.5, H_q)
    beta = rng.uniform(0.5, 1.5, H_q)
    return Q, K, V, g, I.cu_seqlens_of(lens), tau, beta


@pytest.mark.parametrize("lens", [(17,), (5, 33, 1, 12)])
def test_attention_matches_torch_sdpa_with_bias_mask(lens):
    Q, K, V, g, cu, tau, beta = _rand_attn(11, lens)
    got = O.gated_attention(Q, K, V, g, cu, tau, beta)
    ref = _sdpa_reference(Q, K, V, g, cu, tau, beta)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_attention_beta_zero_is_standard_causal_attention():
    Q, K, V, g, cu, tau, _ = _rand_attn(12, (29,))
    beta = np.zeros_like(tau)
    got = O.gated_attention(Q, K, V, g, cu, tau, beta)
    q = torch.from_numpy(Q).permute(1, 0, 2)
    k = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(2, dim=0)
    v = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(2, dim=0)
    for h in range(Q.shape[1]):
        ref = F.scaled_dot_product_attention(q[h:h + 1], k[h:h + 1], v[h:h + 1], is_causal=True,
                                             scale=float(tau[h]) / math.sqrt(Q.shape[2]))[0]
        np.testing.assert_allclose(got[:, h], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_attention_constant_gate_equals_no_gate():
    Q, K, V, _, cu, tau, beta = _rand_attn(13, (3, 21))
    g_const = np.full(Q.shape[0], 0.37)
    a = O.gated_attention(Q, K, V, g_const, cu, tau, beta)
    b = O.gated_attention(Q, K, V, None, cu, tau, beta)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_attention_eq5_product_form_and_rows_sum_to_one():
    n = 16
    rng = np.random.default_rng(14)
    Q = rng.standard_normal((n, 1, n))
    K = rng.standard_normal((n, 1, n))
    V = np.eye(n)[:, None, :]                      # o_i = the weight vector alpha_i
    g = rng.uniform(0.05, 1.0, n)
    tau, beta = np.array([1.3]), np.array([0.7])
    o = O.gated_attention(Q, K, V, g, [0, n], tau, beta)[:, 0, :]
    for i in range(n):
        w = O.gated_attention_weights_eq5(Q, K, g, 1.3, 0.7, i)
        np.testing.assert_allclose(o[i, :i + 1], w, rtol=1e-12, atol=1e-14)
        assert np.all(o[i, i + 1:] == 0.0)
        assert abs(o[i].sum() - 1.0) < 1e-12


def test_attention_zero_logits_closed_form():
    fx = _golden("attention_zero_logits.json")
    got = O.gated_attention(np.array(fx["Q"]), np.array(fx["K"]), np.array(fx["V"]),
                            np.array(fx["g"]), [0, 3], fx["tau"], fx["beta"])
    np.testing.assert_allclose(got, np.array(fx["O"]), rtol=0, atol=1e-15)


def test_attention_single_token_returns_its_value():
    Q, K, V, g, _, tau, beta = _rand_attn(15, (1,))
    got = O.gated_attention(Q, K, V, g, [0, 1], tau, beta)
    np.testing.assert_allclose(got[0], np.repeat(V[0], 2, axis=0), rtol=0, atol=0)


def test_attention_tiny_gate_removes_key():
    Q, K, V, g, cu, tau, _ = _rand_attn(16, (12,))
    beta = np.ones_like(tau)
    g = g.copy()
    g[4] = 1e-300
    got = O.gated_attention(Q, K, V, g, cu, tau, beta)
    keep = [j for j in range(12) if j != 4]
    sub = O.gated_attention(Q[keep], K[keep], V[keep], g[keep], [0, 11], tau, beta)
    np.testing.assert_allclose(got[keep], sub, rtol=1e-9, atol=1e-12)


def test_attention_all_zero_gates_give_zero_rows():
    Q, K, V, _, cu, tau, beta = _rand_attn(17, (6,))
    g = np.zeros(6)
    got = O.gated_attention(Q, K, V, g, cu, tau, beta)
    assert np.all(got == 0.0)


def test_attention_sequences_are_independent_and_rows_subset():
    Q, K, V, g, cu, tau, beta = _rand_attn(18, (9, 14))
    whole = O.gated_attention(Q, K, V, g, cu, tau, beta)
    second = O.gated_attention(Q[9:], K[9:], V[9:], g[9:], [0, 14], tau, beta)
    np.testing.assert_allclose(whole[9:], second, rtol=1e-12, atol=1e-14)
    rows = [0, 8, 9, 22]
    np.testing.assert_allclose(O.gated_attention(Q, K, V, g, cu, tau, beta, rows=rows), whole[rows],
                               rtol=0, atol=0)


# ---------------------------------------------------------------------------
# The paper's exact gate form: Eq. (3) normalisation, Eq. (7) temperature, Eq. (8) attention
# ---------------------------------------------------------------------------

def test_normalize_scores_closed_form():
    fx = _golden("normalized_scores_closed_form.json")
    b = O.normalize_scores(np.array(fx["s"]), np.array(fx["instr_mask"]), fx["cu_seqlens"], eps=0.0)
    np.testing.assert_allclose(b, fx["b"], rtol=0, atol=1e-15)
    for m, p, want in fx["tau_cases"]:
        assert abs(O.query_temperature(fx["temp"], m, p) - want) < 1e-15


def test_normalize_scores_invariants():
    rng = np.random.default_rng(31)
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(40, 0, 25), instr_lens=(6, 3, 0), instr_where="scattered")
    mask = I.make_instr_mask(wl)
    cu = I.cu_seqlens_of(wl.seq_lens)
    s = rng.standard_normal(wl.T_total) * 3.0
    b = O.normalize_scores(s, mask, cu, eps=0.0)
    assert np.all(b[mask == 1] == 0.0)
    assert np.all(b[cu[1]:cu[2]] == 0.0)                      # no prunable rows: nothing to scale
    for i in (0, 2):
        doc = [j for j in range(cu[i], cu[i + 1]) if mask[j] == 0]
        assert abs(np.mean(b[doc] ** 2) - 1.0) < 1e-12          # unit RMS over P
        assert np.array_equal(np.argsort(-s[doc], kind="stable"), np.argsort(-b[doc], kind="stable"))
    np.testing.assert_allclose(O.normalize_scores(7.5 * s, mask, cu, eps=0.0), b, rtol=1e-12)


def _sdpa_eq8_rows(Q, K, V, b, pos, cu, gain, temp):
    """torch CPU fp64 scaled_dot_product_attention, one query row at a time: scale tau_i/sqrt(d_h)
    and additive mask tau_i * gain_h * b_j over the row's visible keys."""
    M, H_q, d_h = Q.shape
    group = H_q // K.shape[1]
    out = torch.zeros(M, H_q, d_h, dtype=torch.float64)
    for i in range(M):
        seq = int(np.searchsorted(cu, i, side="right") - 1)
        a = int(cu[seq])
        m, p = i - a + 1, int(pos[i]) + 1
        for h in range(H_q):
            tau = temp[h] * math.log(m) / math.log(max(2, p))
            q = torch.from_numpy(Q[i:i + 1, h][None])                       # [1, 1, d]
            k = torch.from_numpy(K[a:i + 1, h // group][None])              # [1, m, d]
            v = torch.from_numpy(V[a:i + 1, h // group][None])
            mask = torch.from_numpy(tau * gain[h] * np.asarray(b[a:i + 1], np.float64))[None, None, :]
            o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=tau / math.sqrt(d_h))
            out[i, h] = o[0, 0]
    return out.numpy()


def _eq8_case(seed, lens):
    rng = np.random.default_rng(seed)
    Q, K, V, _, cu, _, _ = _rand_attn(seed, lens)
    M = Q.shape[0]
    b = rng.standard_normal(M)
    pos = np.zeros(M, dtype=np.int64)
    for i in range(len(lens)):                                # strictly increasing original ids with gaps
        a, e = int(cu[i]), int(cu[i + 1])
        pos[a:e] = np.cumsum(rng.integers(1, 6, e - a)) - 1
    gain = rng.uniform(0.2, 1.5, Q.shape[1])
    temp = rng.uniform(0.5, 1.5, Q.shape[1])
    return Q, K, V, b, pos, cu, gain, temp


@pytest.mark.parametrize("lens", [(13,), (4, 1, 17)])
def test_eq8_attention_matches_rowwise_sdpa(lens):
    Q, K, V, b, pos, cu, gain, temp = _eq8_case(41, lens)
    got = O.gated_attention_eq8(Q, K, V, b, pos, cu, gain, temp)
    ref = _sdpa_eq8_rows(Q, K, V, b, pos, cu, gain, temp)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_eq8_without_pruning_reduces_to_the_log_gate_form():
    # m_i = p_i (nothing pruned) and softplus(sigma) = 1 give tau_i = 1 (row 0 sees only itself);
    # gain_h * b_j is then the log-bias beta_h ln g_j with g = exp(b), beta = gain
    Q, K, V, b, _, cu, gain, _ = _eq8_case(42, (11, 5))
    pos = np.concatenate([np.arange(11), np.arange(5)])
    got = O.gated_attention_eq8(Q, K, V, b, pos, cu, gain, np.ones(Q.shape[1]))
    ref = O.gated_attention(Q, K, V, np.exp(b), cu, np.ones(Q.shape[1]), gain)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def _planted_eq8(kind, Q, K, V, b, pos, cu, gain, temp):
    """gated_attention_eq8 with one planted mistake, for the pin below."""
    M, H_q, d_h = Q.shape
    group = H_q // K.shape[1]
    out = np.zeros((M, H_q, d_h))
    for i in range(M):
        a = int(cu[np.searchsorted(cu, i, side="right") - 1])
        keys = np.arange(a, i + 1)
        m, p = i - a + 1, int(pos[i]) + 1
        if kind == "p_without_plus_one":
            p -= 1
        for h in range(H_q):
            tau = temp[h] * math.log(m) / math.log(max(2, p))
            z = (K[keys, h // group] @ Q[i, h]) / math.sqrt(d_h)
            if kind == "tau_on_logit_only":
                logits = tau * z + gain[h] * b[keys]
            else:
                logits = tau * (z + gain[h] * b[keys])
            w = np.exp(logits - logits.max())
            out[i, h] = (w / w.sum()) @ V[keys, h // group]
    return out


@pytest.mark.parametrize("kind", ["tau_on_logit_only", "p_without_plus_one"])
def test_planted_eq8_mistakes_fail_the_rowwise_pin(kind):
    Q, K, V, b, pos, cu, gain, temp = _eq8_case(43, (14,))
    ref = _sdpa_eq8_rows(Q, K, V, b, pos, cu, gain, temp)
    assert np.allclose(_planted_eq8("none", Q, K, V, b, pos, cu, gain, temp), ref, rtol=1e-10, atol=1e-12)
    wrong = _planted_eq8(kind, Q, K, V, b, pos, cu, gain, temp)
    assert not np.allclose(wrong, ref, rtol=1e-6, atol=1e-8)


# ---------------------------------------------------------------------------
# The packed two-budget forward (Eq. (9))
# ---------------------------------------------------------------------------

def test_two_budget_pack_invariants():
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(50, 0, 33), instr_lens=(4, 2, 6), d=64, d_g=32)
    gi = I.make_gate_inputs(wl)
    h = I.bf16_bits_to_f64(gi["h"])
    W1, w2 = I.bf16_bits_to_f64(gi["W1"]), I.bf16_bits_to_f64(gi["w2"])
    T, B = wl.T_total, wl.B
    out = O.two_budget_prune_layer(h, gi["pos"], W1, w2, gi["instr_mask"], gi["cu_seqlens"], 7)
    cu = out["cu_packed"]
    assert out["kept_idx"][:T].tolist() == list(range(T))            # K_full = |P| keeps every row
    assert cu[:B + 1].tolist() == gi["cu_seqlens"].tolist() and cu[B] == T
    for b in range(B):                                               # |S_b| = min(K, |P_b|) + |N_b|
        assert cu[B + b + 1] - cu[B + b] == min(7, wl.doc_lens[b]) + wl.instr_lens[b]
    assert np.array_equal(out["h_kept"], h[out["kept_idx"]])
    # sequences are independent: attention over the packed batch = attention over each half
    at = I.make_attention_inputs(wl, int(cu[-1]))
    Q, K, V = (I.bf16_bits_to_f64(at[k]) for k in ("Q", "K", "V"))
    whole = O.gated_attention(Q, K, V, out["g_kept"], cu, at["tau"], at["beta"])
    M = int(cu[-1])
    second = O.gated_attention(Q[T:], K[T:], V[T:], out["g_kept"][T:], cu[B:] - T, at["tau"], at["beta"])
    np.testing.assert_allclose(whole[T:M], second, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# Backward of token-gated attention
# ---------------------------------------------------------------------------

def _torch_forward(Q, K, V, g, cu, tau, beta):
    """The same forward written with torch CPU fp64 ops (causal softmax with the log-gate bias),
    differentiable in Q, K, V and the per-head bias tensor."""
    M, H_q, d_h = Q.shape
    group = H_q // K.shape[1]
    q, k, v = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (Q, K, V))
    lng = torch.log(torch.tensor(g, dtype=torch.float64))
    bias = (torch.tensor(beta, dtype=torch.float64)[None, :] * lng[:, None]).detach().requires_grad_(True)
    outs = []
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        n = e - a
        mask = torch.full((n, n), float("-inf"), dtype=torch.float64).triu(1)
        heads = []
        for h in range(H_q):
            z = (q[a:e, h] @ k[a:e, h // group].T) * (float(tau[h]) / math.sqrt(d_h))
            w = torch.softmax(z + bias[a:e, h][None, :] + mask, dim=1)
            heads.append(w @ v[a:e, h // group])
        outs.append(torch.stack(heads, dim=1))
    return torch.cat(outs, dim=0), (q, k, v, bias)


def test_attention_bwd_matches_torch_autograd():
    Q, K, V, g, cu, tau, beta = _rand_attn(51, (9, 1, 14))
    dO = np.random.default_rng(52).standard_normal(Q.shape)
    dQ, dK, dV, dbias = O.gated_attention_bwd(Q, K, V, g, dO, cu, tau, beta)
    out, (q, k, v, bias) = _torch_forward(Q, K, V, g, cu, tau, beta)
    np.testing.assert_allclose(out.detach().numpy(), O.gated_attention(Q, K, V, g, cu, tau, beta),
                               rtol=1e-12, atol=1e-12)
    (out * torch.from_numpy(dO)).sum().backward()
    for got, ref in ((dQ, q.grad), (dK, k.grad), (dV, v.grad), (dbias, bias.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_attention_bwd_bias_gradient_by_finite_differences():
    # d/d(ln g_j) of sum(dO * o) = sum_h beta_h dbias[j, h]: central differences on ln g
    Q, K, V, g, cu, tau, beta = _rand_attn(53, (7, 5))
    dO = np.random.default_rng(54).standard_normal(Q.shape)
    _, _, _, dbias = O.gated_attention_bwd(Q, K, V, g, dO, cu, tau, beta)
    loss = lambda gg: float(np.sum(dO * O.gated_attention(Q, K, V, gg, cu, tau, beta)))
    eps = 1e-6
    for j in (0, 3, 6, 7, 11):
        up, dn = g.copy(), g.copy()
        up[j] *= math.exp(eps)
        dn[j] *= math.exp(-eps)
        fd = (loss(up) - loss(dn)) / (2 * eps)
        assert abs(fd - float(dbias[j] @ beta)) < 1e-6 * max(1.0, abs(fd))


def test_attention_lse_matches_torch_logsumexp():
    Q, K, V, g, cu, tau, beta = _rand_attn(57, (6, 11))
    got = O.gated_attention_lse(Q, K, g, cu, tau, beta)
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        for h in range(Q.shape[1]):
            z = torch.from_numpy(Q[a:e, h] @ K[a:e, h // 2].T) * (tau[h] / math.sqrt(Q.shape[2]))
            z = z + beta[h] * torch.log(torch.from_numpy(g[a:e]))[None, :]
            z = z.masked_fill(torch.ones(e - a, e - a, dtype=torch.bool).triu(1), float("-inf"))
            np.testing.assert_allclose(got[a:e, h], torch.logsumexp(z, dim=1).numpy(), rtol=1e-12, atol=1e-12)


def test_gate_score_grad_chain():
    # ds_j = (1 - g_j) * sum_h beta_h dbias[j, h] on kept rows, 0 elsewhere; by finite
    # differences through g = sigmoid(s) on a kept document row
    Q, K, V, _, cu, tau, beta = _rand_attn(55, (10,))
    rng = np.random.default_rng(56)
    s = rng.standard_normal(10)
    g = 1.0 / (1.0 + np.exp(-s))
    dO = rng.standard_normal(Q.shape)
    _, _, _, dbias = O.gated_attention_bwd(Q, K, V, g, dO, cu, tau, beta)
    kept = np.arange(10) * 2                                  # rows of a 20-row input
    ds = O.gate_score_grad(dbias, beta, g, kept, 20)
    assert np.all(ds[1::2] == 0.0)
    loss = lambda ss: float(np.sum(dO * O.gated_attention(Q, K, V, 1.0 / (1.0 + np.exp(-ss)), cu, tau, beta)))
    for j in (2, 5, 9):
        up, dn = s.copy(), s.copy()
        up[j] += 1e-6
        dn[j] -= 1e-6
        assert abs((loss(up) - loss(dn)) / 2e-6 - ds[kept[j]]) < 1e-6


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def test_rope_matches_complex_rotation_and_is_relative():
    rng = np.random.default_rng(19)
    M, H, d_h = 7, 3, 8
    X = rng.standard_normal((M, H, d_h))
    pos = rng.integers(0, 5000, M)
    out = O.apply_rope(X, pos, 1.0e6)
    half = d_h // 2
    z = X[..., :half] + 1j * X[..., half:]
    freq = 1.0e6 ** (-np.arange(half) * 2.0 / d_h)
    zr = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    np.testing.assert_allclose(out, np.concatenate([zr.real, zr.imag], axis=-1), rtol=1e-12, atol=1e-12)
    assert np.allclose(O.apply_rope(X, np.zeros(M, int), 1e6), X)
    np.testing.assert_allclose(np.linalg.norm(out, axis=-1), np.linalg.norm(X, axis=-1), rtol=1e-12)
    q, k = X[:1], X[1:2]
    a = O.apply_rope(q, np.array([40]), 1e4)[0, 0] @ O.apply_rope(k, np.array([25]), 1e4)[0, 0]
    b = O.apply_rope(q, np.array([1040]), 1e4)[0, 0] @ O.apply_rope(k, np.array([1025]), 1e4)[0, 0]
    assert abs(a - b) < 1e-9


# ---------------------------------------------------------------------------
# Planted mistakes: each variant must fail at least one pin above
# ---------------------------------------------------------------------------

def _planted_attention(kind):
    def f(Q, K, V, g, cu_kept, tau, beta, rows=None):
        if kind == "bias_sign":
            return O.gated_attention(Q, K, V, None if g is None else 1.0 / np.asarray(g), cu_kept, tau, beta, rows)
        if kind == "no_tau":
            return O.gated_attention(Q, K, V, g, cu_kept, np.ones_like(tau), beta, rows)
        if kind == "gqa_modulo":
            H_q, H_kv = Q.shape[1], K.shape[1]
            Kp = np.stack([K[:, h % H_kv] for h in range(H_q)], axis=1)
            Vp = np.stack([V[:, h % H_kv] for h in range(H_q)], axis=1)
            return O.gated_attention(Q, Kp, Vp, g, cu_kept, tau, beta, rows)
        raise ValueError(kind)
    return f


@pytest.mark.parametrize("kind", ["bias_sign", "no_tau", "gqa_modulo"])
def test_planted_attention_mistakes_fail_the_sdpa_pin(kind):
    Q, K, V, g, cu, tau, beta = _rand_attn(11, (17,))
    got = _planted_attention(kind)(Q, K, V, g, cu, tau, beta)
    ref = _sdpa_reference(Q, K, V, g, cu, tau, beta)
    assert not np.allclose(got, ref, rtol=1e-6, atol=1e-8)


def test_planted_selection_mistake_fails_brute_force():
    # ties to the higher index instead of the lower one
    s, mask, cu = _tiny_select_cases()[0]
    kept_bad = []
    for b in range(len(cu) - 1):
        rows = range(cu[b], cu[b + 1])
        doc = [j for j in rows if mask[j] == 0]
        ranked = sorted(doc, key=lambda j: (-float(s[j]), -j))[:min(5, len(doc))]
        kept_bad.extend(sorted(ranked + [j for j in rows if mask[j]]))
    ref, _ = _brute_force_keep(s, mask, cu, 5)
    assert kept_bad != ref.tolist()


# ---------------------------------------------------------------------------
# Per-head gate scores and uniform head aggregation (deep dive section 3.4)
# ---------------------------------------------------------------------------

def _heads_case(H_g, seed=61):
    wl = I.WORKLOADS["tiny"]
    gi = I.make_gate_inputs(wl)
    rng = np.random.default_rng(seed)
    h = I.bf16_bits_to_f64(gi["h"])
    W1 = I.bf16_bits_to_f64(gi["W1"])
    W2 = rng.standard_normal((H_g, wl.d_g)) * 0.05
    b1 = rng.standard_normal(wl.d_g) * 0.1
    b2 = rng.standard_normal(H_g) * 0.2
    return wl, gi, h, W1, W2, b1, b2


@pytest.mark.parametrize("H_g", [1, 2, 4])
def test_gate_score_heads_match_torch_mlp(H_g):
    wl, gi, h, W1, W2, b1, b2 = _heads_case(H_g)
    s, g = O.gate_score(h, W1, W2, gi["instr_mask"], b1, b2)
    assert s.shape == (wl.T_total, H_g) and g.shape == (wl.T_total, H_g)
    hid = F.silu(F.linear(torch.from_numpy(h), torch.from_numpy(W1), torch.from_numpy(b1)))
    ref_s = F.linear(hid, torch.from_numpy(W2), torch.from_numpy(b2))
    ref_g = torch.sigmoid(ref_s)
    ref_g[torch.from_numpy(gi["instr_mask"].astype(bool))] = 1.0
    np.testing.assert_allclose(s, ref_s.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g, ref_g.numpy(), rtol=1e-12, atol=1e-12)


def test_uniform_aggregation_is_the_score_of_the_mean_head():
    # the second layer is linear: the mean of H_g head scores is the single-head score of the
    # mean row of W2 (and the mean b2); torch.mean gives the same row means
    wl, gi, h, W1, W2, b1, b2 = _heads_case(4, seed=62)
    s, _ = O.gate_score(h, W1, W2, gi["instr_mask"], b1, b2)
    agg = O.aggregate_heads(s)
    s1, _ = O.gate_score(h, W1, W2.mean(axis=0), gi["instr_mask"], b1, float(b2.mean()))
    np.testing.assert_allclose(agg, s1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(agg, torch.from_numpy(s).mean(dim=1).numpy(), rtol=1e-14, atol=1e-14)
    # one head: aggregation changes nothing
    assert np.array_equal(O.aggregate_heads(s[:, 0]), s[:, 0])


def test_per_head_normalisation_is_columnwise_unit_rms():
    rng = np.random.default_rng(63)
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(30, 22), instr_lens=(4, 0), instr_where="scattered")
    mask = I.make_instr_mask(wl)
    cu = I.cu_seqlens_of(wl.seq_lens)
    s = rng.standard_normal((wl.T_total, 3)) * np.array([0.5, 3.0, 11.0])
    b = O.normalize_scores(s, mask, cu, eps=0.0)
    assert np.all(b[mask == 1] == 0.0)
    for i in range(2):
        doc = [j for j in range(cu[i], cu[i + 1]) if mask[j] == 0]
        np.testing.assert_allclose(np.mean(b[doc] ** 2, axis=0), np.ones(3), rtol=1e-12)
        # a per-head positive scale leaves the order within each head unchanged
        for c in range(3):
            assert np.array_equal(np.argsort(-s[doc, c], kind="stable"), np.argsort(-b[doc, c], kind="stable"))


def _sdpa_reference_heads(Q, K, V, G, cu, tau, beta):
    """torch CPU fp64 SDPA with a per-head additive mask; query head h adds beta_h ln of gate
    column h * H_g // H_q."""
    M, H_q, d_h = Q.shape
    H_kv, H_g = K.shape[1], G.shape[1]
    out = torch.zeros(M, H_q, d_h, dtype=torch.float64)
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        n = e - a
        if n == 0:
            continue
        causal = torch.full((n, n), float("-inf"), dtype=torch.float64).triu(1)
        for h in range(H_q):
            col = h * H_g // H_q
            kv = h * H_kv // H_q
            mask = causal + float(beta[h]) * torch.log(torch.from_numpy(G[a:e, col]))[None, :]
            o = F.scaled_dot_product_attention(torch.from_numpy(Q[a:e, h])[None], torch.from_numpy(K[a:e, kv])[None],
                                               torch.from_numpy(V[a:e, kv])[None], attn_mask=mask,
                                               scale=float(tau[h]) / math.sqrt(d_h))
            out[a:e, h] = o[0]
    return out.numpy()


@pytest.mark.parametrize("H_g", [2, 4])
def test_attention_with_per_head_gates_matches_torch_sdpa(H_g):
    Q, K, V, _, cu, tau, beta = _rand_attn(64, (9, 1, 15))
    G = np.random.default_rng(65).uniform(0.02, 1.0, (Q.shape[0], H_g))
    got = O.gated_attention(Q, K, V, G, cu, tau, beta)
    np.testing.assert_allclose(got, _sdpa_reference_heads(Q, K, V, G, cu, tau, beta), rtol=1e-10, atol=1e-12)
    # one gate column is the shared gate of the single-head form
    np.testing.assert_allclose(O.gated_attention(Q, K, V, G[:, :1], cu, tau, beta),
                               _sdpa_reference(Q, K, V, G[:, 0], cu, tau, beta), rtol=1e-10, atol=1e-12)


def test_planted_gate_column_mistake_fails_the_sdpa_pin(monkeypatch):
    # query heads spread over the gate heads modulo instead of in consecutive groups
    Q, K, V, _, cu, tau, beta = _rand_attn(66, (13,))
    G = np.random.default_rng(67).uniform(0.02, 1.0, (Q.shape[0], 2))
    monkeypatch.setattr(O, "gate_column", lambda h, H_q, H_g: h % H_g)
    got = O.gated_attention(Q, K, V, G, cu, tau, beta)
    assert not np.allclose(got, _sdpa_reference_heads(Q, K, V, G, cu, tau, beta), rtol=1e-6, atol=1e-8)


def test_eq8_attention_with_per_head_bias_matches_rowwise_sdpa():
    Q, K, V, _, pos, cu, gain, temp = _eq8_case(68, (7, 12))
    M, H_q, d_h = Q.shape
    Bh = np.random.default_rng(69).standard_normal((M, 2))
    got = O.gated_attention_eq8(Q, K, V, Bh, pos, cu, gain, temp)
    # each query head is the single-bias form with its own column, which the row-wise torch pin checks
    ref = np.zeros_like(got)
    for h in range(H_q):
        col = h * 2 // H_q
        ref[:, h] = _sdpa_eq8_rows(Q, K, V, Bh[:, col], pos, cu, gain, temp)[:, h]
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def _torch_forward_heads(Q, K, V, G, cu, tau, beta):
    """torch CPU fp64 forward with per-head gates, differentiable in Q, K, V and the bias."""
    M, H_q, d_h = Q.shape
    H_kv, H_g = K.shape[1], G.shape[1]
    q, k, v = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (Q, K, V))
    lng = torch.log(torch.tensor(G, dtype=torch.float64))
    bias = torch.stack([float(beta[h]) * lng[:, h * H_g // H_q] for h in range(H_q)], dim=1)
    bias = bias.detach().requires_grad_(True)
    outs = []
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        n = e - a
        mask = torch.full((n, n), float("-inf"), dtype=torch.float64).triu(1)
        heads = []
        for h in range(H_q):
            kv = h * H_kv // H_q
            z = (q[a:e, h] @ k[a:e, kv].T) * (float(tau[h]) / math.sqrt(d_h))
            heads.append(torch.softmax(z + bias[a:e, h][None, :] + mask, dim=1) @ v[a:e, kv])
        outs.append(torch.stack(heads, dim=1))
    return torch.cat(outs, dim=0), (q, k, v, bias)


def test_attention_bwd_with_per_head_gates_matches_torch_autograd():
    Q, K, V, _, cu, tau, beta = _rand_attn(70, (8, 13))
    G = np.random.default_rng(71).uniform(0.02, 1.0, (Q.shape[0], 4))
    dO = np.random.default_rng(72).standard_normal(Q.shape)
    dQ, dK, dV, dbias = O.gated_attention_bwd(Q, K, V, G, dO, cu, tau, beta)
    out, (q, k, v, bias) = _torch_forward_heads(Q, K, V, G, cu, tau, beta)
    (out * torch.from_numpy(dO)).sum().backward()
    for got, ref in ((dQ, q.grad), (dK, k.grad), (dV, v.grad), (dbias, bias.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)
    lse = O.gated_attention_lse(Q, K, G, cu, tau, beta)
    assert np.all(np.isfinite(lse))


def test_gate_score_grad_per_head_by_finite_differences():
    # ds[j, c] through g[:, c] = sigmoid(s[:, c]), for two gate heads shared by two query heads each
    Q, K, V, _, cu, tau, beta = _rand_attn(73, (9,))
    rng = np.random.default_rng(74)
    S = rng.standard_normal((9, 2))
    sig = lambda x: 1.0 / (1.0 + np.exp(-x))
    dO = rng.standard_normal(Q.shape)
    _, _, _, dbias = O.gated_attention_bwd(Q, K, V, sig(S), dO, cu, tau, beta)
    kept = np.arange(9) * 3 + 1
    ds = O.gate_score_grad(dbias, beta, sig(S), kept, 27)
    assert ds.shape == (27, 2) and np.all(np.delete(ds, kept, axis=0) == 0.0)
    loss = lambda SS: float(np.sum(dO * O.gated_attention(Q, K, V, sig(SS), cu, tau, beta)))
    for j, c in ((0, 0), (4, 1), (8, 1), (3, 0)):
        up, dn = S.copy(), S.copy()
        up[j, c] += 1e-6
        dn[j, c] -= 1e-6
        assert abs((loss(up) - loss(dn)) / 2e-6 - ds[kept[j], c]) < 1e-6


# ---------------------------------------------------------------------------
# Planted slips in the oracle's own source: each edit below makes one plausible mistake
# in a copy of an oracle function (a dropped term, a transposed operand, a wrong axis,
# sign or scale), and the pin that guards that function must reject the copy. The
# unedited function passes the same check, so the pin, not the harness, tells them apart.
# ---------------------------------------------------------------------------

def _planted_oracle(fn, edits):
    """fn with each (old, new) edit applied to its source (old found exactly once), compiled
    in the oracle module's namespace."""
    src = textwrap.dedent(inspect.getsource(fn))
    for old, new in edits:
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    ns = dict(vars(O))
    exec(compile(src, f"<planted {fn.__name__}>", "exec"), ns)
    return ns[fn.__name__]


def _close_all(got, refs, rtol, atol):
    return all(np.allclose(a, r, rtol=rtol, atol=atol) for a, r in zip(got, refs))


_BWD_SLIPS = {
    "row_dot_dropped": [("dX = P * (dP - D)", "dX = P * dP")],
    "row_dot_without_P": [("D = np.sum(do * o, axis=1, keepdims=True)", "D = np.sum(dP, axis=1, keepdims=True)")],
    "dV_untransposed": [("dV[a:e, kv] += P.T @ do", "dV[a:e, kv] += P @ do")],
    "dK_unscaled": [("dK[a:e, kv] += float(tau[h]) * c * (dX.T @ q)", "dK[a:e, kv] += float(tau[h]) * (dX.T @ q)")],
    "dQ_transposed": [("dQ[a:e, h] = float(tau[h]) * c * (dX @ k)", "dQ[a:e, h] = float(tau[h]) * c * (dX.T @ k)")],
    "dbias_over_queries": [("dbias[a:e, h] = dX.sum(axis=0)", "dbias[a:e, h] = dX.sum(axis=1)")],
    "kv_head_modulo": [("kv = h // group", "kv = h % H_kv")],
}


@pytest.mark.parametrize("kind", sorted(_BWD_SLIPS))
def test_planted_backward_slips_fail_the_autograd_pin(kind):
    Q, K, V, g, cu, tau, beta = _rand_attn(51, (9, 1, 14))
    dO = np.random.default_rng(52).standard_normal(Q.shape)
    out, (q, k, v, bias) = _torch_forward(Q, K, V, g, cu, tau, beta)
    (out * torch.from_numpy(dO)).sum().backward()
    refs = [t.grad.numpy() for t in (q, k, v, bias)]
    assert _close_all(O.gated_attention_bwd(Q, K, V, g, dO, cu, tau, beta), refs, 1e-10, 1e-12)
    bad = _planted_oracle(O.gated_attention_bwd, _BWD_SLIPS[kind])
    assert not _close_all(bad(Q, K, V, g, dO, cu, tau, beta), refs, 1e-10, 1e-12)


_SCORE_SLIPS = {
    "silu_as_sigmoid": [("a = u / (1.0 + np.exp(-u))", "a = 1.0 / (1.0 + np.exp(-u))")],
    "gate_sign": [("g = 1.0 / (1.0 + np.exp(-s))", "g = 1.0 / (1.0 + np.exp(s))")],
    "instruction_gate_not_one": [("g = np.where(keep if g.ndim == 1 else keep[:, None], 1.0, g)", "g = g")],
    "b1_dropped": [("u = u + np.asarray(b1, dtype=np.float64)[None, :]", "u = u")],
    "b2_dropped": [("s = a @ w2 + float(b2)", "s = a @ w2")],
}


@pytest.mark.parametrize("kind", sorted(_SCORE_SLIPS))
def test_planted_gate_score_slips_fail_the_torch_pin(kind):
    wl = I.WORKLOADS["tiny"]
    gi = I.make_gate_inputs(wl)
    h, W1, w2 = (I.bf16_bits_to_f64(gi[k]) for k in ("h", "W1", "w2"))
    b1, b2 = np.random.default_rng(5).standard_normal(wl.d_g), 0.3
    ref_s = F.linear(F.silu(F.linear(torch.from_numpy(h), torch.from_numpy(W1), torch.from_numpy(b1))),
                     torch.from_numpy(w2)[None, :]).squeeze(1) + b2
    ref_g = torch.sigmoid(ref_s)
    ref_g[torch.from_numpy(gi["instr_mask"].astype(bool))] = 1.0
    refs = (ref_s.numpy(), ref_g.numpy())
    assert _close_all(O.gate_score(h, W1, w2, gi["instr_mask"], b1, b2), refs, 1e-12, 1e-12)
    bad = _planted_oracle(O.gate_score, _SCORE_SLIPS[kind])
    assert not _close_all(bad(h, W1, w2, gi["instr_mask"], b1, b2), refs, 1e-12, 1e-12)


_NORM_SLIPS = {
    "rms_over_every_row": [("doc = [j for j in range(a, e) if instr_mask[j] == 0]", "doc = list(range(a, e))")],
    "variance_not_rooted": [("b[j] = s[j] / math.sqrt(ms + eps)", "b[j] = s[j] / (ms + eps)")],
    "mean_absolute_value": [("ms = sum(s[j] * s[j] for j in doc) / len(doc)", "ms = sum(abs(s[j]) for j in doc) / len(doc)")],
}


@pytest.mark.parametrize("kind", sorted(_NORM_SLIPS))
def test_planted_normalisation_slips_fail_the_closed_form(kind):
    fx = _golden("normalized_scores_closed_form.json")
    args = (np.array(fx["s"]), np.array(fx["instr_mask"]), fx["cu_seqlens"])
    assert np.allclose(O.normalize_scores(*args, eps=0.0), fx["b"], rtol=0, atol=1e-15)
    bad = _planted_oracle(O.normalize_scores, _NORM_SLIPS[kind])
    assert not np.allclose(bad(*args, eps=0.0), fx["b"], rtol=0, atol=1e-15)


_GRAD_SLIPS = {
    "sigmoid_factor_dropped": [("ds[kept_idx] = (dbias @ beta) * (1.0 - g_kept)", "ds[kept_idx] = dbias @ beta")],
    "factor_g_not_one_minus_g": [("ds[kept_idx] = (dbias @ beta) * (1.0 - g_kept)", "ds[kept_idx] = (dbias @ beta) * g_kept")],
    "beta_dropped": [("ds[kept_idx] = (dbias @ beta) * (1.0 - g_kept)", "ds[kept_idx] = dbias.sum(axis=1) * (1.0 - g_kept)")],
}


@pytest.mark.parametrize("kind", sorted(_GRAD_SLIPS))
def test_planted_score_gradient_slips_fail_finite_differences(kind):
    Q, K, V, _, cu, tau, beta = _rand_attn(55, (10,))
    rng = np.random.default_rng(56)
    s = rng.standard_normal(10)
    sig = lambda x: 1.0 / (1.0 + np.exp(-x))
    dO = rng.standard_normal(Q.shape)
    _, _, _, dbias = O.gated_attention_bwd(Q, K, V, sig(s), dO, cu, tau, beta)
    kept = np.arange(10) * 2
    loss = lambda ss: float(np.sum(dO * O.gated_attention(Q, K, V, sig(ss), cu, tau, beta)))
    fd = []
    for j in range(10):
        up, dn = s.copy(), s.copy()
        up[j] += 1e-6
        dn[j] -= 1e-6
        fd.append((loss(up) - loss(dn)) / 2e-6)
    matches = lambda ds: np.allclose(ds[kept], fd, rtol=0, atol=1e-6)
    assert matches(O.gate_score_grad(dbias, beta, sig(s), kept, 20))
    assert not matches(_planted_oracle(O.gate_score_grad, _GRAD_SLIPS[kind])(dbias, beta, sig(s), kept, 20))


_ROPE_SLIPS = {
    "rotation_sign": [("x1 * c - x2 * s", "x1 * c + x2 * s")],
    "frequency_exponent": [("theta ** (-2.0 * i / d_h)", "theta ** (-1.0 * i / d_h)")],
    "interleaved_pairs": [("x1 = X[..., :half]", "x1 = X[..., 0::2]"), ("x2 = X[..., half:]", "x2 = X[..., 1::2]")],
}


@pytest.mark.parametrize("kind", sorted(_ROPE_SLIPS))
def test_planted_rope_slips_fail_the_complex_rotation(kind):
    rng = np.random.default_rng(19)
    X = rng.standard_normal((7, 3, 8))
    pos = rng.integers(0, 5000, 7)
    z = X[..., :4] + 1j * X[..., 4:]
    zr = z * np.exp(1j * pos[:, None, None] * (1.0e6 ** (-np.arange(4) * 2.0 / 8))[None, None, :])
    ref = np.concatenate([zr.real, zr.imag], axis=-1)
    assert np.allclose(O.apply_rope(X, pos, 1.0e6), ref, rtol=1e-12, atol=1e-12)
    assert not np.allclose(_planted_oracle(O.apply_rope, _ROPE_SLIPS[kind])(X, pos, 1.0e6), ref,
                           rtol=1e-12, atol=1e-12)


_LSE_SLIPS = {
    "no_causal_mask": [("x = np.where(causal,", "x = np.where(np.ones_like(causal),")],
    "bias_dropped": [("+ bias[None, :],", ",")],
    "max_not_added_back": [("out[a:e, h][fin] = mx[fin] + np.log(", "out[a:e, h][fin] = np.log(")],
}


@pytest.mark.parametrize("kind", sorted(_LSE_SLIPS))
def test_planted_lse_slips_fail_torch_logsumexp(kind):
    Q, K, V, g, cu, tau, beta = _rand_attn(57, (6, 11))
    ref = np.full((Q.shape[0], Q.shape[1]), np.nan)
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        for h in range(Q.shape[1]):
            z = torch.from_numpy(Q[a:e, h] @ K[a:e, h // 2].T) * (tau[h] / math.sqrt(Q.shape[2]))
            z = z + beta[h] * torch.log(torch.from_numpy(g[a:e]))[None, :]
            z = z.masked_fill(torch.ones(e - a, e - a, dtype=torch.bool).triu(1), float("-inf"))
            ref[a:e, h] = torch.logsumexp(z, dim=1).numpy()
    assert np.allclose(O.gated_attention_lse(Q, K, g, cu, tau, beta), ref, rtol=1e-12, atol=1e-12)
    bad = _planted_oracle(O.gated_attention_lse, _LSE_SLIPS[kind])
    assert not np.allclose(bad(Q, K, g, cu, tau, beta), ref, rtol=1e-12, atol=1e-12)


def test_planted_aggregation_slip_fails_the_mean_head_pin():
    wl, gi, h, W1, W2, b1, b2 = _heads_case(4, seed=62)
    s, _ = O.gate_score(h, W1, W2, gi["instr_mask"], b1, b2)
    s1, _ = O.gate_score(h, W1, W2.mean(axis=0), gi["instr_mask"], b1, float(b2.mean()))
    assert np.allclose(O.aggregate_heads(s), s1, rtol=1e-12, atol=1e-12)
    bad = _planted_oracle(O.aggregate_heads, [("s.mean(axis=1)", "s.sum(axis=1)")])
    assert not np.allclose(bad(s), s1, rtol=1e-12, atol=1e-12)


_SELECT_SLIPS = {
    "budget_counts_instruction_rows": [("K_b = min(K, len(prunable))",
                                        "K_b = max(0, min(K - len(keep_always), len(prunable)))")],
    "instruction_rows_dropped": [("keep = sorted(selected + keep_always)", "keep = sorted(selected)")],
    "kept_in_score_order": [("keep = sorted(selected + keep_always)", "keep = selected + sorted(keep_always)")],
    "smallest_scores_kept": [("return (0, -(x + 0.0))", "return (0, x + 0.0)")],
    "negative_zero_below_zero": [("return (0, -(x + 0.0))", "return (0, -x, math.copysign(1.0, x) < 0)")],
}


@pytest.mark.parametrize("kind", sorted(_SELECT_SLIPS))
def test_planted_selection_slips_fail_brute_force(kind):
    # every budget from 0 to one past the largest document count, on every tiny case
    def agrees(select):
        for s, mask, cu in _tiny_select_cases():
            max_doc = max(int(np.sum(mask[cu[b]:cu[b + 1]] == 0)) for b in range(len(cu) - 1))
            for K in range(0, max_doc + 2):
                kept, cu_k = select(s, mask, cu, K)
                ref, ref_cu = _brute_force_keep(s, mask, cu, K)
                if kept.tolist() != ref.tolist() or cu_k.tolist() != ref_cu.tolist():
                    return False
        return True
    assert agrees(O.topk_select)
    fn = O._rank_key if kind in ("smallest_scores_kept", "negative_zero_below_zero") else O.topk_select
    bad = _planted_oracle(fn, _SELECT_SLIPS[kind])
    if fn is O._rank_key:  # the key function is a helper: select with the planted key in place
        ns = dict(vars(O))
        ns["_rank_key"] = bad
        exec(compile(textwrap.dedent(inspect.getsource(O.topk_select)), "<planted topk_select>", "exec"), ns)
        bad = ns["topk_select"]
    assert not agrees(bad)


_GATHER_SLIPS = {
    "positions_from_zero_over_the_batch": [
        ("p_k = (kept_idx - np.asarray(cu_seqlens, dtype=np.int64)[seq_of]).astype(np.int32)",
         "p_k = kept_idx.astype(np.int32)")],
    "positions_of_the_kept_list": [
        ("p_k = (kept_idx - np.asarray(cu_seqlens, dtype=np.int64)[seq_of]).astype(np.int32)",
         "p_k = np.arange(len(kept_idx), dtype=np.int32)")],
    "gate_values_not_gathered": [("g_k = np.asarray(g)[kept_idx]", "g_k = np.asarray(g)[:len(kept_idx)]")],
}


@pytest.mark.parametrize("kind", sorted(_GATHER_SLIPS))
def test_planted_gather_slips_fail_the_original_id_pin(kind):
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(20, 30), instr_lens=(4, 6))
    cu = I.cu_seqlens_of(wl.seq_lens)
    rng = np.random.default_rng(3)
    kept = np.sort(rng.choice(wl.T_total, size=25, replace=False)).astype(np.int32)
    h = rng.standard_normal((wl.T_total, 8))
    g = rng.random(wl.T_total)
    want_pos = [j if j < cu[1] else j - cu[1] for j in kept]

    def agrees(gather):
        hk, pk, gk = gather(h, None, g, kept, cu)
        return (pk.tolist() == want_pos and np.array_equal(hk, h[kept]) and np.array_equal(gk, g[kept]))
    assert agrees(O.gather_kept)
    assert not agrees(_planted_oracle(O.gather_kept, _GATHER_SLIPS[kind]))


_TWO_BUDGET_SLIPS = {
    "pruned_offsets_not_shifted": [('T + prune["cu_kept"][1:]', 'prune["cu_kept"][1:]')],
    "pruned_half_first": [('cat = lambda k: np.concatenate([full[k], prune[k]])',
                           'cat = lambda k: np.concatenate([prune[k], full[k]])')],
    "full_budget_of_one_sequence": [("cu_seqlens, len(instr_mask), b1, b2)",
                                     "cu_seqlens, int(cu_seqlens[1] - cu_seqlens[0]) // 2, b1, b2)")],
}


@pytest.mark.parametrize("kind", sorted(_TWO_BUDGET_SLIPS))
def test_planted_two_budget_slips_fail_the_pack_invariants(kind):
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(50, 0, 33), instr_lens=(4, 2, 6), d=64, d_g=32)
    gi = I.make_gate_inputs(wl)
    h = I.bf16_bits_to_f64(gi["h"])
    W1, w2 = I.bf16_bits_to_f64(gi["W1"]), I.bf16_bits_to_f64(gi["w2"])
    T, B = wl.T_total, wl.B

    def agrees(pack):
        out = pack(h, gi["pos"], W1, w2, gi["instr_mask"], gi["cu_seqlens"], 7)
        cu = out["cu_packed"]
        return (out["kept_idx"][:T].tolist() == list(range(T))
                and cu[:B + 1].tolist() == gi["cu_seqlens"].tolist()
                and all(cu[B + b + 1] - cu[B + b] == min(7, wl.doc_lens[b]) + wl.instr_lens[b] for b in range(B))
                and np.array_equal(out["h_kept"], h[out["kept_idx"]]))
    assert agrees(O.two_budget_prune_layer)
    assert not agrees(_planted_oracle(O.two_budget_prune_layer, _TWO_BUDGET_SLIPS[kind]))
