"""GPU parity: per-head gate scores with uniform head aggregation for selection (TokenGate deep
dive, section 3.4: a per-head bias; "uniform head aggregation for selection"), through every
stage that carries the gate: scoring, normalisation, top-K on the head mean, gather, the
log-gate and Eq. (8) attention, and the backward. Against the fp64 oracle.

Tolerances are the single-head ones: scores 2e-3 + 1e-3 relative (the head mean is a mean of
values each within that bar), gates 1e-2, normalised scores 1e-5 relative + 1e-6, attention
2e-2 max-abs and 1e-2 mean-relative; the backward uses the derived bound of its own tests."""
import numpy as np
import pytest
import torch

from learned_token_pruning_07_b300 import binding as tg
from learned_token_pruning_07_b300 import inputs as I
from oracle import tokengate_oracle as O
from tests._helpers import (ATTN_MAX_ABS, ATTN_MEAN_REL, G_ATOL, S_ATOL, S_RTOL, attention_close, bf16_dev_to_f64,
                            dev, host, sampled_rows, status_word, zeros_i32)
from tests.test_gpu_backward import _rounding_bounds

pytestmark = pytest.mark.gpu

SENTINEL = 12345.0


def _sentinel(*shape):
    return torch.full(shape, SENTINEL, dtype=torch.float32, device="cuda")


def _score_heads(wl, H_g, b1=None, rmsnorm=False, ln_eps=1e-6, rows=None):
    gi = I.make_gate_inputs(wl)
    hw = I.make_gate_head_weights(wl, H_g)
    T = wl.T_total
    h_bits = gi["h"]
    W1_bits = gi["W1"]
    ln_bits = None
    if rmsnorm:
        rng = np.random.default_rng(71)
        scale = rng.uniform(0.2, 8.0, T).astype(np.float32)
        h_bits = I.f32_to_bf16_bits(I.bf16_bits_to_f32(gi["h"]) * scale[:, None])
        ln_bits = I.f32_to_bf16_bits(rng.uniform(0.5, 1.5, wl.d).astype(np.float32))
        W1f = torch.zeros_like(dev(gi["W1"]))
        tg.fold_rmsnorm_weight(dev(gi["W1"]), dev(ln_bits), W1f)
        W1_dev = W1f
    else:
        W1_dev = dev(W1_bits)
    s = _sentinel(T + 8, H_g)
    g = _sentinel(T + 8, H_g)
    sel = _sentinel(T + 8)
    st = status_word()
    tg.gate_score_heads(dev(h_bits), W1_dev, dev(hw["W2"]), s[:T], sel[:T], g_heads=g[:T],
                        instr_mask=dev(gi["instr_mask"]), b1=None if b1 is None else dev(b1.astype(np.float32)),
                        b2=hw["b2"], rmsnorm=rmsnorm, ln_eps=ln_eps, status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    s_h, g_h, sel_h = host(s), host(g), host(sel)
    assert np.all(s_h[T:] == SENTINEL) and np.all(g_h[T:] == SENTINEL) and np.all(sel_h[T:] == SENTINEL)
    r = slice(None) if rows is None else rows
    W2 = I.bf16_bits_to_f64(hw["W2"])
    ref_s, ref_g = O.gate_score(I.bf16_bits_to_f64(h_bits[r]), I.bf16_bits_to_f64(W1_bits), W2,
                                gi["instr_mask"][r], None if b1 is None else b1.astype(np.float32).astype(np.float64),
                                hw["b2"].astype(np.float64),
                                ln_weight=None if ln_bits is None else I.bf16_bits_to_f64(ln_bits), ln_eps=ln_eps)
    tol = S_ATOL + S_RTOL * np.abs(ref_s)
    if rmsnorm:
        # the folded weight's bf16 rounding, per head: 6 sigma of its first-order effect (the
        # single-head derivation with w2 replaced by the head's row of W2)
        h64 = I.bf16_bits_to_f64(h_bits[r])
        x = h64 / np.sqrt(np.mean(h64 * h64, axis=1, keepdims=True) + ln_eps)
        W1w = I.bf16_bits_to_f64(W1_bits) * I.bf16_bits_to_f64(ln_bits)[None, :]
        var = ((W1w ** 2) @ (x ** 2).T).T @ (W2 ** 2).T                                  # [rows, H_g]
        tol = tol + 6.0 * 1.1 * 2.0 ** -8 / np.sqrt(3.0) * np.sqrt(var)
    got_s = s_h[:T][r]
    assert np.all(np.abs(got_s - ref_s) <= tol)
    np.testing.assert_allclose(g_h[:T][r], ref_g, rtol=0, atol=G_ATOL)
    ref_sel = O.aggregate_heads(ref_s)
    assert np.all(np.abs(sel_h[:T][r] - ref_sel) <= tol.mean(axis=1) + 1e-6)
    # the head mean is formed from the GPU's own per-head scores: sum in head order, then / H_g
    own = np.zeros(got_s.shape[0], np.float32)
    for c in range(H_g):
        own = (own + got_s[:, c]).astype(np.float32)
    np.testing.assert_array_equal(sel_h[:T][r], (own / np.float32(H_g)).astype(np.float32))
    return gi, hw, s_h[:T], g_h[:T], sel_h[:T]


@pytest.mark.parametrize("H_g", [2, 3, 4, 16])
def test_score_heads_tiny_with_biases(H_g):
    wl = I.WORKLOADS["tiny"]
    b1 = np.random.default_rng(72).standard_normal(wl.d_g) * 0.3
    _score_heads(wl, H_g, b1=b1)


def test_score_heads_ragged_tail_two_slices():
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(900,), instr_lens=(17,), d=512, d_g=384)
    _score_heads(wl, 8)


def test_score_heads_slices_of_an_odd_multiple_of_16():
    # d_g = 480: two slices of 240 columns, each ending with a 16-column chunk
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(700,), instr_lens=(9,), d=256, d_g=480)
    _score_heads(wl, 4)
    _score_heads(wl, 16, rmsnorm=True)


def test_score_heads_clusters_of_four_several_tiles():
    # 80 pair tiles with 8 gate heads: clusters of four, several tiles each (see test_gpu_score)
    wl = I.with_changes(I.WORKLOADS["sweep_32k"], doc_lens=(20224,), instr_lens=(256,))
    rng = np.random.default_rng(31)
    rows = np.unique(np.concatenate([np.arange(0, 300), np.arange(wl.T_total - 300, wl.T_total),
                                     rng.integers(0, wl.T_total, 1500)]))
    _score_heads(wl, 8, rows=rows)


def test_score_heads_qwen3_gate_layer_8k():
    _score_heads(I.WORKLOADS["qwen3_1p7b_8k"], 16)


@pytest.mark.parametrize("H_g", [1, 8])
def test_score_heads_with_fused_rmsnorm(H_g):
    _score_heads(I.WORKLOADS["tiny"], H_g, rmsnorm=True)


def test_score_heads_full_size_sampled_rows():
    wl = I.WORKLOADS["sweep_32k"]
    rng = np.random.default_rng(73)
    rows = np.unique(np.concatenate([np.arange(0, 200), np.arange(wl.T_total - 200, wl.T_total),
                                     rng.integers(0, wl.T_total, 1500)]))
    _score_heads(wl, 8, rows=rows)


@pytest.mark.parametrize("H_g", [2, 5, 16])
def test_normalize_per_head_and_head_mean(H_g):
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(0, 1, 37, 600), instr_lens=(5, 0, 2, 9),
                        instr_where="scattered")
    T = wl.T_total
    mask, cu = I.make_instr_mask(wl), I.cu_seqlens_of(wl.seq_lens)
    s = np.stack([I.make_scores(wl, tag_extra=c) for c in range(H_g)], axis=1).astype(np.float32)
    s *= np.linspace(0.5, 4.0, H_g, dtype=np.float32)[None, :]
    b = _sentinel(T + 4, H_g)
    bsel = _sentinel(T + 4)
    st = status_word()
    tg.normalize_scores(dev(s), dev(cu), b[:T], instr_mask=dev(mask), eps=1e-6, b_sel=bsel[:T], status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    got, got_sel = host(b), host(bsel)
    assert np.all(got[T:] == SENTINEL) and np.all(got_sel[T:] == SENTINEL)
    ref = O.normalize_scores(s, mask, cu, eps=1e-6)
    np.testing.assert_allclose(got[:T], ref, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(got_sel[:T], O.aggregate_heads(ref), rtol=1e-5, atol=1e-6)
    assert np.all(got[:T][mask == 1] == 0.0) and np.all(got_sel[:T][mask == 1] == 0.0)


def test_prune_layer_heads_selects_on_the_head_mean():
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    H_g, K = 8, wl.K
    gi = I.make_gate_inputs(wl)
    hw = I.make_gate_head_weights(wl, H_g)
    T, B = wl.T_total, wl.B
    s = torch.zeros((T, H_g), dtype=torch.float32, device="cuda")
    g = torch.zeros((T, H_g), dtype=torch.float32, device="cuda")
    sel = torch.zeros(T, dtype=torch.float32, device="cuda")
    kept, cu_kept = zeros_i32(T), zeros_i32(B + 1)
    h_kept = torch.zeros((T, wl.d), dtype=torch.int16, device="cuda")
    pos_kept = zeros_i32(T)
    g_kept = _sentinel(T, H_g)
    st = status_word()
    tg.gate_prune_layer_heads(dev(gi["h"]), dev(gi["cu_seqlens"]), dev(gi["W1"]), dev(hw["W2"]), K, s, g, sel,
                              kept, cu_kept, h_kept, pos_kept=pos_kept, g_kept=g_kept, pos=dev(gi["pos"]),
                              instr_mask=dev(gi["instr_mask"]), b2=hw["b2"], status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    s_h, g_h, sel_h = host(s), host(g), host(sel)
    ref = O.gate_prune_layer(I.bf16_bits_to_f64(gi["h"]), gi["pos"], I.bf16_bits_to_f64(gi["W1"]),
                             I.bf16_bits_to_f64(hw["W2"]), gi["instr_mask"], gi["cu_seqlens"], K,
                             b2=hw["b2"].astype(np.float64))
    np.testing.assert_allclose(s_h, ref["s"], rtol=S_RTOL, atol=S_ATOL)
    cuk = host(cu_kept)
    assert cuk.tolist() == ref["cu_kept"].tolist()
    M = int(cuk[-1])
    kept_h = host(kept)[:M]
    mask = gi["instr_mask"]
    gk = set(kept_h.tolist())
    doc = np.nonzero(mask == 0)[0]
    kd = [j for j in doc if j in gk]
    pd = [j for j in doc if j not in gk]
    # top-K on the GPU's own head mean; the oracle's set differs only at the threshold
    assert set(np.nonzero(mask)[0].tolist()) <= gk and np.all(np.diff(kept_h) > 0)
    assert sel_h[kd].min() >= sel_h[pd].max()
    ref_sel = O.aggregate_heads(ref["s"])
    diff = gk ^ set(ref["kept_idx"].tolist())
    if diff:
        thr = np.sort(ref_sel[doc])[::-1][K - 1]
        assert all(abs(ref_sel[j] - thr) <= 2 * (S_ATOL + S_RTOL * abs(thr)) for j in diff), sorted(diff)
    assert np.array_equal(host(h_kept)[:M], gi["h"][kept_h])
    assert np.array_equal(host(pos_kept)[:M], gi["pos"][kept_h])
    got_gk = host(g_kept)
    assert np.array_equal(got_gk[:M], g_h[kept_h]) and np.all(got_gk[M:] == SENTINEL)


def _attn_heads(wl, lens, H_g, rows=None, seed=0):
    cu = I.cu_seqlens_of(lens)
    M = int(cu[-1])
    at = I.make_attention_inputs(wl, M, tag_extra=seed)
    G = I.make_head_gates(wl, M, H_g, tag_extra=seed)
    O_d = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    st = status_word()
    tg.gated_attention(dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(cu), at["tau"], at["beta"], O_d,
                       max_seqlen=max(lens), g=dev(G), status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    got = bf16_dev_to_f64(O_d)
    want = O.gated_attention(I.bf16_bits_to_f64(at["Q"]), I.bf16_bits_to_f64(at["K"]), I.bf16_bits_to_f64(at["V"]),
                             G.astype(np.float64), cu, at["tau"].astype(np.float64), at["beta"].astype(np.float64),
                             rows=rows)
    mx, mr = attention_close(got if rows is None else got[rows], want)
    assert mx <= ATTN_MAX_ABS and mr <= ATTN_MEAN_REL, (mx, mr)


@pytest.mark.parametrize("H_g", [2, 8, 16])
def test_attention_with_per_head_gates(H_g):
    _attn_heads(I.WORKLOADS["qwen3_1p7b_8k"], [300, 129, 1, 0, 640], H_g, seed=H_g)


def test_attention_per_head_gates_odd_group_and_dh64():
    # a group of 3 query heads per kv head (one head per CTA) with 6 gate heads; d_h = 64
    _attn_heads(I.with_changes(I.WORKLOADS["qwen3_1p7b_8k"], H_q=6, H_kv=2), [257, 130], 6, seed=3)
    _attn_heads(I.WORKLOADS["tiny"], [200, 77], 2, seed=4)


def test_attention_per_head_gates_long_sequence_sampled():
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    lens = [4100, 2000]
    cu = I.cu_seqlens_of(lens)
    rows = sampled_rows(cu, [], 200, seed=5)
    _attn_heads(wl, lens, 4, rows=rows, seed=5)


def test_eq8_attention_with_per_head_bias():
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    lens = [300, 1, 520]
    cu = I.cu_seqlens_of(lens)
    M = int(cu[-1])
    at = I.make_attention_inputs(wl, M, tag_extra=6)
    rng = np.random.default_rng(76)
    Bh = rng.standard_normal((M, 4)).astype(np.float32)
    pos = np.concatenate([np.cumsum(rng.integers(1, 9, n)) - 1 for n in lens]).astype(np.int32)
    gain = rng.uniform(0.2, 1.5, wl.H_q).astype(np.float32)
    temp = rng.uniform(0.5, 1.5, wl.H_q).astype(np.float32)
    O_d = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    st = status_word()
    tg.gated_attention_eq8(dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(cu), dev(pos), gain, temp, O_d,
                           max_seqlen=max(lens), b=dev(Bh), status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    rows = sampled_rows(cu, [], 150, seed=7)
    want = O.gated_attention_eq8(I.bf16_bits_to_f64(at["Q"]), I.bf16_bits_to_f64(at["K"]),
                                 I.bf16_bits_to_f64(at["V"]), Bh.astype(np.float64), pos, cu,
                                 gain.astype(np.float64), temp.astype(np.float64), rows=rows)
    mx, mr = attention_close(bf16_dev_to_f64(O_d)[rows], want)
    assert mx <= ATTN_MAX_ABS and mr <= ATTN_MEAN_REL, (mx, mr)


def test_gather_moves_every_gate_head():
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(300, 41), instr_lens=(12, 3))
    H_g = 16
    gi = I.make_gate_inputs(wl)
    T, B = wl.T_total, wl.B
    G = I.make_head_gates(wl, T, H_g)
    rng = np.random.default_rng(77)
    cu = gi["cu_seqlens"]
    kept = np.sort(rng.choice(T, 150, replace=False)).astype(np.int32)
    cu_kept = np.array([0, int(np.sum(kept < cu[1])), 150], np.int32)
    h_kept = torch.zeros((T, wl.d), dtype=torch.int16, device="cuda")
    g_kept = _sentinel(T, H_g)
    st = status_word()
    tg.gather_kept(dev(gi["h"]), dev(cu), dev(kept), dev(cu_kept), h_kept, g=dev(G), g_kept=g_kept, status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    got = host(g_kept)
    assert np.array_equal(got[:150], G[kept]) and np.all(got[150:] == SENTINEL)
    assert np.array_equal(host(h_kept)[:150], gi["h"][kept])


def test_backward_with_per_head_gates_and_score_gradient():
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    lens = [200, 1, 131]
    H_g = 4
    cu = I.cu_seqlens_of(lens)
    M = int(cu[-1])
    at = I.make_attention_inputs(wl, M, tag_extra=8)
    G = I.make_head_gates(wl, M, H_g, tag_extra=8)
    dO = I.f32_to_bf16_bits(np.random.default_rng(78).standard_normal((M, wl.H_q, wl.d_h)).astype(np.float32))
    Qd, Kd, Vd, Gd, cud = dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(G), dev(cu)
    O_d = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    lse = torch.zeros((M, wl.H_q), dtype=torch.float32, device="cuda")
    st = status_word()
    tg.gated_attention_lse(Qd, Kd, Vd, cud, at["tau"], at["beta"], O_d, lse, max_seqlen=max(lens), g=Gd, status=st)
    out = [torch.zeros(sh, dtype=torch.float32, device="cuda")
           for sh in ((M, wl.H_q, wl.d_h), (M, wl.H_kv, wl.d_h), (M, wl.H_kv, wl.d_h), (M, wl.H_q))]
    tg.gated_attention_bwd(Qd, Kd, Vd, O_d, dev(dO), lse, cud, at["tau"], at["beta"], *out, max_seqlen=max(lens),
                           g=Gd, status=st)
    T = 2 * M
    kept = np.sort(np.random.default_rng(79).choice(T, M, replace=False)).astype(np.int32)
    ds = torch.zeros((T, H_g), dtype=torch.float32, device="cuda")
    tg.gate_score_grad(out[3], at["beta"], Gd, dev(kept), cud, ds)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    Q64, K64, V64 = (I.bf16_bits_to_f64(at[k]) for k in ("Q", "K", "V"))
    G64, dO64 = G.astype(np.float64), I.bf16_bits_to_f64(dO)
    tau, beta = at["tau"].astype(np.float64), at["beta"].astype(np.float64)
    np.testing.assert_allclose(host(lse), O.gated_attention_lse(Q64, K64, G64, cu, tau, beta), rtol=0, atol=1e-3)
    ref = O.gated_attention_bwd(Q64, K64, V64, G64, dO64, cu, tau, beta)
    bounds = _rounding_bounds(Q64, K64, V64, G64, dO64, cu, tau, beta)
    for name, a, b, bnd in zip(("dQ", "dK", "dV", "dbias"), [host(t).astype(np.float64) for t in out], ref, bounds):
        tol = bnd + 1e-4 * float(np.max(np.abs(b))) + 1e-7
        assert np.all(np.abs(a - b) <= tol), (name, float(np.abs(a - b).max()))
    want = O.gate_score_grad(ref[3], beta, G64, kept, T)
    per = wl.H_q // H_g
    tol_ds = np.zeros((T, H_g))
    for c in range(H_g):
        hs = slice(c * per, (c + 1) * per)
        tol_ds[kept, c] = (bounds[3][:, hs] @ beta[hs]) * (1.0 - G64[:, c]) + 1e-4 * float(np.max(np.abs(want))) + 1e-7
    assert np.all(np.abs(host(ds) - want) <= tol_ds)
