"""GPU parity: gate scoring (tcgen05 GEMM + fused SiLU . w2 + sigmoid) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from learned_token_pruning_07_b300 import binding as tg
from learned_token_pruning_07_b300 import inputs as I
from oracle import tokengate_oracle as O
from tests._helpers import G_ATOL, S_ATOL, S_RTOL, dev, host, status_word

pytestmark = pytest.mark.gpu


def _score(wl, rows=None, b1=None, b2=0.0, with_mask=True):
    gi = I.make_gate_inputs(wl)
    T = wl.T_total
    s = torch.full((T + 32,), 12345.0, dtype=torch.float32, device="cuda")
    g = torch.full((T + 32,), 12345.0, dtype=torch.float32, device="cuda")
    st = status_word()
    mask = gi["instr_mask"] if with_mask else np.zeros(T, np.uint8)
    tg.gate_score(dev(gi["h"]), dev(gi["W1"]), dev(gi["w2"]), s[:T], g[:T],
                  instr_mask=dev(mask) if with_mask else None,
                  b1=None if b1 is None else dev(b1.astype(np.float32)), b2=b2, status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    s_h, g_h = host(s), host(g)
    assert np.all(s_h[T:] == 12345.0) and np.all(g_h[T:] == 12345.0)  # nothing past T
    h64 = I.bf16_bits_to_f64(gi["h"] if rows is None else gi["h"][rows])
    m = mask if rows is None else mask[rows]
    ref_s, ref_g = O.gate_score(h64, I.bf16_bits_to_f64(gi["W1"]), I.bf16_bits_to_f64(gi["w2"]), m,
                                None if b1 is None else b1.astype(np.float32).astype(np.float64), b2)
    got_s = s_h[:T] if rows is None else s_h[rows]
    got_g = g_h[:T] if rows is None else g_h[rows]
    np.testing.assert_allclose(got_s, ref_s, rtol=S_RTOL, atol=S_ATOL)
    np.testing.assert_allclose(got_g, ref_g, rtol=0, atol=G_ATOL)
    return got_s, ref_s


def test_score_tiny():
    _score(I.WORKLOADS["tiny"])


def test_score_ragged_tail_and_bias():
    # T not a multiple of the 128-row tile; d_g = 384 splits into two 192-wide MMAs
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(900,), instr_lens=(17,), d=512, d_g=384)
    b1 = np.random.default_rng(4).standard_normal(384) * 0.5
    _score(wl, b1=b1, b2=-0.25)


@pytest.mark.parametrize("d_g", [288, 480])
def test_score_slices_of_an_odd_multiple_of_16(d_g):
    # d_g > 256 splits into two slices of d_g / 2 = 144 or 240 columns: each ends with a
    # 16-column chunk, which must not pick up the next slice's columns; T spans 3 pair tiles
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(700,), instr_lens=(9,), d=256, d_g=d_g)
    b1 = np.random.default_rng(d_g).standard_normal(d_g) * 0.5
    _score(wl, b1=b1, b2=0.125)


def test_score_small_dg_no_mask():
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(130,), instr_lens=(0,), d=64, d_g=32)
    _score(wl, with_mask=False)


def test_score_qwen3_gate_layer_8k():
    got, ref = _score(I.WORKLOADS["qwen3_1p7b_8k"])
    # the score error is far below the spread of the scores, so top-K sees the same order
    assert np.max(np.abs(got - ref)) < 1e-3 * np.std(ref) + 1e-4


def test_score_full_size_sweep_sampled_rows():
    wl = I.WORKLOADS["sweep_32k"]
    rng = np.random.default_rng(21)
    rows = np.unique(np.concatenate([np.arange(0, 256), np.arange(wl.T_total - 300, wl.T_total),
                                     rng.integers(0, wl.T_total, 2000)]))
    _score(wl, rows=rows)


# ---------------------------------------------------------------------------
# Fused LN_2 (RMSNorm) in front of the score MLP (deep dive section 2, Eq. (1))
# ---------------------------------------------------------------------------

def _rmsnorm_case(wl, rows=None, ln_eps=1e-6):
    gi = I.make_gate_inputs(wl)
    T, d = wl.T_total, wl.d
    rng = np.random.default_rng(61)
    # the raw residual: rows of very different scale, so 1/rms matters
    scale = rng.uniform(0.2, 8.0, T).astype(np.float32)
    h_bits = I.f32_to_bf16_bits(I.bf16_bits_to_f32(gi["h"]) * scale[:, None])
    ln_bits = I.f32_to_bf16_bits(rng.uniform(0.5, 1.5, d).astype(np.float32))
    W1_d = dev(gi["W1"])
    W1f = torch.zeros_like(W1_d)
    tg.fold_rmsnorm_weight(W1_d, dev(ln_bits), W1f)
    torch.cuda.synchronize()
    # folding is a bf16 product rounded to nearest even
    want_fold = I.f32_to_bf16_bits(I.bf16_bits_to_f32(gi["W1"]) * I.bf16_bits_to_f32(ln_bits)[None, :])
    assert np.array_equal(host(W1f), want_fold)
    s = torch.full((T + 32,), 12345.0, dtype=torch.float32, device="cuda")
    g = torch.full((T + 32,), 12345.0, dtype=torch.float32, device="cuda")
    st = status_word()
    tg.gate_score_rmsnorm(dev(h_bits), W1f, dev(gi["w2"]), s[:T], g[:T], instr_mask=dev(gi["instr_mask"]),
                          ln_eps=ln_eps, status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    s_h, g_h = host(s), host(g)
    assert np.all(s_h[T:] == 12345.0) and np.all(g_h[T:] == 12345.0)
    sel = slice(None) if rows is None else rows
    ref_s, ref_g = O.gate_score(I.bf16_bits_to_f64(h_bits[sel]), I.bf16_bits_to_f64(gi["W1"]),
                                I.bf16_bits_to_f64(gi["w2"]), gi["instr_mask"][sel],
                                ln_weight=I.bf16_bits_to_f64(ln_bits), ln_eps=ln_eps)
    # The folded weight adds one bf16 rounding to every W1 diag(w_ln) entry: round to nearest with
    # an 8-bit significand, so a relative error e_kc of at most 2^-8 (the unit roundoff), taken as
    # uniform and independent per entry. To first order it moves s by
    # sum_k w2_k SiLU'(u_k) sum_c e_kc W1w_kc x_c, x = h / rms; with |SiLU'| <= 1.1 its standard
    # deviation is at most sigma = 1.1 * 2^-8 / sqrt(3) * sqrt(sum_k w2_k^2 sum_c (W1w_kc x_c)^2).
    # Allowed: 6 sigma on top of the plain score tolerance (fp32 accumulation).
    h64 = I.bf16_bits_to_f64(h_bits[sel])
    x = h64 / np.sqrt(np.mean(h64 * h64, axis=1, keepdims=True) + ln_eps)
    W1w = I.bf16_bits_to_f64(gi["W1"]) * I.bf16_bits_to_f64(ln_bits)[None, :]
    var = (I.bf16_bits_to_f64(gi["w2"]) ** 2) @ ((W1w ** 2) @ (x ** 2).T)        # [rows]
    sigma = 1.1 * 2.0 ** -8 / np.sqrt(3.0) * np.sqrt(var)
    err = np.abs(s_h[:T][sel] - ref_s)
    assert np.all(err <= 6.0 * sigma + S_ATOL + S_RTOL * np.abs(ref_s)), float(np.max(err / (6.0 * sigma + S_ATOL)))
    assert float(np.mean(err)) < 2.0 * float(np.mean(sigma)) + S_ATOL          # and typical errors are ~sigma
    np.testing.assert_allclose(g_h[:T][sel], ref_g, rtol=0, atol=G_ATOL)


def test_score_rmsnorm_tiny():
    _rmsnorm_case(I.WORKLOADS["tiny"])


def test_score_rmsnorm_ragged_tail_two_slices():
    _rmsnorm_case(I.with_changes(I.WORKLOADS["tiny"], doc_lens=(900,), instr_lens=(17,), d=512, d_g=384),
                  ln_eps=1e-5)


def test_score_rmsnorm_slices_of_an_odd_multiple_of_16():
    _rmsnorm_case(I.with_changes(I.WORKLOADS["tiny"], doc_lens=(700,), instr_lens=(9,), d=256, d_g=288))


def test_score_rmsnorm_clusters_of_four_several_tiles():
    # 20,480 rows = 80 pair tiles: the launch takes clusters of four (fewer slice-rounds than pairs),
    # each with several tiles, so slice 1's partial sums are handed over again after the reply
    wl = I.with_changes(I.WORKLOADS["sweep_32k"], doc_lens=(20224,), instr_lens=(256,))
    rng = np.random.default_rng(29)
    rows = np.unique(np.concatenate([np.arange(0, 300), np.arange(wl.T_total - 300, wl.T_total),
                                     rng.integers(0, wl.T_total, 1500)]))
    _rmsnorm_case(wl, rows=rows)


def test_score_rmsnorm_qwen3_gate_layer_8k():
    _rmsnorm_case(I.WORKLOADS["qwen3_1p7b_8k"])


def test_score_rmsnorm_full_size_sweep_sampled_rows():
    wl = I.WORKLOADS["sweep_32k"]
    rng = np.random.default_rng(62)
    rows = np.unique(np.concatenate([np.arange(0, 200), np.arange(wl.T_total - 200, wl.T_total),
                                     rng.integers(0, wl.T_total, 1500)]))
    _rmsnorm_case(wl, rows=rows)


@pytest.mark.parametrize("name,doc", [("sweep_32k", None), ("qwen3_1p7b_8k", None), ("sweep_32k", 20224)])
def test_score_is_bit_identical_across_runs(name, doc):
    # Pairs at 32K, clusters of four at 8K and 20K: every partial w2 dot is added in a fixed
    # order (column halves, then slices), so two runs give the same bits, with and without the
    # fused RMSNorm and with eight gate heads
    wl = I.WORKLOADS[name] if doc is None else I.with_changes(I.WORKLOADS[name], doc_lens=(doc,), instr_lens=(256,))
    gi = I.make_gate_inputs(wl)
    T = wl.T_total
    h, W1, w2, mask = dev(gi["h"]), dev(gi["W1"]), dev(gi["w2"]), dev(gi["instr_mask"])
    W2 = dev(I.make_gate_head_weights(wl, 8)["W2"])

    def run():
        s = torch.empty(T, dtype=torch.float32, device="cuda")
        g = torch.empty(T, dtype=torch.float32, device="cuda")
        tg.gate_score(h, W1, w2, s, g, instr_mask=mask)
        sn = torch.empty(T, dtype=torch.float32, device="cuda")
        tg.gate_score_rmsnorm(h, W1, w2, sn, instr_mask=mask)
        sh = torch.empty(T, 8, dtype=torch.float32, device="cuda")
        sel = torch.empty(T, dtype=torch.float32, device="cuda")
        tg.gate_score_heads(h, W1, W2, sh, sel, instr_mask=mask)
        torch.cuda.synchronize()
        return [host(x).view(np.uint32).copy() for x in (s, g, sn, sh, sel)]

    first, second = run(), run()
    for a, b in zip(first, second):
        assert np.array_equal(a, b)

