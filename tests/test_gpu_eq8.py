"""GPU parity: the paper's exact gate form (TokenGate deep dive, section 3.1 Eq. (3); section
3.2 Eqs. (7)-(8)) against the fp64 oracle.

Normalised scores: 1e-5 relative + 1e-6 absolute (one fp32 sum of squares per sequence).
Attention: 2e-2 max-abs and 1e-2 mean-relative, bf16 output against fp64."""
import numpy as np
import pytest
import torch

from learned_token_pruning_07_b300 import binding as tg
from learned_token_pruning_07_b300 import inputs as I
from oracle import tokengate_oracle as O
from tests._helpers import (ATTN_MAX_ABS, ATTN_MEAN_REL, S_ATOL, S_RTOL, attention_close, bf16_dev_to_f64, dev, host,
                            sampled_rows, status_word, zeros_i32)

pytestmark = pytest.mark.gpu


def _normalize(s, mask, cu, eps=1e-6):
    b = torch.full((len(s) + 16,), 777.0, dtype=torch.float32, device="cuda")
    st = status_word()
    tg.normalize_scores(dev(s), dev(cu), b[:len(s)], instr_mask=None if mask is None else dev(mask), eps=eps,
                        status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    out = host(b)
    assert np.all(out[len(s):] == 777.0)
    return out[:len(s)]


@pytest.mark.parametrize("name", ["tiny", "sweep_32k", "ragged_b8", "long_128k"])
def test_normalize_scores_matches_oracle(name):
    wl = I.WORKLOADS[name]
    s, mask, cu = I.make_scores(wl), I.make_instr_mask(wl), I.cu_seqlens_of(wl.seq_lens)
    got = _normalize(s, mask, cu)
    ref = O.normalize_scores(s, mask, cu, eps=1e-6)
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)
    assert np.all(got[mask == 1] == 0.0)


def test_normalize_scores_edge_sequences():
    # empty sequence, an all-instruction sequence, one-token sequences, no mask
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(0, 0, 1, 37, 600), instr_lens=(0, 5, 0, 2, 9),
                        instr_where="scattered")
    s, mask, cu = I.make_scores(wl), I.make_instr_mask(wl), I.cu_seqlens_of(wl.seq_lens)
    np.testing.assert_allclose(_normalize(s, mask, cu), O.normalize_scores(s, mask, cu, 1e-6), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(_normalize(s, None, cu, eps=0.0), O.normalize_scores(s, np.zeros_like(mask), cu, 0.0),
                               rtol=1e-5, atol=1e-6)


def _positions(lens, seed):
    rng = np.random.default_rng(seed)
    pos = []
    for n in lens:
        pos.append(np.cumsum(rng.integers(1, 9, n)) - 1)        # strictly increasing, with gaps
    return np.concatenate(pos).astype(np.int32) if pos else np.zeros(0, np.int32)


def _eq8_run(wl, lens, rows=None, with_b=True, seed=0):
    cu = I.cu_seqlens_of(lens)
    M = int(cu[-1])
    at = I.make_attention_inputs(wl, M, tag_extra=seed)
    rng = np.random.default_rng(100 + seed)
    b = rng.standard_normal(M).astype(np.float32)
    pos = _positions(lens, 200 + seed)
    gain = rng.uniform(0.2, 1.5, wl.H_q).astype(np.float32)
    temp = rng.uniform(0.6, 1.4, wl.H_q).astype(np.float32)
    O_d = torch.full((M, wl.H_q, wl.d_h), 0x7FC0, dtype=torch.int16, device="cuda")
    st = status_word()
    tg.gated_attention_eq8(dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(cu), dev(pos), gain, temp, O_d,
                           max_seqlen=max(lens), b=dev(b) if with_b else None, status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    got = bf16_dev_to_f64(O_d)
    ref = O.gated_attention_eq8(I.bf16_bits_to_f64(at["Q"]), I.bf16_bits_to_f64(at["K"]),
                                I.bf16_bits_to_f64(at["V"]), b.astype(np.float64) if with_b else None, pos, cu,
                                gain.astype(np.float64), temp.astype(np.float64), rows=rows)
    return (got if rows is None else got[rows]), ref


def _close(got, ref):
    mx, mr = attention_close(got, ref)
    assert np.all(np.isfinite(got))
    assert mx <= ATTN_MAX_ABS and mr <= ATTN_MEAN_REL, (mx, mr)


def test_eq8_attention_tiny_dh64():
    _close(*_eq8_run(I.WORKLOADS["tiny"], [96, 130], seed=1))


@pytest.mark.parametrize("lens", [[1], [128, 1, 129], [300]])
def test_eq8_attention_varlen_dh128(lens):
    _close(*_eq8_run(I.WORKLOADS["qwen3_1p7b_8k"], lens, seed=len(lens)))


def test_eq8_attention_without_score_bias():
    _close(*_eq8_run(I.WORKLOADS["qwen3_1p7b_8k"], [200, 77], with_b=False, seed=5))


def test_eq8_attention_sweep_k4096_sampled_rows():
    wl = I.WORKLOADS["sweep_32k"]
    M = 4096 + 256
    rows = sampled_rows(I.cu_seqlens_of([M]), list(range(M - 256, M)), 300, seed=9)
    _close(*_eq8_run(wl, [M], rows=rows, seed=6))


def test_paper_form_pipeline_qwen3_8k():
    # score -> normalise -> select (on s; the order is the same for b) -> gather (b, positions)
    # -> Eq. (8) attention, against the oracle run the same way on the same inputs
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    gi = I.make_gate_inputs(wl)
    T, B = wl.T_total, wl.B
    s = torch.zeros(T, dtype=torch.float32, device="cuda")
    g = torch.zeros(T, dtype=torch.float32, device="cuda")
    bn = torch.zeros(T, dtype=torch.float32, device="cuda")
    kept, cu_kept = zeros_i32(T), zeros_i32(B + 1)
    h_kept = torch.zeros((T, wl.d), dtype=torch.int16, device="cuda")
    pos_kept = zeros_i32(T)
    b_kept = torch.zeros(T, dtype=torch.float32, device="cuda")
    st = status_word()
    h_d, cu_d, mask_d = dev(gi["h"]), dev(gi["cu_seqlens"]), dev(gi["instr_mask"])
    tg.gate_score(h_d, dev(gi["W1"]), dev(gi["w2"]), s, g, instr_mask=mask_d, status=st)
    tg.normalize_scores(s, cu_d, bn, instr_mask=mask_d, status=st)
    tg.topk_select(s, cu_d, wl.K, kept, cu_kept, instr_mask=mask_d, status=st)
    tg.gather_kept(h_d, cu_d, kept, cu_kept, h_kept, pos=dev(gi["pos"]), g=bn, pos_kept=pos_kept,
                   g_kept=b_kept, status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    ref = O.gate_prune_layer(I.bf16_bits_to_f64(gi["h"]), gi["pos"], I.bf16_bits_to_f64(gi["W1"]),
                             I.bf16_bits_to_f64(gi["w2"]), gi["instr_mask"], gi["cu_seqlens"], wl.K)
    np.testing.assert_allclose(host(s), ref["s"], rtol=S_RTOL, atol=S_ATOL)
    # selection: bit-exact against the oracle's top-K on the same fp32 score buffer
    want_idx, want_cu = O.topk_select(host(s), gi["instr_mask"], gi["cu_seqlens"], wl.K)
    M = int(want_cu[-1])
    assert host(cu_kept).tolist() == want_cu.tolist() == ref["cu_kept"].tolist()
    kept_np = host(kept)[:M]
    assert kept_np.tolist() == want_idx.tolist()
    ref_b = O.normalize_scores(ref["s"], gi["instr_mask"], gi["cu_seqlens"], 1e-6)
    np.testing.assert_allclose(host(bn), ref_b, rtol=2e-3, atol=2e-3)   # the scores differ by the score tolerance
    at = I.make_attention_inputs(wl, M)
    rng = np.random.default_rng(77)
    gain = rng.uniform(0.5, 1.5, wl.H_q).astype(np.float32)
    temp = rng.uniform(0.8, 1.2, wl.H_q).astype(np.float32)
    O_d = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    tg.gated_attention_eq8(dev(at["Q"]), dev(at["K"]), dev(at["V"]), cu_kept, pos_kept[:M], gain, temp, O_d,
                           max_seqlen=M, b=b_kept[:M], status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    rows = sampled_rows(want_cu, list(range(M - 128, M)), 250, seed=11)
    # the oracle on the same kept rows, with its own normalised scores and the original positions
    want = O.gated_attention_eq8(I.bf16_bits_to_f64(at["Q"]), I.bf16_bits_to_f64(at["K"]),
                                 I.bf16_bits_to_f64(at["V"]), ref_b[kept_np], gi["pos"][kept_np],
                                 want_cu, gain.astype(np.float64), temp.astype(np.float64), rows=rows)
    _close(bf16_dev_to_f64(O_d)[rows], want)
