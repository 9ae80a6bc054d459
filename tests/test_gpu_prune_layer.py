"""GPU end-to-end: the fused prune layer (score -> top-K -> gather) and gated attention on
the kept rows, against the oracle run on the same seeded inputs.

Selection is compared bit for bit where both sides select from the same fp32 score buffer:
the fused layer's kept indices and boundaries must equal the oracle's top-K run on the score
buffer the layer itself wrote (the score buffer is checked against the oracle's own fp64
scores, within the score tolerance, in the same test). Against the oracle's end-to-end path,
whose fp64 scores may order a near-tie at the threshold the other way, the kept sets may
differ only by rows whose oracle scores lie within the score tolerance of the K-th largest
score, and the counts must match exactly. The attention that follows runs on the layer's kept
rows; the oracle gets the same rows with its own gate values."""
import numpy as np
import pytest
import torch

from learned_token_pruning_07_b300 import binding as tg
from learned_token_pruning_07_b300 import inputs as I
from oracle import tokengate_oracle as O
from tests._helpers import (ATTN_MAX_ABS, ATTN_MEAN_REL, G_ATOL, S_ATOL, S_RTOL, attention_close, sampled_rows,
                            bf16_dev_to_f64, dev, host, status_word, zeros_i32)

pytestmark = pytest.mark.gpu


def _prune_gpu(wl, K):
    gi = I.make_gate_inputs(wl)
    T, B = wl.T_total, wl.B
    t = {
        "h": dev(gi["h"]), "cu": dev(gi["cu_seqlens"]), "W1": dev(gi["W1"]), "w2": dev(gi["w2"]),
        "mask": dev(gi["instr_mask"]), "pos": dev(gi["pos"]),
        "s": torch.zeros(T, dtype=torch.float32, device="cuda"),
        "g": torch.zeros(T, dtype=torch.float32, device="cuda"),
        "kept": zeros_i32(T), "cu_kept": zeros_i32(B + 1),
        "h_kept": torch.zeros((T, wl.d), dtype=torch.int16, device="cuda"),
        "pos_kept": zeros_i32(T), "g_kept": torch.zeros(T, dtype=torch.float32, device="cuda"),
        "st": status_word(),
    }
    tg.gate_prune_layer(t["h"], t["cu"], t["W1"], t["w2"], K, t["s"], t["g"], t["kept"], t["cu_kept"],
                        t["h_kept"], pos_kept=t["pos_kept"], g_kept=t["g_kept"], pos=t["pos"],
                        instr_mask=t["mask"], status=t["st"])
    torch.cuda.synchronize()
    assert int(host(t["st"])[0]) == 0
    return gi, {k: host(v) for k, v in t.items()}


def _check_selection_on_own_scores(s_gpu, mask, cu, K, kept, cu_kept, base=0):
    """Bit-exact: the GPU's keep list equals the oracle's top-K on the GPU's fp32 score buffer."""
    want_idx, want_cu = O.topk_select(s_gpu, mask, cu, K)
    assert (np.asarray(cu_kept) - base).tolist() == want_cu.tolist()
    M = int(want_cu[-1])
    assert np.asarray(kept[:M]).tolist() == want_idx.tolist()
    return want_idx, want_cu


def _check_prune(wl, K, score_rows=None):
    gi, out = _prune_gpu(wl, K)
    mask = gi["instr_mask"]
    cu = gi["cu_seqlens"]
    # selection: bit-exact on the layer's own score buffer
    _check_selection_on_own_scores(out["s"], mask, cu, K, out["kept"], out["cu_kept"])
    # scores and gates against the oracle's fp64 scoring (all rows, or a sample at full size)
    h64 = I.bf16_bits_to_f64(gi["h"])
    W1, w2 = I.bf16_bits_to_f64(gi["W1"]), I.bf16_bits_to_f64(gi["w2"])
    rows = np.arange(wl.T_total) if score_rows is None else score_rows
    ref_s, ref_g = O.gate_score(h64[rows], W1, w2, mask[rows])
    np.testing.assert_allclose(out["s"][rows], ref_s, rtol=S_RTOL, atol=S_ATOL)
    np.testing.assert_allclose(out["g"][rows], ref_g, rtol=0, atol=G_ATOL)
    M = int(out["cu_kept"][-1])
    kept = out["kept"][:M]
    ref = None
    if score_rows is None:
        # against the oracle's own end-to-end path: differences only at near-ties at the threshold
        ref = O.gate_prune_layer(h64, gi["pos"], W1, w2, mask, cu, K)
        assert out["cu_kept"].tolist() == ref["cu_kept"].tolist()
        for b in range(wl.B):
            a, e = int(out["cu_kept"][b]), int(out["cu_kept"][b + 1])
            diff = set(kept[a:e].tolist()) ^ set(ref["kept_idx"][a:e].tolist())
            if diff:
                doc = [j for j in range(cu[b], cu[b + 1]) if not mask[j]]
                thr = np.sort(ref["s"][doc])[::-1][min(K, len(doc)) - 1]
                tol = S_ATOL + S_RTOL * abs(thr)
                assert all(abs(ref["s"][j] - thr) <= 2 * tol for j in diff), sorted(diff)
    # gathered rows are the rows of h at the kept indices; positions are the original ids
    assert np.array_equal(out["h_kept"][:M], gi["h"][kept])
    assert np.array_equal(out["pos_kept"][:M], gi["pos"][kept])
    assert np.array_equal(out["g_kept"][:M], out["g"][kept])
    return gi, out, ref


def test_prune_layer_tiny():
    _check_prune(I.WORKLOADS["tiny"], 64)


def test_prune_layer_qwen3_8k_and_attention_on_kept_rows():
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    gi, out, ref = _check_prune(wl, wl.K)
    M = int(out["cu_kept"][-1])
    kept = out["kept"][:M]
    at = I.make_attention_inputs(wl, M)
    cu_k = dev(out["cu_kept"])
    O_d = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    st = status_word()
    Qd, Kd = dev(at["Q"]), dev(at["K"])
    # RoPE on the original position ids of the kept rows, then gated attention with the kept gates
    pos_d = dev(out["pos_kept"][:M])
    tg.apply_rope(Qd, pos_d, wl.rope_theta, cu_kept=cu_k)
    tg.apply_rope(Kd, pos_d, wl.rope_theta, cu_kept=cu_k)
    tg.gated_attention(Qd, Kd, dev(at["V"]), cu_k, at["tau"], at["beta"], O_d, max_seqlen=M,
                       g=dev(out["g_kept"][:M]), status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    # the oracle on the same kept rows: its own gates and the original positions at those rows
    q = O.apply_rope(I.bf16_bits_to_f64(at["Q"]), gi["pos"][kept], wl.rope_theta)
    k = O.apply_rope(I.bf16_bits_to_f64(at["K"]), gi["pos"][kept], wl.rope_theta)
    # the GPU rounds rotated Q/K to bf16 before attention; the oracle keeps them exact
    want = O.gated_attention(q, k, I.bf16_bits_to_f64(at["V"]), ref["g"][kept], out["cu_kept"],
                             at["tau"].astype(np.float64), at["beta"].astype(np.float64))
    mx, mr = attention_close(bf16_dev_to_f64(O_d), want)
    assert mx <= ATTN_MAX_ABS and mr <= ATTN_MEAN_REL, (mx, mr)


@pytest.mark.slow
def test_prune_layer_ragged_b8_full_size():
    # the full ragged batch of eight sequences (4K-16K documents, 64-512 instruction tokens),
    # budget K = 2048 per sequence: one select cluster per sequence, every boundary exact
    wl = I.WORKLOADS["ragged_b8"]
    cu = I.cu_seqlens_of(wl.seq_lens)
    rng = np.random.default_rng(23)
    rows = np.unique(np.concatenate([cu[:-1], cu[1:] - 1, rng.integers(0, wl.T_total, 3000)]))
    gi, out, _ = _check_prune(wl, wl.K, score_rows=rows)
    lens = np.diff(out["cu_kept"])
    assert lens.tolist() == [min(wl.K, a) + b for a, b in zip(wl.doc_lens, wl.instr_lens)]


def test_rope_matches_oracle():
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    M = 700
    at = I.make_attention_inputs(wl, M, tag_extra=3)
    pos = np.sort(np.random.default_rng(2).choice(131072, M, replace=False)).astype(np.int32)
    X = dev(at["Q"])
    tg.apply_rope(X, dev(pos), wl.rope_theta)
    torch.cuda.synchronize()
    got = bf16_dev_to_f64(X)
    want = O.apply_rope(I.bf16_bits_to_f64(at["Q"]), pos, wl.rope_theta)
    # one bf16 rounding of values of magnitude up to ~5: half an ulp is 2^-8 * 4 / 2
    np.testing.assert_allclose(got, want, rtol=0, atol=2e-2)
    assert np.mean(np.abs(got - want)) < 2e-3


# ---------------------------------------------------------------------------
# The packed two-budget forward (deep dive section 3.3, Eq. (9))
# ---------------------------------------------------------------------------

def _two_budget(wl, K_prune):
    gi = I.make_gate_inputs(wl)
    T, B = wl.T_total, wl.B
    t = {"s": torch.zeros(T, dtype=torch.float32, device="cuda"),
         "g": torch.zeros(T, dtype=torch.float32, device="cuda"),
         "kept": torch.full((2 * T,), -7, dtype=torch.int32, device="cuda"),
         "cu": torch.full((2 * B + 1,), -7, dtype=torch.int32, device="cuda"),
         "h_kept": torch.zeros((2 * T, wl.d), dtype=torch.int16, device="cuda"),
         "pos_kept": zeros_i32(2 * T), "g_kept": torch.zeros(2 * T, dtype=torch.float32, device="cuda"),
         "st": status_word()}
    tg.two_budget_prune_layer(dev(gi["h"]), dev(gi["cu_seqlens"]), dev(gi["W1"]), dev(gi["w2"]), K_prune, t["s"],
                              t["g"], t["kept"], t["cu"], t["h_kept"], pos_kept=t["pos_kept"], g_kept=t["g_kept"],
                              pos=dev(gi["pos"]), instr_mask=dev(gi["instr_mask"]), status=t["st"])
    torch.cuda.synchronize()
    assert int(host(t["st"])[0]) == 0
    out = {k: host(v) for k, v in t.items()}
    ref = O.two_budget_prune_layer(I.bf16_bits_to_f64(gi["h"]), gi["pos"], I.bf16_bits_to_f64(gi["W1"]),
                                   I.bf16_bits_to_f64(gi["w2"]), gi["instr_mask"], gi["cu_seqlens"], K_prune)
    np.testing.assert_allclose(out["s"], ref["s"], rtol=S_RTOL, atol=S_ATOL)
    np.testing.assert_allclose(out["g"], ref["g"], rtol=0, atol=G_ATOL)
    assert out["cu"].tolist() == ref["cu_packed"].tolist()
    M = int(ref["cu_packed"][-1])
    assert out["kept"][:T].tolist() == list(range(T))
    assert np.all(out["kept"][M:] == -7)                                  # nothing past the packed list
    # the pruned half: bit-exact against the oracle's top-K on the layer's own score buffer,
    # listed after the T rows of the full half
    want_idx, want_cu = O.topk_select(out["s"], gi["instr_mask"], gi["cu_seqlens"], K_prune)
    assert (out["cu"][B:] - T).tolist() == want_cu.tolist()
    assert out["kept"][T:M].tolist() == want_idx.tolist()
    kept = out["kept"][:M]
    assert np.array_equal(out["h_kept"][:M], gi["h"][kept])
    assert np.array_equal(out["pos_kept"][:M], gi["pos"][kept])
    assert np.array_equal(out["g_kept"][:M], out["g"][kept])
    return gi, out, ref


def test_two_budget_prune_tiny():
    _two_budget(I.WORKLOADS["tiny"], 37)


def test_two_budget_prune_ragged_and_one_attention_call():
    wl = I.with_changes(I.WORKLOADS["qwen3_1p7b_8k"], doc_lens=(700, 0, 1500), instr_lens=(40, 8, 64))
    gi, out, ref = _two_budget(wl, 300)
    cu = out["cu"]
    M = int(cu[-1])
    at = I.make_attention_inputs(wl, M)
    O_d = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    st = status_word()
    lens = np.diff(cu)
    tg.gated_attention(dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(cu), at["tau"], at["beta"], O_d,
                       max_seqlen=int(lens.max()), g=dev(out["g_kept"][:M]), status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    rows = sampled_rows(cu, [], 300, seed=13)
    want = O.gated_attention(I.bf16_bits_to_f64(at["Q"]), I.bf16_bits_to_f64(at["K"]),
                             I.bf16_bits_to_f64(at["V"]), out["g_kept"][:M].astype(np.float64), cu,
                             at["tau"].astype(np.float64), at["beta"].astype(np.float64), rows=rows)
    mx, mr = attention_close(bf16_dev_to_f64(O_d)[rows], want)
    assert mx <= ATTN_MAX_ABS and mr <= ATTN_MEAN_REL, (mx, mr)
