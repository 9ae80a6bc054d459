"""The seeded generators: deterministic bytes, bf16 rounding that matches torch, shapes."""
import numpy as np
import pytest
import torch

from learned_token_pruning_07_b300 import inputs as I

pytestmark = pytest.mark.cpu


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 37.0
    x[:4] = [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]      # exact ties round to even
    ours = I.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = I.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_bf16_rounding_of_special_values():
    special = np.array([np.inf, -np.inf, 3.4e38, -3.4e38, 1e-40, -1e-45], np.float32)
    ours = I.f32_to_bf16_bits(special)
    ref = torch.from_numpy(special).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)                  # infinities, overflow to inf, subnormals
    # NaNs stay NaN with their sign, including the signalling ones whose payload sits in the
    # low 16 bits (adding the rounding bias to those would carry into the infinity pattern)
    nans = np.array([0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001, 0x7FBFFFFF], np.uint32).view(np.float32)
    out = I.f32_to_bf16_bits(nans)
    assert np.all(np.isnan(I.bf16_bits_to_f32(out)))
    assert [int(v) >> 15 for v in out] == [0, 1, 0, 1, 0]


def test_generators_are_deterministic_and_shaped():
    wl = I.WORKLOADS["tiny"]
    a, b = I.make_gate_inputs(wl), I.make_gate_inputs(wl)
    for k in ("h", "W1", "w2", "instr_mask", "cu_seqlens", "pos"):
        assert np.array_equal(a[k], b[k])
    assert a["h"].shape == (512, 256) and a["W1"].shape == (64, 256) and a["w2"].shape == (64,)
    assert a["instr_mask"][-32:].all() and not a["instr_mask"][:480].any()
    at = I.make_attention_inputs(wl, 96)
    assert at["Q"].shape == (96, 4, 64) and at["K"].shape == (96, 2, 64) and at["g"].shape == (96,)
    assert np.all(at["g"] > 0) and np.all(at["g"] <= 1)


def test_workload_table_matches_the_named_shapes():
    w = I.WORKLOADS
    assert w["qwen3_1p7b_8k"].T_total == 8320
    assert w["sweep_32k"].T_total == 33024 and w["sweep_32k"].budgets == (256, 1024, 4096, 16384)
    assert w["long_128k"].T_total == 131584
    r = w["ragged_b8"]
    assert r.B == 8 and all(4096 <= x <= 16384 for x in r.doc_lens)
    assert all(64 <= x <= 512 for x in r.instr_lens)


def test_heavy_rows_and_quantised_scores():
    wl = I.with_changes(I.WORKLOADS["tiny"], heavy_frac=0.02)
    h = I.bf16_bits_to_f32(I.make_gate_inputs(wl)["h"])
    norms = np.linalg.norm(h, axis=1)
    assert np.sum(norms > 2.5 * np.median(norms)) == round(0.02 * wl.T_total)
    wq = I.with_changes(I.WORKLOADS["ragged_b8"], doc_lens=(3000, 2000), instr_lens=(100, 64))
    s = I.make_scores(wq)
    mask = I.make_instr_mask(wq)
    cu = I.cu_seqlens_of(wq.seq_lens)
    for b in range(2):
        seg = s[cu[b]:cu[b + 1]][mask[cu[b]:cu[b + 1]] == 0]
        assert len(np.unique(seg)) <= 256
