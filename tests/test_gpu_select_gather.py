"""GPU parity: top-K selection and the gather of kept rows (bit-exact against the oracle).

Both sides select from the same seeded fp32 score buffer, so kept indices must match
exactly, ties included."""
import numpy as np
import pytest
import torch

from learned_token_pruning_07_b300 import binding as tg
from learned_token_pruning_07_b300 import inputs as I
from oracle import tokengate_oracle as O
from tests._helpers import dev, host, status_word, zeros_i32

pytestmark = pytest.mark.gpu


def _select_gpu(s, mask, cu, K, capacity=None):
    T = s.shape[0]
    B = len(cu) - 1
    cap = T if capacity is None else capacity
    kept = torch.full((cap + 64,), -7, dtype=torch.int32, device="cuda")  # guard band after capacity
    cu_k = zeros_i32(B + 1)
    st = status_word()
    tg.topk_select(dev(s.astype(np.float32)), dev(cu.astype(np.int32)), K, kept[:cap], cu_k,
                   instr_mask=None if mask is None else dev(mask.astype(np.uint8)), status=st)
    torch.cuda.synchronize()
    return host(kept), host(cu_k), int(host(st)[0])


def _check_select(s, mask, cu, K):
    kept, cu_k, st = _select_gpu(s, mask, cu, K)
    ref_idx, ref_cu = O.topk_select(s, np.zeros(len(s), np.uint8) if mask is None else mask, cu, K)
    assert st == 0
    assert cu_k.tolist() == ref_cu.tolist()
    assert kept[:len(ref_idx)].tolist() == ref_idx.tolist()
    assert np.all(kept[len(s):] == -7)          # guard band untouched


@pytest.mark.parametrize("where", ["last", "first", "scattered"])
@pytest.mark.parametrize("K", [0, 1, 7, 64, 479, 480, 1000])
def test_select_tiny(where, K):
    wl = I.with_changes(I.WORKLOADS["tiny"], instr_where=where)
    _check_select(I.make_scores(wl), I.make_instr_mask(wl), I.cu_seqlens_of(wl.seq_lens), K)


@pytest.mark.parametrize("K", [0, 3, 50, 300, 5000])
def test_select_ragged_with_empty_and_tiny_sequences(K):
    wl = I.with_changes(I.WORKLOADS["tiny"], doc_lens=(300, 0, 1, 2000, 0, 77), instr_lens=(5, 0, 0, 40, 3, 1),
                        instr_where="scattered")
    _check_select(I.make_scores(wl), I.make_instr_mask(wl), I.cu_seqlens_of(wl.seq_lens), K)


@pytest.mark.parametrize("levels", [2, 16, 256])
def test_select_ties_quantised(levels):
    wl = I.with_changes(I.WORKLOADS["ragged_b8"], doc_lens=(3000, 1500, 5000), instr_lens=(64, 100, 512),
                        score_levels=levels)
    s = I.make_scores(wl)
    for K in (1, 100, 777, 2048):
        _check_select(s, I.make_instr_mask(wl), I.cu_seqlens_of(wl.seq_lens), K)


def test_select_special_values_and_no_mask():
    s = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1.0, -0.0, np.nan, 0.0, -1.0] * 30, np.float32)
    cu = np.array([0, 100, 300], np.int32)
    for K in range(0, 12):
        _check_select(s, None, cu, K)
    mask = (np.arange(300) % 7 == 0).astype(np.uint8)
    for K in (0, 5, 50, 300):
        _check_select(s, mask, cu, K)


def test_select_all_equal_scores():
    s = np.full(4096, 0.5, np.float32)
    cu = np.array([0, 4096], np.int32)
    mask = np.zeros(4096, np.uint8)
    mask[-100:] = 1
    for K in (1, 1000, 3996):
        _check_select(s, mask, cu, K)


@pytest.mark.parametrize("name", ["sweep_32k", "ragged_b8", "long_128k"])
def test_select_full_size(name):
    wl = I.WORKLOADS[name]
    s = I.make_scores(wl)
    mask = I.make_instr_mask(wl)
    cu = I.cu_seqlens_of(wl.seq_lens)
    for K in wl.budgets_or_k():
        _check_select(s, mask, cu, K)


@pytest.mark.parametrize("doc_lens,instr_lens", [((60000, 150), (300, 50)), ((60000,), (300,))])
def test_select_long_sequences_with_ties(doc_lens, instr_lens):
    # a 60K sequence (7,500 keys per CTA of its cluster), alone and next to a short one;
    # quantised scores keep ties at the threshold, and K = 40000 keeps most of the long one
    wl = I.with_changes(I.WORKLOADS["ragged_b8"], doc_lens=doc_lens, instr_lens=instr_lens, score_levels=256)
    s = I.make_scores(wl)
    for K in (1, 777, 40000):
        _check_select(s, I.make_instr_mask(wl), I.cu_seqlens_of(wl.seq_lens), K)


def test_select_capacity_overflow_is_reported_and_bounded():
    wl = I.WORKLOADS["tiny"]
    s = I.make_scores(wl)
    mask = I.make_instr_mask(wl)
    cu = I.cu_seqlens_of(wl.seq_lens)
    kept, cu_k, st = _select_gpu(s, mask, cu, 64, capacity=50)
    ref_idx, ref_cu = O.topk_select(s, mask, cu, 64)
    assert st & tg.TG_DEV_CAPACITY
    assert cu_k.tolist() == ref_cu.tolist()             # untruncated counts
    assert kept[:50].tolist() == ref_idx[:50].tolist()  # prefix written in order
    assert np.all(kept[50:] == -7)                      # nothing past capacity


def test_select_bad_seqlens_reported():
    s = np.zeros(100, np.float32)
    cu = np.array([0, 60, 50, 100], np.int32)  # decreasing
    _, _, st = _select_gpu(s, None, cu, 5)
    assert st & tg.TG_DEV_BAD_SEQLENS


# ---------------------------------------------------------------------------
# gather
# ---------------------------------------------------------------------------

def _gather_case(wl, K, with_pos, with_g):
    gi = I.make_gate_inputs(wl)
    cu = gi["cu_seqlens"]
    s = I.make_scores(wl)
    ref_idx, ref_cu = O.topk_select(s, gi["instr_mask"], cu, K)
    T = wl.T_total
    M = len(ref_idx)
    g = np.random.default_rng(9).random(T).astype(np.float32)
    h_d = dev(gi["h"])
    h_kept = torch.zeros((T, wl.d), dtype=torch.int16, device="cuda")
    pos_kept = zeros_i32(T)
    g_kept = torch.zeros(T, dtype=torch.float32, device="cuda")
    st = status_word()
    tg.gather_kept(h_d, dev(cu), dev(ref_idx), dev(ref_cu), h_kept,
                   pos=dev(gi["pos"]) if with_pos else None, g=dev(g) if with_g else None,
                   pos_kept=pos_kept, g_kept=g_kept, status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    hk, pk, gk = O.gather_kept(gi["h"], gi["pos"] if with_pos else None, g, ref_idx, cu)
    assert np.array_equal(host(h_kept)[:M], hk)
    assert np.array_equal(host(pos_kept)[:M], pk)
    if with_g:
        assert np.array_equal(host(g_kept)[:M], gk)
    assert np.all(host(h_kept)[M:] == 0)


@pytest.mark.parametrize("with_pos,with_g", [(True, True), (False, True), (False, False)])
def test_gather_tiny(with_pos, with_g):
    _gather_case(I.WORKLOADS["tiny"], 64, with_pos, with_g)


def test_gather_ragged_d2048():
    wl = I.with_changes(I.WORKLOADS["ragged_b8"], doc_lens=(1000, 0, 333), instr_lens=(64, 5, 70))
    _gather_case(wl, 200, False, True)


def test_gather_full_size_sweep():
    wl = I.WORKLOADS["sweep_32k"]
    _gather_case(wl, 16384, True, True)


def test_gather_bad_index_reported():
    h = torch.zeros((10, 16), dtype=torch.int16, device="cuda")
    kept = dev(np.array([0, 3, 99], np.int32))
    cu_k = dev(np.array([0, 3], np.int32))
    out = torch.zeros((3, 16), dtype=torch.int16, device="cuda")
    st = status_word()
    tg.gather_kept(h, dev(np.array([0, 10], np.int32)), kept, cu_k, out, status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) & tg.TG_DEV_BAD_INDEX
