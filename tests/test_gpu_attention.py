"""GPU parity: token-gated causal GQA attention (tcgen05) against the fp64 oracle.

Bar: 2e-2 max-abs and 1e-2 mean-relative error, bf16 output against fp64."""
import numpy as np
import pytest
import torch

from learned_token_pruning_07_b300 import binding as tg
from learned_token_pruning_07_b300 import inputs as I
from oracle import tokengate_oracle as O
from tests._helpers import (ATTN_MAX_ABS, ATTN_MEAN_REL, attention_close, bf16_dev_to_f64, dev, host,
                            sampled_rows, status_word)

pytestmark = pytest.mark.gpu


def _run(wl, lens, tag=0, use_g=True, beta_zero=False, rows=None, capacity=None, g_override=None):
    cu = I.cu_seqlens_of(lens)
    M = int(cu[-1])
    at = I.make_attention_inputs(wl, M, tag_extra=tag)
    g = at["g"] if g_override is None else g_override
    tau, beta = at["tau"], at["beta"]
    if beta_zero:
        beta = np.zeros_like(beta)
    cap = M if capacity is None else capacity
    Qd, Kd, Vd = dev(at["Q"]), dev(at["K"]), dev(at["V"])
    O_d = torch.full((M, wl.H_q, wl.d_h), 0x7FC0, dtype=torch.int16, device="cuda")  # NaN fill
    st = status_word()
    tg.gated_attention(Qd[:cap], Kd[:cap], Vd[:cap], dev(cu), tau, beta, O_d[:cap],
                       max_seqlen=max(lens) if lens else 0, g=dev(g) if use_g else None, status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    got = bf16_dev_to_f64(O_d)
    ref = O.gated_attention(I.bf16_bits_to_f64(at["Q"]), I.bf16_bits_to_f64(at["K"]),
                            I.bf16_bits_to_f64(at["V"]), g.astype(np.float64) if use_g else None,
                            cu, tau.astype(np.float64), beta.astype(np.float64), rows=rows)
    return got if rows is None else got[rows], ref


def _assert_close(got, ref):
    mx, mr = attention_close(got, ref)
    assert np.all(np.isfinite(got))
    assert mx <= ATTN_MAX_ABS and mr <= ATTN_MEAN_REL, (mx, mr)


def test_attention_tiny_dh64():
    wl = I.WORKLOADS["tiny"]
    _assert_close(*_run(wl, [96]))


@pytest.mark.parametrize("lens", [[1], [127], [128], [129], [300, 1, 45, 256], [0, 200, 0]])
def test_attention_varlen_dh128(lens):
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    _assert_close(*_run(wl, lens, tag=len(lens)))


def test_attention_qwen3_8k_full():
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    _assert_close(*_run(wl, [1152]))


def test_attention_beta_zero_and_no_gate_are_plain_causal():
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    a_got, a_ref = _run(wl, [400], beta_zero=True)
    b_got, b_ref = _run(wl, [400], use_g=False)
    _assert_close(a_got, a_ref)
    _assert_close(b_got, b_ref)
    np.testing.assert_allclose(a_ref, b_ref, rtol=0, atol=1e-12)


def test_attention_strong_gates_and_zero_gates():
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    M = 260
    g = np.random.default_rng(3).uniform(1e-6, 1.0, M).astype(np.float32)
    g[::5] = 1e-30
    _assert_close(*_run(wl, [M], g_override=g))
    g0 = np.zeros(M, np.float32)
    got, ref = _run(wl, [M], g_override=g0)          # every key has zero weight -> zeros
    assert np.all(ref == 0.0) and np.all(got == 0.0)


def test_attention_subnormal_gates_keep_their_weight():
    # Gates below the smallest normal fp32 (2^-126 ~ 1.18e-38; a score under about -87.3) are
    # still gates: each key keeps the weight g^beta. With every key subnormal, a kernel that
    # flushed them to zero would output zero rows; the oracle gives proper weighted averages.
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    M = 300
    rng = np.random.default_rng(17)
    g = (rng.uniform(1.0, 50.0, M) * 1e-40).astype(np.float32)
    assert np.all(g < np.finfo(np.float32).tiny) and np.all(g > 0)
    got, ref = _run(wl, [M], g_override=g)
    assert np.all(np.abs(ref).max(axis=(1, 2)) > 0.0)
    _assert_close(got, ref)
    # a mix: subnormal keys beside normal ones, over several key tiles
    M2 = 700
    g2 = rng.uniform(0.05, 1.0, M2).astype(np.float32)
    g2[: M2 // 2] = (rng.uniform(1.0, 50.0, M2 // 2) * 1e-41).astype(np.float32)
    _assert_close(*_run(wl, [M2], g_override=g2, tag=5))


def test_attention_odd_group_one_head_per_cta():
    wl = I.with_changes(I.WORKLOADS["qwen3_1p7b_8k"], H_q=6, H_kv=2)   # group of 3
    _assert_close(*_run(wl, [333]))


def test_attention_mha_group_of_one():
    wl = I.with_changes(I.WORKLOADS["qwen3_1p7b_8k"], H_q=4, H_kv=4)
    _assert_close(*_run(wl, [200, 70]))


def test_attention_at_the_largest_head_count():
    # 128 query heads, the most the call takes, over 64 kv heads of 64
    wl = I.with_changes(I.WORKLOADS["tiny"], H_q=128, H_kv=64)
    _assert_close(*_run(wl, [70, 130]))


def test_attention_sweep_k4096_full():
    wl = I.WORKLOADS["sweep_32k"]
    _assert_close(*_run(wl, [4096 + 256]))


def test_attention_sweep_k16384_sampled_rows():
    wl = I.WORKLOADS["sweep_32k"]
    M = 16384 + 256
    cu = I.cu_seqlens_of([M])
    rows = sampled_rows(cu, list(range(M - 256, M)), 900, seed=5)
    assert len(rows) >= 1024
    _assert_close(*_run(wl, [M], rows=rows))


def test_attention_back_to_back_launches_never_time_out():
    # Many launches queued without a host sync, at a length where every CTA walks up to 260 key
    # tiles: the pipeline barriers must hold their phases whatever the relative speed of the
    # softmax and MMA warps (a phase overrun shows as a timeout in the status word)
    wl = I.WORKLOADS["sweep_32k"]
    M = 16384 + 256
    at = I.make_attention_inputs(wl, M, tag_extra=3)
    Qd, Kd, Vd, gd, cud = dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(at["g"]), dev(I.cu_seqlens_of([M]))
    st = status_word()
    outs = [torch.empty((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda") for _ in range(2)]
    tg.set_wait_limit_ns(200_000_000)
    try:
        for i in range(24):
            tg.gated_attention(Qd, Kd, Vd, cud, at["tau"], at["beta"], outs[i % 2], max_seqlen=M, g=gd, status=st)
        torch.cuda.synchronize()
    finally:
        tg.set_wait_limit_ns(0)
    assert int(host(st)[0]) == 0
    assert torch.equal(outs[0], outs[1])


def test_attention_ragged_batch_sampled_rows():
    wl = I.WORKLOADS["ragged_b8"]
    lens = [min(2048, d) + n for d, n in zip(wl.doc_lens, wl.instr_lens)]
    cu = I.cu_seqlens_of(lens)
    rows = sampled_rows(cu, [], 1000, seed=6)
    assert len(rows) >= 1024
    _assert_close(*_run(wl, lens, rows=rows))


def test_attention_long_context_pruned_sampled_rows():
    # 128K context pruned to K = 8192 document tokens plus 512 instruction tokens
    wl = I.WORKLOADS["long_128k"]
    M = 8192 + 512
    cu = I.cu_seqlens_of([M])
    rows = sampled_rows(cu, list(range(M - 512, M)), 900, seed=7)
    assert len(rows) >= 1024
    _assert_close(*_run(wl, [M], rows=rows))


@pytest.mark.slow
def test_attention_long_context_full_causal_sampled_rows():
    # the layers at or below the gate: plain causal GQA over all 131,584 tokens (no gate,
    # tau = 1, beta = 0), the unpruned side of the long-context comparison
    wl = I.with_changes(I.WORKLOADS["long_128k"], fixed_tau_beta=1.0)
    M = wl.T_total
    cu = I.cu_seqlens_of([M])
    rows = sampled_rows(cu, [], 160, seed=8)
    at = I.make_attention_inputs(wl, M)
    beta = np.zeros(wl.H_q, np.float32)
    O_d = torch.full((M, wl.H_q, wl.d_h), 0x7FC0, dtype=torch.int16, device="cuda")
    st = status_word()
    tg.gated_attention(dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(cu), at["tau"], beta, O_d,
                       max_seqlen=M, g=None, status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    got = I.bf16_bits_to_f64(host(O_d[torch.from_numpy(rows).cuda()]))
    del O_d
    # fp64 query rows only where sampled (np.zeros pages are not touched elsewhere)
    Q64 = np.zeros((M, wl.H_q, wl.d_h))
    Q64[rows] = I.bf16_bits_to_f64(at["Q"][rows])
    ref = O.gated_attention(Q64, I.bf16_bits_to_f64(at["K"]), I.bf16_bits_to_f64(at["V"]), None, cu,
                            at["tau"].astype(np.float64), beta.astype(np.float64), rows=rows)
    _assert_close(got, ref)


# ---------------------------------------------------------------------------
# Split key ranges (tg_gated_attention_ws): short kept sequences, where one CTA per query tile
# would leave SMs idle, against the oracle and against the unsplit kernel
# ---------------------------------------------------------------------------

def _run_ws(wl, lens, tag=0, repeats=2):
    cu = I.cu_seqlens_of(lens)
    M = int(cu[-1])
    at = I.make_attention_inputs(wl, M, tag_extra=tag)
    Qd, Kd, Vd, gd, cud = dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(at["g"]), dev(cu)
    mx = max(lens)
    ws = tg.attention_workspace(len(lens), mx, wl.H_q, wl.H_kv, wl.d_h)
    outs = []
    for _ in range(repeats):
        O_d = torch.full((M, wl.H_q, wl.d_h), 0x7FC0, dtype=torch.int16, device="cuda")
        st = status_word()
        tg.gated_attention(Qd, Kd, Vd, cud, at["tau"], at["beta"], O_d, max_seqlen=mx, g=gd, status=st,
                           workspace=ws)
        torch.cuda.synchronize()
        assert int(host(st)[0]) == 0
        outs.append(host(O_d))
    plain = torch.full((M, wl.H_q, wl.d_h), 0x7FC0, dtype=torch.int16, device="cuda")
    tg.gated_attention(Qd, Kd, Vd, cud, at["tau"], at["beta"], plain, max_seqlen=mx, g=gd)
    torch.cuda.synchronize()
    ref = O.gated_attention(I.bf16_bits_to_f64(at["Q"]), I.bf16_bits_to_f64(at["K"]), I.bf16_bits_to_f64(at["V"]),
                            at["g"].astype(np.float64), cu, at["tau"].astype(np.float64),
                            at["beta"].astype(np.float64))
    return ws, outs, host(plain), ref


@pytest.mark.parametrize("wname,M", [("sweep_32k", 1024 + 256), ("qwen3_1p7b_8k", 1024 + 128)])
def test_split_attention_at_the_small_budgets(wname, M):
    # K = 1024 kept from the 32K sweep (1,280 rows) and from the 8K gate layer (1,152 rows):
    # 10 and 9 query tiles x 8 head pairs leave SMs idle, so the key ranges split
    wl = I.WORKLOADS[wname]
    ws, outs, plain, ref = _run_ws(wl, [M], tag=M)
    assert ws.numel() > 0                                   # this shape splits
    got = I.bf16_bits_to_f64(outs[0])
    _assert_close(got, ref)
    assert np.array_equal(outs[0], outs[1])                 # chunks combine in a fixed order
    # against the unsplit kernel: both within bf16 rounding of the same values
    assert np.max(np.abs(got - I.bf16_bits_to_f64(plain))) <= 2 * ATTN_MAX_ABS
    n_cnt = ws.view(torch.int32)[:64].cpu().numpy()
    assert np.all(n_cnt == 0)                               # arrival counters are left at zero


def test_split_attention_ragged_and_empty_tail_tiles():
    # two sequences of different length: the shorter one has no query tiles past its end
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    ws, outs, plain, ref = _run_ws(wl, [900, 300], tag=21)
    assert ws.numel() > 0
    _assert_close(I.bf16_bits_to_f64(outs[0]), ref)
    assert np.array_equal(outs[0], outs[1])


def test_split_attention_dh64():
    wl = I.WORKLOADS["tiny"]
    ws, outs, plain, ref = _run_ws(wl, [1000], tag=22)
    assert ws.numel() > 0
    _assert_close(I.bf16_bits_to_f64(outs[0]), ref)
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("M", [4096 + 256, 256 + 256])
def test_workspace_call_without_split_is_the_plain_kernel(M):
    # enough query tiles for every SM (K = 4096), or too few key tiles for a split to pay (K = 256):
    # no workspace needed, and the result is bit-identical to the plain call
    wl = I.WORKLOADS["sweep_32k"]
    assert tg.gated_attention_workspace_size(1, M, wl.H_q, wl.H_kv, wl.d_h) == 0
    ws, outs, plain, ref = _run_ws(wl, [M], tag=23, repeats=1)
    assert np.array_equal(outs[0], plain)


def test_split_attention_rejects_a_small_workspace():
    wl = I.WORKLOADS["sweep_32k"]
    M = 1024 + 256
    n = tg.gated_attention_workspace_size(1, M, wl.H_q, wl.H_kv, wl.d_h)
    at = I.make_attention_inputs(wl, M)
    small = torch.zeros(n - 256, dtype=torch.uint8, device="cuda")
    O_d = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    with pytest.raises(tg.TGError) as e:
        tg.gated_attention(dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(I.cu_seqlens_of([M])), at["tau"],
                           at["beta"], O_d, max_seqlen=M, g=dev(at["g"]), workspace=small)
    assert e.value.status == tg.TG_ERR_INVALID_ARG
