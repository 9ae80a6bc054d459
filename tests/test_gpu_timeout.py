"""GPU: a pipeline wait that runs out is reported through the status word, and the CUDA
context stays usable.

The test hook tg_set_test_withhold makes a kernel's copy producer issue no loads, so its
consumers wait on barriers that nothing completes. Every such wait is bounded: with the
wait limit set to 20 ms the kernel gives up, sets TG_DEV_TIMEOUT, frees its tensor memory and
returns. The next call, with the hook cleared, must produce correct results. Nothing here
faults, traps or hangs the GPU.
"""
import numpy as np
import pytest
import torch

from learned_token_pruning_07_b300 import binding as tg
from learned_token_pruning_07_b300 import inputs as I
from oracle import tokengate_oracle as O
from tests._helpers import (ATTN_MAX_ABS, ATTN_MEAN_REL, G_ATOL, attention_close, bf16_dev_to_f64,
                            dev, host, status_word)

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000


@pytest.fixture
def withheld():
    def arm(mask):
        tg.set_wait_limit_ns(LIMIT_NS)
        tg.set_test_withhold(mask)
    yield arm
    tg.set_test_withhold(0)
    tg.set_wait_limit_ns(0)


def _score(wl):
    gi = I.make_gate_inputs(wl)
    s = torch.zeros(wl.T_total, dtype=torch.float32, device="cuda")
    g = torch.zeros(wl.T_total, dtype=torch.float32, device="cuda")
    st = status_word()
    tg.gate_score(dev(gi["h"]), dev(gi["W1"]), dev(gi["w2"]), s, g, instr_mask=dev(gi["instr_mask"]),
                  status=st)
    return gi, g, st


def test_gate_score_wait_runs_out_then_recovers(withheld):
    wl = I.WORKLOADS["tiny"]
    withheld(tg.TG_WITHHOLD_GATE_SCORE)
    _, _, st = _score(wl)
    raw = tg.read_device_status(st)
    assert raw & tg.TG_DEV_TIMEOUT
    assert tg.load().tg_read_device_status(st.data_ptr(), None, None) == tg.TG_ERR_INVALID_ARG
    tg.set_test_withhold(0)
    tg.set_wait_limit_ns(0)
    gi, g, st = _score(wl)
    assert tg.read_device_status(st) == 0
    _, ref_g = O.gate_score(I.bf16_bits_to_f64(gi["h"]), I.bf16_bits_to_f64(gi["W1"]),
                            I.bf16_bits_to_f64(gi["w2"]), gi["instr_mask"])
    np.testing.assert_allclose(host(g), ref_g, rtol=0, atol=G_ATOL)


@pytest.mark.parametrize("name", ["tiny", "qwen3_1p7b_8k"])
def test_gate_score_one_cta_of_each_pair_withholds(withheld, name):
    # Only the CTAs of odd cluster rank issue no loads: every stage of the leader's barrier
    # misses one half, the MMAs never start, and the abort raised by the CTA that gives up first
    # reaches every CTA of the cluster (pairs at the tiny size, clusters of four at 8K). The
    # drain is bounded in total, and the next call is correct.
    wl = I.WORKLOADS[name]
    withheld(tg.TG_WITHHOLD_GATE_SCORE_PEER)
    _, _, st = _score(wl)
    assert tg.read_device_status(st) & tg.TG_DEV_TIMEOUT
    tg.set_test_withhold(0)
    tg.set_wait_limit_ns(0)
    gi, g, st = _score(wl)
    assert tg.read_device_status(st) == 0
    _, ref_g = O.gate_score(I.bf16_bits_to_f64(gi["h"]), I.bf16_bits_to_f64(gi["W1"]),
                            I.bf16_bits_to_f64(gi["w2"]), gi["instr_mask"])
    np.testing.assert_allclose(host(g), ref_g, rtol=0, atol=G_ATOL)


def _attention(wl, M):
    at = I.make_attention_inputs(wl, M)
    cu = I.cu_seqlens_of([M])
    O_d = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    st = status_word()
    tg.gated_attention(dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(cu), at["tau"], at["beta"], O_d,
                       max_seqlen=M, g=dev(at["g"]), status=st)
    return at, cu, O_d, st


def test_attention_wait_runs_out_then_recovers(withheld):
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    M = 300
    withheld(tg.TG_WITHHOLD_ATTENTION)
    _, _, _, st = _attention(wl, M)
    assert tg.read_device_status(st) & tg.TG_DEV_TIMEOUT
    tg.set_test_withhold(0)
    tg.set_wait_limit_ns(0)
    at, cu, O_d, st = _attention(wl, M)
    assert tg.read_device_status(st) == 0
    want = O.gated_attention(I.bf16_bits_to_f64(at["Q"]), I.bf16_bits_to_f64(at["K"]),
                             I.bf16_bits_to_f64(at["V"]), at["g"].astype(np.float64), cu,
                             at["tau"].astype(np.float64), at["beta"].astype(np.float64))
    mx, mr = attention_close(bf16_dev_to_f64(O_d), want)
    assert mx <= ATTN_MAX_ABS and mr <= ATTN_MEAN_REL, (mx, mr)


def test_timeout_is_translated_by_read_device_status(withheld):
    withheld(tg.TG_WITHHOLD_GATE_SCORE)
    _, _, st = _score(I.WORKLOADS["tiny"])
    out = np.zeros(1, dtype=np.int32)
    code = tg.load().tg_read_device_status(st.data_ptr(), out.ctypes.data,
                                          torch.cuda.current_stream().cuda_stream)
    assert code == tg.TG_ERR_DEVICE_TIMEOUT and out[0] & tg.TG_DEV_TIMEOUT


def test_backward_wait_runs_out_then_recovers(withheld):
    # the dK/dV and dQ passes: their TMA warps issue nothing, so the MMA warp, the column
    # producer and the eight elementwise warps (which agree through barrier.red before leaving)
    # all give up after the limit; the next call, with the hook cleared, matches the oracle
    from tests.test_gpu_backward import _case
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    lens = [300, 129]
    cu = I.cu_seqlens_of(lens)
    M = int(cu[-1])
    at = I.make_attention_inputs(wl, M)
    Qd, Kd, Vd, gd, cud = dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(at["g"]), dev(cu)
    O_d = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    lse = torch.zeros((M, wl.H_q), dtype=torch.float32, device="cuda")
    st = status_word()
    withheld(tg.TG_WITHHOLD_BACKWARD)
    tg.gated_attention_lse(Qd, Kd, Vd, cud, at["tau"], at["beta"], O_d, lse, max_seqlen=max(lens), g=gd, status=st)
    assert tg.read_device_status(st) == 0  # the forward is not withheld
    f = lambda *shape: torch.zeros(shape, dtype=torch.float32, device="cuda")
    tg.gated_attention_bwd(Qd, Kd, Vd, O_d, O_d, lse, cud, at["tau"], at["beta"], f(M, wl.H_q, wl.d_h),
                           f(M, wl.H_kv, wl.d_h), f(M, wl.H_kv, wl.d_h), f(M, wl.H_q), max_seqlen=max(lens), g=gd,
                           status=st)
    assert tg.read_device_status(st) & tg.TG_DEV_TIMEOUT
    tg.set_test_withhold(0)
    tg.set_wait_limit_ns(0)
    _case(wl, lens, seed=5)
