"""The attention entry point for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc for a workspace: the device's memory already belongs to
another allocator (a framework's caching pool, a serving runtime that reserved it up front), or
their hot path must not allocate. tg_gated_attention_noalloc gives them the split attention with
the library's own fixed 16 MiB scratch array in place of a caller workspace. These tests call it
through the C ABI twice in a row and compare each output with the workspace entry point's
(tg_gated_attention_ws) within the attention tolerance. The file is collected last, so a
failure here leaves every other test already run."""
import numpy as np
import pytest
import torch

from learned_token_pruning_07_b300 import binding as tg
from learned_token_pruning_07_b300 import inputs as I
from tests._helpers import ATTN_MAX_ABS, ATTN_MEAN_REL, attention_close, bf16_dev_to_f64, dev, host, status_word

pytestmark = pytest.mark.gpu

FIXED_SCRATCH_BYTES = 16 << 20


def _inputs(wl, M, tag):
    at = I.make_attention_inputs(wl, M, tag_extra=tag)
    return at, {k: dev(at[k]) for k in ("Q", "K", "V", "g")}, dev(I.cu_seqlens_of([M]))


def _noalloc_twice_against_workspace_call(wl, M, tag):
    at, t, cu = _inputs(wl, M, tag)
    ws = tg.attention_workspace(1, M, wl.H_q, wl.H_kv, wl.d_h)
    want = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    st = status_word()
    tg.gated_attention(t["Q"], t["K"], t["V"], cu, at["tau"], at["beta"], want, max_seqlen=M, g=t["g"],
                       status=st, workspace=ws)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    ref = bf16_dev_to_f64(want)
    outs = []
    for _ in range(2):  # two calls in a row: the second starts from the first one's leftover scratch
        got = torch.full((M, wl.H_q, wl.d_h), 0x7FC0, dtype=torch.int16, device="cuda")
        st = status_word()
        tg.gated_attention_noalloc(t["Q"], t["K"], t["V"], cu, at["tau"], at["beta"], got, max_seqlen=M, g=t["g"],
                                   status=st)
        torch.cuda.synchronize()
        assert int(host(st)[0]) == 0
        out = bf16_dev_to_f64(got)
        assert np.all(np.isfinite(out))
        mx, mr = attention_close(out, ref)
        assert mx <= ATTN_MAX_ABS and mr <= ATTN_MEAN_REL, (mx, mr)
        outs.append(out)
    return ws.numel(), outs


def test_noalloc_matches_the_workspace_call_dh128():
    # 8 query / 4 kv heads of 128 over 1,280 kept rows: 10 query tiles x 4 head pairs leave SMs
    # idle, so the key ranges split, and the split's scratch fits the fixed array
    wl = I.with_changes(I.WORKLOADS["qwen3_1p7b_8k"], H_q=8, H_kv=4)
    n, outs = _noalloc_twice_against_workspace_call(wl, 1280, tag=41)
    assert 0 < n <= FIXED_SCRATCH_BYTES


def test_noalloc_matches_the_workspace_call_dh64():
    wl = I.WORKLOADS["tiny"]
    n, outs = _noalloc_twice_against_workspace_call(wl, 1000, tag=42)
    assert 0 < n <= FIXED_SCRATCH_BYTES


def test_noalloc_without_split_needs_no_scratch():
    wl = I.WORKLOADS["sweep_32k"]
    n, outs = _noalloc_twice_against_workspace_call(wl, 4096 + 256, tag=43)
    assert n == 0


def test_noalloc_rejects_a_split_larger_than_the_fixed_array():
    # 16 query / 8 kv heads over 1,280 kept rows: the split needs about 19 MB of scratch
    wl = I.WORKLOADS["sweep_32k"]
    M = 1024 + 256
    assert tg.gated_attention_workspace_size(1, M, wl.H_q, wl.H_kv, wl.d_h) > FIXED_SCRATCH_BYTES
    at, t, cu = _inputs(wl, M, 44)
    out = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    with pytest.raises(tg.TGError) as e:
        tg.gated_attention_noalloc(t["Q"], t["K"], t["V"], cu, at["tau"], at["beta"], out, max_seqlen=M, g=t["g"])
    assert e.value.status == tg.TG_ERR_UNSUPPORTED
