"""The C-ABI library: it loads without a GPU, exports every entry point the header declares,
and rejects bad host arguments before launching anything."""
import ctypes
import os
import re

import numpy as np
import pytest

from learned_token_pruning_07_b300 import binding, build

pytestmark = pytest.mark.cpu
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tokengate.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(tg_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(binding.SIGNATURES)


def test_version_and_status_strings(lib):
    assert lib.tg_version() == 200
    assert lib.tg_status_string(binding.TG_OK) == b"ok"
    assert b"capacity" in lib.tg_status_string(binding.TG_ERR_CAPACITY)


FAKE = 0x1000  # never dereferenced: every call below fails validation first


def test_gate_score_rejects_bad_arguments(lib):
    f = lib.tg_gate_score
    assert f(None, 8, 256, None, FAKE, None, FAKE, 0.0, 64, FAKE, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(FAKE, -1, 256, None, FAKE, None, FAKE, 0.0, 64, FAKE, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(FAKE, 8, 250, None, FAKE, None, FAKE, 0.0, 64, FAKE, None, None, None) == binding.TG_ERR_UNSUPPORTED
    assert f(FAKE, 8, 256, None, FAKE, None, FAKE, 0.0, 1024, FAKE, None, None, None) == binding.TG_ERR_UNSUPPORTED
    assert f(FAKE + 2, 8, 256, None, FAKE, None, FAKE, 0.0, 64, FAKE, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(FAKE, 8, 256, None, FAKE, None, FAKE, float("nan"), 64, FAKE, None, None, None) == binding.TG_ERR_INVALID_ARG


def test_select_rejects_bad_arguments(lib):
    f = lib.tg_topk_select
    assert f(FAKE, None, FAKE, 1, 10, -1, FAKE, 10, FAKE, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(FAKE, None, FAKE, 0, 10, 3, FAKE, 10, FAKE, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(FAKE, None, FAKE, 1, 10, 3, None, 10, FAKE, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(FAKE, None, FAKE, 5000, 10, 3, FAKE, 10, FAKE, None, None) == binding.TG_ERR_UNSUPPORTED


def test_gather_rejects_bad_arguments(lib):
    f = lib.tg_gather_kept
    assert f(FAKE, None, None, 1, FAKE, 1, 10, 12, FAKE, FAKE, 10, FAKE, None, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(FAKE, None, None, 1, FAKE, 1, 10, 16, None, FAKE, 10, FAKE, None, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(FAKE, None, None, 0, FAKE, 1, 10, 16, FAKE, FAKE, 10, FAKE, None, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(FAKE, None, None, 17, FAKE, 1, 10, 16, FAKE, FAKE, 10, FAKE, None, None, None, None) == binding.TG_ERR_UNSUPPORTED


def test_attention_rejects_bad_arguments(lib):
    f = lib.tg_gated_attention
    tau = np.ones(4, np.float32)
    beta = np.ones(4, np.float32)
    bad_tau = np.array([1, 0, 1, 1], np.float32)
    neg_beta = np.array([1, -1, 1, 1], np.float32)
    args = lambda t, b, hq=4, hkv=2, dh=64, hg=1: (FAKE, FAKE, FAKE, None, hg, FAKE, 1, 64, 64, hq, hkv, dh,
                                                   t.ctypes.data, b.ctypes.data, FAKE, None, None)
    assert f(*args(bad_tau, beta)) == binding.TG_ERR_INVALID_ARG
    assert f(*args(tau, neg_beta)) == binding.TG_ERR_INVALID_ARG
    assert f(*args(tau, beta, hq=4, hkv=3)) == binding.TG_ERR_UNSUPPORTED
    assert f(*args(tau, beta, dh=96)) == binding.TG_ERR_UNSUPPORTED
    assert f(*args(tau, beta, hg=0)) == binding.TG_ERR_INVALID_ARG       # gate heads >= 1
    assert f(*args(tau, beta, hg=3)) == binding.TG_ERR_UNSUPPORTED       # H_q % H_g != 0


def test_rope_rejects_bad_arguments(lib):
    f = lib.tg_apply_rope
    assert f(FAKE, FAKE, None, 0, 10, 2, 63, 1e6, None) == binding.TG_ERR_INVALID_ARG
    assert f(FAKE, FAKE, None, 0, 10, 2, 64, -1.0, None) == binding.TG_ERR_INVALID_ARG
    assert f(FAKE, FAKE, None, 0, 10, 2, 512, 1e6, None) == binding.TG_ERR_UNSUPPORTED


def test_wait_limit_setter(lib):
    assert lib.tg_set_wait_limit_ns(1000) == binding.TG_OK
    assert lib.tg_set_wait_limit_ns(0) == binding.TG_OK


def test_test_withhold_hook_validates_its_mask(lib):
    all_bits = (binding.TG_WITHHOLD_GATE_SCORE | binding.TG_WITHHOLD_ATTENTION | binding.TG_WITHHOLD_BACKWARD
                | binding.TG_WITHHOLD_GATE_SCORE_PEER)
    assert all_bits == 15
    assert lib.tg_set_test_withhold(all_bits) == binding.TG_OK
    assert lib.tg_set_test_withhold(16) == binding.TG_ERR_INVALID_ARG
    assert lib.tg_set_test_withhold(0) == binding.TG_OK


def test_normalize_scores_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(16)
    f = lib.tg_normalize_scores
    assert f(None, 1, None, p, 1, 8, 1e-6, p, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(p, 1, None, p, 0, 8, 1e-6, p, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(p, 1, None, p, 1, 8, -1.0, p, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(p, 1, None, p, 1, 8, float("nan"), p, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(p, 1, None, p, 2000, 8, 1e-6, p, None, None, None) == binding.TG_ERR_UNSUPPORTED
    assert f(p, 0, None, p, 1, 8, 1e-6, p, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert f(p, 32, None, p, 1, 8, 1e-6, p, None, None, None) == binding.TG_ERR_UNSUPPORTED


def test_eq8_attention_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    ones = np.ones(16, np.float32)
    neg = ones.copy()
    neg[3] = -0.5
    f = lambda a: a.ctypes.data
    call = lambda pos, gain, temp, hq=16, hkv=8, dh=128, hg=1: lib.tg_gated_attention_eq8(
        p, p, p, None, hg, pos, p, 1, 100, 100, hq, hkv, dh, gain, temp, p, None, None)
    assert call(None, f(ones), f(ones)) == binding.TG_ERR_INVALID_ARG          # positions required
    assert call(p, f(neg), f(ones)) == binding.TG_ERR_INVALID_ARG              # gain >= 0
    assert call(p, f(ones), f(neg)) == binding.TG_ERR_INVALID_ARG              # temperature >= 0
    assert call(p, f(ones), f(ones), dh=96) == binding.TG_ERR_UNSUPPORTED
    assert call(p, f(ones), f(ones), hq=12, hkv=8) == binding.TG_ERR_UNSUPPORTED
    assert call(p, f(ones), f(ones), hg=3) == binding.TG_ERR_UNSUPPORTED


def test_rmsnorm_entry_points_reject_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    assert lib.tg_gate_score_rmsnorm(p, 10, 64, None, p, None, p, 0.0, 32, -1.0, p, None, None, None) == binding.TG_ERR_INVALID_ARG
    assert lib.tg_gate_score_rmsnorm(p, 10, 64, None, p, None, p, 0.0, 33, 1e-6, p, None, None, None) == binding.TG_ERR_UNSUPPORTED
    assert lib.tg_fold_rmsnorm_weight(None, p, 4, 4, p, None) == binding.TG_ERR_INVALID_ARG
    assert lib.tg_fold_rmsnorm_weight(p, p, 0, 4, p, None) == binding.TG_ERR_INVALID_ARG


def test_gate_score_heads_entry_points_reject_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    b2 = np.zeros(4, np.float32)
    bad_b2 = b2.copy()
    bad_b2[2] = np.inf
    f = lib.tg_gate_score_heads
    call = lambda hg=4, rms=0, eps=1e-6, s_sel=p, b=b2: f(p, 128, 256, None, p, None, p, b.ctypes.data, 64, hg,
                                                          rms, eps, p, None, s_sel, None, None)
    assert call(hg=0) == binding.TG_ERR_INVALID_ARG
    assert call(hg=17) == binding.TG_ERR_UNSUPPORTED
    assert call(s_sel=None) == binding.TG_ERR_INVALID_ARG            # the head mean is required
    assert call(rms=2) == binding.TG_ERR_INVALID_ARG
    assert call(rms=1, eps=-1.0) == binding.TG_ERR_INVALID_ARG
    assert call(b=bad_b2) == binding.TG_ERR_INVALID_ARG
    g = lib.tg_gate_prune_layer_heads
    assert g(p, None, None, p, 1, 128, 256, p, None, p, None, 64, 4, 8, p, None, p, p, 128, p, p, None, None,
             None, None) == binding.TG_ERR_INVALID_ARG               # g_heads required
    assert g(p, None, None, p, 1, 128, 256, p, None, p, None, 64, 4, -1, p, p, p, p, 128, p, p, None, None,
             None, None) == binding.TG_ERR_INVALID_ARG               # K >= 0
    s = lib.tg_gate_score_grad
    beta = np.ones(4, np.float32)
    assert s(p, beta.ctypes.data, p, 3, p, p, 1, 8, 4, 16, p, None) == binding.TG_ERR_UNSUPPORTED


def test_backward_entry_points_reject_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    tau = np.ones(4, np.float32)
    beta = np.ones(4, np.float32)
    # tg_gated_attention_lse: the log-sum-exp output is required
    lse = lambda out: lib.tg_gated_attention_lse(p, p, p, None, 1, p, 1, 64, 64, 4, 2, 64, tau.ctypes.data,
                                                 beta.ctypes.data, p, out, None, None)
    assert lse(None) == binding.TG_ERR_INVALID_ARG
    # tg_gated_attention_bwd: dO, lse and every gradient buffer are required; shapes as the forward
    bwd = lambda dO=p, lse_=p, dq=p, dbias=p, dh=64, hg=1: lib.tg_gated_attention_bwd(
        p, p, p, None, hg, p, dO, lse_, p, 1, 64, 64, 4, 2, dh, tau.ctypes.data, beta.ctypes.data,
        dq, p, p, dbias, None, None)
    assert bwd(dO=None) == binding.TG_ERR_INVALID_ARG
    assert bwd(lse_=None) == binding.TG_ERR_INVALID_ARG
    assert bwd(dq=None) == binding.TG_ERR_INVALID_ARG
    assert bwd(dbias=None) == binding.TG_ERR_INVALID_ARG
    assert bwd(dh=96) == binding.TG_ERR_UNSUPPORTED
    assert bwd(hg=3) == binding.TG_ERR_UNSUPPORTED


def test_prune_layer_entry_points_reject_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    layer = lambda g_out=p, K=8, d=256, d_g=64, b2=0.0: lib.tg_gate_prune_layer(
        p, None, None, p, 1, 128, d, p, None, p, b2, d_g, K, p, g_out, p, 128, p, p, None, None, None, None)
    assert layer(g_out=None) == binding.TG_ERR_INVALID_ARG        # the gate buffer is required here
    assert layer(K=-1) == binding.TG_ERR_INVALID_ARG
    assert layer(b2=float("inf")) == binding.TG_ERR_INVALID_ARG
    assert layer(d=100) == binding.TG_ERR_UNSUPPORTED             # d % 32 != 0
    assert layer(d_g=1024) == binding.TG_ERR_UNSUPPORTED          # d_g > 512
    two = lambda capacity: lib.tg_two_budget_prune_layer(
        p, None, None, p, 1, 128, 256, p, None, p, 0.0, 64, 8, p, p, p, capacity, p, p, None, None, None, None)
    assert two(127) == binding.TG_ERR_INVALID_ARG                 # the full half alone is T_total rows
    assert lib.tg_read_device_status(None, None, None) == binding.TG_ERR_INVALID_ARG


def test_binding_passes_only_dense_cuda_tensors():
    import torch

    class _Strided:  # stands in for a CUDA view with gaps between its elements
        is_cuda = True
        shape = (4, 2)

        def is_contiguous(self):
            return False

        def stride(self):
            return (4, 1)

    assert binding._ptr(None) is None
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding._ptr(torch.zeros(4))                   # host memory is never handed to a kernel
    with pytest.raises(ValueError, match="contiguous"):
        binding._ptr(_Strided())
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.gate_score(torch.zeros(8, 256, dtype=torch.int16), torch.zeros(64, 256, dtype=torch.int16),
                           torch.zeros(64, dtype=torch.int16), torch.zeros(8))


def _declared_params():
    """name -> [parameter C type] for every TG_API declaration in the header."""
    text = re.sub(r"/\*.*?\*/", " ", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"TG_API\s+[\w\s\*]+?\b(tg_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(2).split(",")]
        if params == ["void"]:
            params = []
        # drop the parameter name: the type is everything before the last identifier
        out[m.group(1)] = [re.sub(r"\s*\b\w+\s*$", "", p).replace(" ", "") for p in params]
    return out


def _ctype_of(c_type):
    if c_type.endswith("*") or c_type == "tg_stream_t":
        return ctypes.c_void_p
    return {"int32_t": ctypes.c_int32, "tg_status": ctypes.c_int32, "float": ctypes.c_float,
            "uint64_t": ctypes.c_uint64, "size_t": ctypes.c_size_t}[c_type]


def test_binding_argument_types_match_the_header():
    # a parameter added, dropped or retyped on one side only would pass the wrong bytes
    decls = _declared_params()
    assert set(decls) == set(binding.SIGNATURES)
    for name, c_params in decls.items():
        _, argtypes = binding.SIGNATURES[name]
        assert [_ctype_of(t) for t in c_params] == list(argtypes), name


def test_attention_workspace_size_by_hand(lib):
    # Without a device the library plans for 148 SMs. Kept length 1,280 (the 32K sweep at K = 1024),
    # 16 query / 8 kv heads of 128: 10 query tiles x 8 head pairs = 80 CTAs, fewer than 148, so the
    # key ranges split. Chunks of c key tiles give sum_t ceil((t+1)/c) CTAs per head pair; at most
    # 3 chunks per tile means c >= 4, and c = 4 gives 18 x 8 = 144 <= 148 CTAs.
    # Bytes: 10 x 8 int32 counters rounded up to 256, then 8 x 18 slots of
    # (2 x 128 x 128 + 2 x 128 x 2) fp32.
    f = lib.tg_gated_attention_workspace_size
    slot = (2 * 128 * 128 + 2 * 128 * 2) * 4
    if os.environ.get("CUDA_VISIBLE_DEVICES", "") == "" and not _has_gpu():
        assert f(1, 1280, 16, 8, 128) == 512 + 8 * 18 * slot
    # K = 256: 4 query tiles. The heaviest tile walks only 4 key tiles, fewer than the 6 for which
    # a split pays for its combine, so no split and no workspace.
    assert f(1, 512, 16, 8, 128) == 0
    # 34 query tiles x 8 pairs = 272 CTAs already fill the machine: no split, no workspace
    assert f(1, 4352, 16, 8, 128) == 0
    assert f(1, 100, 16, 8, 128) == 0          # one query tile: nothing to split
    assert f(1, 1280, 16, 6, 128) == 0         # 16 % 6 != 0: invalid shape
    assert f(0, 1280, 16, 8, 128) == 0


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False
