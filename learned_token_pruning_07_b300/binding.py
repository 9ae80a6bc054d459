"""ctypes binding of libtokengate (include/tokengate.h): argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module turns torch
tensors into raw pointers and sizes, calls the C entry point of the same name and
raises on a non-OK status. There is no fallback: if the library is missing or a call
fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtokengate.so")

TG_OK, TG_ERR_INVALID_ARG, TG_ERR_UNSUPPORTED, TG_ERR_CUDA = 0, 1, 2, 3
TG_ERR_CAPACITY, TG_ERR_DEVICE_TIMEOUT, TG_ERR_DEVICE = 4, 5, 6
TG_DEV_BAD_SEQLENS, TG_DEV_BAD_INDEX, TG_DEV_CAPACITY, TG_DEV_TIMEOUT = 1, 2, 4, 8

_P = ctypes.c_void_p
_I = ctypes.c_int32
_F = ctypes.c_float

# name -> (restype, argtypes); mirrors include/tokengate.h
SIGNATURES = {
    "tg_version": (_I, []),
    "tg_status_string": (ctypes.c_char_p, [_I]),
    "tg_last_cuda_error": (_I, []),
    "tg_gate_score": (_I, [_P, _I, _I, _P, _P, _P, _P, _F, _I, _P, _P, _P, _P]),
    "tg_gate_score_rmsnorm": (_I, [_P, _I, _I, _P, _P, _P, _P, _F, _I, _F, _P, _P, _P, _P]),
    "tg_fold_rmsnorm_weight": (_I, [_P, _P, _I, _I, _P, _P]),
    "tg_topk_select": (_I, [_P, _P, _P, _I, _I, _I, _P, _I, _P, _P, _P]),
    "tg_gate_score_heads": (_I, [_P, _I, _I, _P, _P, _P, _P, _P, _I, _I, _I, _F, _P, _P, _P, _P, _P]),
    "tg_gather_kept": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P]),
    "tg_gated_attention": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "tg_gated_attention_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    "tg_gated_attention_ws": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, ctypes.c_size_t,
                                   _P, _P]),
    "tg_gated_attention_noalloc": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "tg_gated_attention_lse": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "tg_gated_attention_bwd": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                    _P, _P, _P, _P]),
    "tg_gate_score_grad": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P]),
    "tg_gate_prune_layer_heads": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P,
                                       _I, _P, _P, _P, _P, _P, _P]),
    "tg_gate_prune_layer": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _F, _I, _I, _P, _P, _P, _I,
                                 _P, _P, _P, _P, _P, _P]),
    "tg_two_budget_prune_layer": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _F, _I, _I, _P, _P, _P, _I,
                                       _P, _P, _P, _P, _P, _P]),
    "tg_apply_rope": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _P]),
    "tg_normalize_scores": (_I, [_P, _I, _P, _P, _I, _I, _F, _P, _P, _P, _P]),
    "tg_gated_attention_eq8": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "tg_read_device_status": (_I, [_P, _P, _P]),
    "tg_set_wait_limit_ns": (_I, [ctypes.c_uint64]),
    "tg_set_test_withhold": (_I, [_I]),
}


class TGError(RuntimeError):
    def __init__(self, name: str, status: int, msg: str):
        super().__init__(f"{name} failed: status {status} ({msg})")
        self.status = status


_LIB: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtokengate.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m learned_token_pruning_07_b300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _ptr(t) -> Optional[int]:
    """Device address of a dense CUDA tensor (the C ABI takes no strides); None stays None.
    A host tensor or a strided view would reach a kernel as a wrong address, so both raise."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got shape {tuple(t.shape)} with strides {tuple(t.stride())}")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _check(name: str, status: int):
    if status != TG_OK:
        lib = load()
        msg = lib.tg_status_string(status).decode()
        if status == TG_ERR_CUDA:
            msg += f", cudaError {lib.tg_last_cuda_error()}"
        raise TGError(name, status, msg)


def _heads(g) -> int:
    """Gate heads of a gate tensor: [rows] is one head, [rows, H_g] is H_g."""
    return 1 if g is None or g.dim() == 1 else int(g.shape[1])


def _host_f32(x):
    import numpy as np
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return a, a.ctypes.data


# ---------------------------------------------------------------------------
# Entry points (tensors are torch CUDA tensors; bf16 data as torch.bfloat16 or int16/uint16)
# ---------------------------------------------------------------------------

def gate_score(h, W1, w2, s_out, g_out=None, instr_mask=None, b1=None, b2: float = 0.0,
               status=None, stream=None):
    T, d = h.shape
    d_g = W1.shape[0]
    st = load().tg_gate_score(_ptr(h), T, d, _ptr(instr_mask), _ptr(W1), _ptr(b1), _ptr(w2), float(b2),
                              d_g, _ptr(s_out), _ptr(g_out), _ptr(status), _stream(stream))
    _check("tg_gate_score", st)


def gate_score_heads(h, W1, W2, s_heads, s_sel, g_heads=None, instr_mask=None, b1=None, b2=None,
                     rmsnorm: bool = False, ln_eps: float = 1e-6, status=None, stream=None):
    """Per-head scores s_heads [T, H_g], gates g_heads and their head mean s_sel [T]."""
    T, d = h.shape
    H_g, d_g = W2.shape
    b2_a, b2_p = _host_f32(b2) if b2 is not None else (None, None)
    st = load().tg_gate_score_heads(_ptr(h), T, d, _ptr(instr_mask), _ptr(W1), _ptr(b1), _ptr(W2), b2_p, d_g,
                                    H_g, int(bool(rmsnorm)), float(ln_eps), _ptr(s_heads), _ptr(g_heads),
                                    _ptr(s_sel), _ptr(status), _stream(stream))
    del b2_a
    _check("tg_gate_score_heads", st)


def gate_score_rmsnorm(h, W1_folded, w2, s_out, g_out=None, instr_mask=None, b1=None, b2: float = 0.0,
                       ln_eps: float = 1e-6, status=None, stream=None):
    T, d = h.shape
    d_g = W1_folded.shape[0]
    st = load().tg_gate_score_rmsnorm(_ptr(h), T, d, _ptr(instr_mask), _ptr(W1_folded), _ptr(b1), _ptr(w2),
                                      float(b2), d_g, float(ln_eps), _ptr(s_out), _ptr(g_out), _ptr(status),
                                      _stream(stream))
    _check("tg_gate_score_rmsnorm", st)


def fold_rmsnorm_weight(W1, ln_weight, W1_out, stream=None):
    d_g, d = W1.shape
    _check("tg_fold_rmsnorm_weight", load().tg_fold_rmsnorm_weight(_ptr(W1), _ptr(ln_weight), d_g, d,
                                                                     _ptr(W1_out), _stream(stream)))


def topk_select(s, cu_seqlens, K: int, kept_idx, cu_kept, instr_mask=None, status=None, stream=None):
    B = cu_seqlens.numel() - 1
    st = load().tg_topk_select(_ptr(s), _ptr(instr_mask), _ptr(cu_seqlens), B, s.numel(), int(K),
                               _ptr(kept_idx), kept_idx.numel(), _ptr(cu_kept), _ptr(status),
                               _stream(stream))
    _check("tg_topk_select", st)


def gather_kept(h, cu_seqlens, kept_idx, cu_kept, h_kept, pos=None, g=None, pos_kept=None,
                g_kept=None, status=None, stream=None):
    T, d = h.shape
    B = cu_seqlens.numel() - 1
    st = load().tg_gather_kept(_ptr(h), _ptr(pos), _ptr(g), _heads(g), _ptr(cu_seqlens), B, T, d, _ptr(kept_idx),
                               _ptr(cu_kept), h_kept.shape[0], _ptr(h_kept), _ptr(pos_kept),
                               _ptr(g_kept), _ptr(status), _stream(stream))
    _check("tg_gather_kept", st)


def gated_attention(Q, K, V, cu_kept, tau, beta, O, max_seqlen: int, g=None, status=None,
                    stream=None, workspace=None):
    """tg_gated_attention, or tg_gated_attention_ws when a workspace tensor is given (see
    attention_workspace)."""
    M, H_q, d_h = Q.shape
    H_kv = K.shape[1]
    B = cu_kept.numel() - 1
    tau_a, tau_p = _host_f32(tau)
    beta_a, beta_p = _host_f32(beta)
    if workspace is None:
        st = load().tg_gated_attention(_ptr(Q), _ptr(K), _ptr(V), _ptr(g), _heads(g), _ptr(cu_kept), B, M,
                                       int(max_seqlen), H_q, H_kv, d_h, tau_p, beta_p, _ptr(O),
                                       _ptr(status), _stream(stream))
        name = "tg_gated_attention"
    else:
        nbytes = workspace.numel() * workspace.element_size()
        st = load().tg_gated_attention_ws(_ptr(Q), _ptr(K), _ptr(V), _ptr(g), _heads(g), _ptr(cu_kept), B, M,
                                          int(max_seqlen), H_q, H_kv, d_h, tau_p, beta_p, _ptr(O),
                                          _ptr(workspace) if nbytes else None, nbytes, _ptr(status),
                                          _stream(stream))
        name = "tg_gated_attention_ws"
    del tau_a, beta_a
    _check(name, st)


def gated_attention_noalloc(Q, K, V, cu_kept, tau, beta, O, max_seqlen: int, g=None, status=None, stream=None):
    """tg_gated_attention_noalloc: the split launch's scratch is the library's fixed array, so the
    caller passes no workspace (for callers that cannot allocate device memory)."""
    M, H_q, d_h = Q.shape
    H_kv = K.shape[1]
    B = cu_kept.numel() - 1
    tau_a, tau_p = _host_f32(tau)
    beta_a, beta_p = _host_f32(beta)
    st = load().tg_gated_attention_noalloc(_ptr(Q), _ptr(K), _ptr(V), _ptr(g), _heads(g), _ptr(cu_kept), B, M,
                                           int(max_seqlen), H_q, H_kv, d_h, tau_p, beta_p, _ptr(O), _ptr(status),
                                           _stream(stream))
    del tau_a, beta_a
    _check("tg_gated_attention_noalloc", st)


def gated_attention_workspace_size(B: int, max_seqlen: int, H_q: int, H_kv: int, d_h: int) -> int:
    return int(load().tg_gated_attention_workspace_size(int(B), int(max_seqlen), int(H_q), int(H_kv), int(d_h)))


def attention_workspace(B: int, max_seqlen: int, H_q: int, H_kv: int, d_h: int, device="cuda"):
    """A zero-filled workspace for gated_attention(..., workspace=...) of this shape (an empty
    tensor when the launch does not split)."""
    import torch
    n = gated_attention_workspace_size(B, max_seqlen, H_q, H_kv, d_h)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def normalize_scores(s, cu_seqlens, b_out, instr_mask=None, eps: float = 1e-6, b_sel=None, status=None,
                     stream=None):
    B = cu_seqlens.numel() - 1
    st = load().tg_normalize_scores(_ptr(s), _heads(s), _ptr(instr_mask), _ptr(cu_seqlens), B, s.shape[0],
                                    float(eps), _ptr(b_out), _ptr(b_sel), _ptr(status), _stream(stream))
    _check("tg_normalize_scores", st)


def gated_attention_eq8(Q, K, V, cu_kept, pos, gain, temp, O, max_seqlen: int, b=None, status=None,
                        stream=None):
    M, H_q, d_h = Q.shape
    H_kv = K.shape[1]
    B = cu_kept.numel() - 1
    gain_a, gain_p = _host_f32(gain)
    temp_a, temp_p = _host_f32(temp)
    st = load().tg_gated_attention_eq8(_ptr(Q), _ptr(K), _ptr(V), _ptr(b), _heads(b), _ptr(pos), _ptr(cu_kept), B, M,
                                       int(max_seqlen), H_q, H_kv, d_h, gain_p, temp_p, _ptr(O), _ptr(status),
                                       _stream(stream))
    del gain_a, temp_a
    _check("tg_gated_attention_eq8", st)


def gated_attention_lse(Q, K, V, cu_kept, tau, beta, O, lse, max_seqlen: int, g=None, status=None, stream=None):
    M, H_q, d_h = Q.shape
    tau_a, tau_p = _host_f32(tau)
    beta_a, beta_p = _host_f32(beta)
    st = load().tg_gated_attention_lse(_ptr(Q), _ptr(K), _ptr(V), _ptr(g), _heads(g), _ptr(cu_kept),
                                       cu_kept.numel() - 1, M,
                                       int(max_seqlen), H_q, K.shape[1], d_h, tau_p, beta_p, _ptr(O), _ptr(lse),
                                       _ptr(status), _stream(stream))
    del tau_a, beta_a
    _check("tg_gated_attention_lse", st)


def gated_attention_bwd(Q, K, V, O, dO, lse, cu_kept, tau, beta, dQ, dK, dV, dbias, max_seqlen: int, g=None,
                        status=None, stream=None):
    M, H_q, d_h = Q.shape
    tau_a, tau_p = _host_f32(tau)
    beta_a, beta_p = _host_f32(beta)
    st = load().tg_gated_attention_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(g), _heads(g), _ptr(O), _ptr(dO), _ptr(lse),
                                       _ptr(cu_kept), cu_kept.numel() - 1, M, int(max_seqlen), H_q, K.shape[1],
                                       d_h, tau_p, beta_p, _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(dbias),
                                       _ptr(status), _stream(stream))
    del tau_a, beta_a
    _check("tg_gated_attention_bwd", st)


def gate_score_grad(dbias, beta, g_kept, kept_idx, cu_kept, ds, stream=None):
    H_q = dbias.shape[1]
    beta_a, beta_p = _host_f32(beta)
    st = load().tg_gate_score_grad(_ptr(dbias), beta_p, _ptr(g_kept), _heads(g_kept), _ptr(kept_idx),
                                   _ptr(cu_kept), cu_kept.numel() - 1, kept_idx.numel(), H_q, ds.shape[0], _ptr(ds),
                                   _stream(stream))
    del beta_a
    _check("tg_gate_score_grad", st)


def gate_prune_layer(h, cu_seqlens, W1, w2, K: int, s_out, g_out, kept_idx, cu_kept, h_kept,
                     pos_kept=None, g_kept=None, pos=None, instr_mask=None, b1=None, b2: float = 0.0,
                     status=None, stream=None):
    T, d = h.shape
    B = cu_seqlens.numel() - 1
    st = load().tg_gate_prune_layer(_ptr(h), _ptr(pos), _ptr(instr_mask), _ptr(cu_seqlens), B, T, d,
                                    _ptr(W1), _ptr(b1), _ptr(w2), float(b2), W1.shape[0], int(K),
                                    _ptr(s_out), _ptr(g_out), _ptr(kept_idx), kept_idx.numel(),
                                    _ptr(cu_kept), _ptr(h_kept), _ptr(pos_kept), _ptr(g_kept),
                                    _ptr(status), _stream(stream))
    _check("tg_gate_prune_layer", st)


def gate_prune_layer_heads(h, cu_seqlens, W1, W2, K: int, s_heads, g_heads, s_sel, kept_idx, cu_kept, h_kept,
                           pos_kept=None, g_kept=None, pos=None, instr_mask=None, b1=None, b2=None,
                           status=None, stream=None):
    T, d = h.shape
    B = cu_seqlens.numel() - 1
    H_g, d_g = W2.shape
    b2_a, b2_p = _host_f32(b2) if b2 is not None else (None, None)
    st = load().tg_gate_prune_layer_heads(_ptr(h), _ptr(pos), _ptr(instr_mask), _ptr(cu_seqlens), B, T, d,
                                          _ptr(W1), _ptr(b1), _ptr(W2), b2_p, d_g, H_g, int(K), _ptr(s_heads),
                                          _ptr(g_heads), _ptr(s_sel), _ptr(kept_idx), kept_idx.numel(),
                                          _ptr(cu_kept), _ptr(h_kept), _ptr(pos_kept), _ptr(g_kept),
                                          _ptr(status), _stream(stream))
    del b2_a
    _check("tg_gate_prune_layer_heads", st)


def two_budget_prune_layer(h, cu_seqlens, W1, w2, K_prune: int, s_out, g_out, kept_idx, cu_packed, h_kept,
                           pos_kept=None, g_kept=None, pos=None, instr_mask=None, b1=None, b2: float = 0.0,
                           status=None, stream=None):
    T, d = h.shape
    B = cu_seqlens.numel() - 1
    st = load().tg_two_budget_prune_layer(_ptr(h), _ptr(pos), _ptr(instr_mask), _ptr(cu_seqlens), B, T, d,
                                          _ptr(W1), _ptr(b1), _ptr(w2), float(b2), W1.shape[0], int(K_prune),
                                          _ptr(s_out), _ptr(g_out), _ptr(kept_idx), kept_idx.numel(),
                                          _ptr(cu_packed), _ptr(h_kept), _ptr(pos_kept), _ptr(g_kept),
                                          _ptr(status), _stream(stream))
    _check("tg_two_budget_prune_layer", st)


def apply_rope(X, pos, theta: float, cu_kept=None, stream=None):
    cap, H, d_h = X.shape
    B = 0 if cu_kept is None else cu_kept.numel() - 1
    st = load().tg_apply_rope(_ptr(X), _ptr(pos), _ptr(cu_kept), B, cap, H, d_h, float(theta),
                              _stream(stream))
    _check("tg_apply_rope", st)


def read_device_status(status, stream=None) -> int:
    """Synchronise and return the raw device status bits (0 = ok)."""
    out = ctypes.c_int32(0)
    st = load().tg_read_device_status(_ptr(status), ctypes.addressof(out), _stream(stream))
    if st in (TG_ERR_INVALID_ARG, TG_ERR_CUDA):
        _check("tg_read_device_status", st)
    return out.value


def set_wait_limit_ns(ns: int):
    _check("tg_set_wait_limit_ns", load().tg_set_wait_limit_ns(int(ns)))


TG_WITHHOLD_GATE_SCORE, TG_WITHHOLD_ATTENTION, TG_WITHHOLD_BACKWARD, TG_WITHHOLD_GATE_SCORE_PEER = 1, 2, 4, 8


def set_test_withhold(mask: int):
    """Test hook: make the named kernels issue no loads so their bounded waits run out."""
    _check("tg_set_test_withhold", load().tg_set_test_withhold(int(mask)))
