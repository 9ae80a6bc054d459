"""GPU parity: the backward of token-gated attention and the gate-score gradient, against the
fp64 oracle (which is pinned to torch autograd and to finite differences).

bf16 rounds to nearest with an 8-bit significand, so a rounded value is off by at most
u = 2^-8 of itself. Two roundings move the GPU's gradients away from the exact ones:
  * like flash-attention backwards, D_i = dO_i . o_i is formed from the forward's bf16 output,
    so |dD_i| <= u sum_d |dO_id o_id|; dX = P (dP - D) is linear in D;
  * the tensor-core products take P and c_h dX as bf16 operands (fp32 accumulation).
To first order the gradients then move by at most, per element (c_h = tau_h / sqrt(d_h)):
    dQ_id:    c_h dD_i sum_j P_ij |k_jd|  +  u c_h sum_j |dX_ij| |k_jd|
    dK_jd:    sum_h [c_h sum_i P_ij dD_i |q_id|  +  u c_h sum_i |dX_ij| |q_id|]
    dV_jd:    sum_h u sum_i P_ij |dO_id|
    dbias_jh: sum_i P_ij dD_i                     (summed from fp32 P and dX)
The bar per element is that bound plus 1e-4 of the gradient's largest magnitude (fp32 sums and
the fp32 log-sum-exp); log-sum-exp within 1e-3 absolute."""
import numpy as np
import pytest
import torch

from learned_token_pruning_07_b300 import binding as tg
from learned_token_pruning_07_b300 import inputs as I
from oracle import tokengate_oracle as O
from tests._helpers import bf16_dev_to_f64, dev, host, status_word

pytestmark = pytest.mark.gpu


def _case(wl, lens, seed, use_g=True, beta_zero=False, g_override=None):
    cu = I.cu_seqlens_of(lens)
    M = int(cu[-1])
    at = I.make_attention_inputs(wl, M, tag_extra=seed)
    if g_override is not None:
        at["g"] = g_override
    rng = np.random.default_rng(300 + seed)
    dO = I.f32_to_bf16_bits(rng.standard_normal((M, wl.H_q, wl.d_h)).astype(np.float32))
    tau, beta = at["tau"], np.zeros_like(at["beta"]) if beta_zero else at["beta"]
    g = at["g"] if use_g else None
    Qd, Kd, Vd = dev(at["Q"]), dev(at["K"]), dev(at["V"])
    O_d = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    lse = torch.full((M, wl.H_q), 7.0, dtype=torch.float32, device="cuda")
    st = status_word()
    mx = max(lens)
    tg.gated_attention_lse(Qd, Kd, Vd, dev(cu), tau, beta, O_d, lse, max_seqlen=mx,
                           g=dev(g) if use_g else None, status=st)
    f = lambda *shape: torch.full(shape, 12345.0, dtype=torch.float32, device="cuda")
    dQ, dK, dV, dbias = f(M, wl.H_q, wl.d_h), f(M, wl.H_kv, wl.d_h), f(M, wl.H_kv, wl.d_h), f(M, wl.H_q)
    tg.gated_attention_bwd(Qd, Kd, Vd, O_d, dev(dO), lse, dev(cu), tau, beta, dQ, dK, dV, dbias, max_seqlen=mx,
                           g=dev(g) if use_g else None, status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    Q64, K64, V64 = (I.bf16_bits_to_f64(at[k]) for k in ("Q", "K", "V"))
    g64 = None if g is None else g.astype(np.float64)
    ref_lse = O.gated_attention_lse(Q64, K64, g64, cu, tau.astype(np.float64), beta.astype(np.float64))
    np.testing.assert_allclose(host(lse), ref_lse, rtol=0, atol=1e-3)
    ref = O.gated_attention_bwd(Q64, K64, V64, g64, I.bf16_bits_to_f64(dO), cu, tau.astype(np.float64),
                                beta.astype(np.float64))
    got = [host(t).astype(np.float64) for t in (dQ, dK, dV, dbias)]
    bounds = _rounding_bounds(Q64, K64, V64, g64, I.bf16_bits_to_f64(dO), cu, tau, beta)
    for name, a, b, bnd in zip(("dQ", "dK", "dV", "dbias"), got, ref, bounds):
        assert np.all(np.isfinite(a)), name
        tol = bnd + 1e-4 * float(np.max(np.abs(b))) + 1e-7
        excess = np.abs(a - b) - tol
        assert float(excess.max()) <= 0.0, (name, float(np.abs(a - b).max()), float(tol.max()))
    return at, cu, g, tau, beta, ref, dbias


U_BF16 = 2.0 ** -8


def _rounding_bounds(Q, K, V, g, dO, cu, tau, beta):
    """Per-element first-order bounds of the gradient change caused by the bf16 roundings of O
    (inside D) and of the tensor-core operands P and c_h dX (see the module docstring). g is
    [M] or [M, H_g] (query head h reads gate column h / (H_q / H_g))."""
    M, H_q, d_h = Q.shape
    group = H_q // K.shape[1]
    bq, bk, bv, bb = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V), np.zeros((M, H_q))
    for s_ in range(len(cu) - 1):
        a, e = int(cu[s_]), int(cu[s_ + 1])
        n = e - a
        if n == 0:
            continue
        tri = np.tril(np.ones((n, n), dtype=bool))
        for h in range(H_q):
            kv = h // group
            c = float(tau[h]) / np.sqrt(d_h)
            x = c * (Q[a:e, h] @ K[a:e, kv].T)
            if g is not None and beta[h] != 0:
                gh = g[a:e] if g.ndim == 1 else g[a:e, h // (H_q // g.shape[1])]
                x = x + float(beta[h]) * np.log(gh)[None, :]
            x = np.where(tri, x, -np.inf)
            P = np.exp(x - x.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            o = P @ V[a:e, kv]
            dP = dO[a:e, h] @ V[a:e, kv].T
            dX = P * (dP - np.sum(dO[a:e, h] * o, axis=1, keepdims=True))
            dD = U_BF16 * np.sum(np.abs(dO[a:e, h] * o), axis=1)          # [n]
            aK, aQ = np.abs(K[a:e, kv]), np.abs(Q[a:e, h])
            bq[a:e, h] = c * dD[:, None] * (P @ aK) + U_BF16 * c * (np.abs(dX) @ aK)
            bk[a:e, kv] += c * (P * dD[:, None]).T @ aQ + U_BF16 * c * np.abs(dX).T @ aQ
            bv[a:e, kv] += U_BF16 * P.T @ np.abs(dO[a:e, h])
            bb[a:e, h] = (P * dD[:, None]).sum(axis=0)
    return bq, bk, bv, bb


def test_backward_tiny_dh64():
    _case(I.WORKLOADS["tiny"], [96, 33], seed=1)


@pytest.mark.parametrize("lens", [[1], [63, 64, 65], [129, 0, 2, 200], [700, 1030]])
def test_backward_varlen_dh128(lens):
    _case(I.WORKLOADS["qwen3_1p7b_8k"], lens, seed=len(lens))


def test_backward_at_the_bench_size():
    # the bench's backward runs on the 32K workload's kept rows at K = 4096: one sequence of
    # 4,096 document + 256 instruction rows (34 key tiles, both heads of every GQA group)
    wl = I.WORKLOADS["sweep_32k"]
    _case(wl, [wl.K + wl.instr_lens[0]], seed=41)


def test_backward_ragged_batch_kept_lengths():
    # the first three sequences of the ragged batch as the prune step keeps them at K = 2048
    wl = I.WORKLOADS["ragged_b8"]
    lens = [min(wl.K, d) + n for d, n in zip(wl.doc_lens[:3], wl.instr_lens[:3])]
    _case(I.WORKLOADS["qwen3_1p7b_8k"], lens, seed=42)


def test_backward_mha_and_odd_group():
    _case(I.with_changes(I.WORKLOADS["qwen3_1p7b_8k"], H_q=4, H_kv=4), [130, 70], seed=21)
    _case(I.with_changes(I.WORKLOADS["qwen3_1p7b_8k"], H_q=6, H_kv=2), [130, 70], seed=22)


def test_backward_at_the_largest_head_count():
    # 128 query heads, the most the call takes, over 64 kv heads of 64
    _case(I.with_changes(I.WORKLOADS["tiny"], H_q=128, H_kv=64), [70, 130], seed=23)


def test_backward_is_deterministic():
    # every output element is written once after a fixed-order sum: two runs agree bit for bit
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    lens = [300, 129]
    cu = I.cu_seqlens_of(lens)
    M = int(cu[-1])
    at = I.make_attention_inputs(wl, M, tag_extra=31)
    dO = I.f32_to_bf16_bits(np.random.default_rng(331).standard_normal((M, wl.H_q, wl.d_h)).astype(np.float32))
    Qd, Kd, Vd, gd, cud, dOd = dev(at["Q"]), dev(at["K"]), dev(at["V"]), dev(at["g"]), dev(cu), dev(dO)
    O_d = torch.zeros((M, wl.H_q, wl.d_h), dtype=torch.int16, device="cuda")
    lse = torch.zeros((M, wl.H_q), dtype=torch.float32, device="cuda")
    st = status_word()
    tg.gated_attention_lse(Qd, Kd, Vd, cud, at["tau"], at["beta"], O_d, lse, max_seqlen=max(lens), g=gd, status=st)
    runs = []
    for _ in range(2):
        out = [torch.zeros(sh, dtype=torch.float32, device="cuda")
               for sh in ((M, wl.H_q, wl.d_h), (M, wl.H_kv, wl.d_h), (M, wl.H_kv, wl.d_h), (M, wl.H_q))]
        tg.gated_attention_bwd(Qd, Kd, Vd, O_d, dOd, lse, cud, at["tau"], at["beta"], *out, max_seqlen=max(lens),
                               g=gd, status=st)
        runs.append([host(t) for t in out])
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    for a, b in zip(*runs):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_backward_without_gate_and_with_beta_zero():
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    _case(wl, [150], seed=7, use_g=False)
    _case(wl, [150], seed=8, beta_zero=True)


def test_backward_with_subnormal_gates():
    # every key's gate below the smallest normal fp32: the key bias is beta_h ln g_j of the
    # subnormal value itself (no flush to zero), in the forward and in both backward passes
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    M = 200
    g = (np.random.default_rng(41).uniform(1.0, 50.0, M) * 1e-40).astype(np.float32)
    assert np.all(g < np.finfo(np.float32).tiny) and np.all(g > 0)
    _case(wl, [M], seed=12, g_override=g)


def test_gate_score_gradient_through_kept_rows():
    wl = I.WORKLOADS["qwen3_1p7b_8k"]
    lens = [180, 77]
    at, cu, g, tau, beta, ref, dbias = _case(wl, lens, seed=9)
    M = int(cu[-1])
    T = 3 * M
    kept = np.sort(np.random.default_rng(10).choice(T, M, replace=False)).astype(np.int32)
    ds = torch.zeros(T, dtype=torch.float32, device="cuda")
    tg.gate_score_grad(dbias, beta, dev(g), dev(kept), dev(cu), ds)
    torch.cuda.synchronize()
    want = O.gate_score_grad(ref[3], beta.astype(np.float64), g.astype(np.float64), kept, T)
    got = host(ds).astype(np.float64)
    assert np.all(got[np.setdiff1d(np.arange(T), kept)] == 0.0)
    # the bias-gradient bound carried through the same chain: sum_h beta_h bound_jh (1 - g_j)
    Q64, K64, V64 = (I.bf16_bits_to_f64(at[k]) for k in ("Q", "K", "V"))
    rng = np.random.default_rng(300 + 9)
    dO64 = I.bf16_bits_to_f64(I.f32_to_bf16_bits(rng.standard_normal((M, wl.H_q, wl.d_h)).astype(np.float32)))
    bb = _rounding_bounds(Q64, K64, V64, g.astype(np.float64), dO64, cu, tau, beta)[3]
    tol = np.zeros(T)
    tol[kept] = (bb @ beta.astype(np.float64)) * (1.0 - g) + 1e-4 * float(np.max(np.abs(want))) + 1e-7
    assert np.all(np.abs(got - want) <= tol)
