"""Shared helpers for the GPU parity tests (device transfer, tolerances, sampled rows)."""
import numpy as np
import torch

from learned_token_pruning_07_b300 import inputs as I

# Tolerances. Gate values: 1e-2 absolute. Attention: 2e-2 max-abs and 1e-2 mean-relative
# (bf16 output against the fp64 oracle). Scores: the fp32 accumulation of d exact bf16
# products carries ~d * 2^-24 * sum|terms| of rounding (well under 1e-3 at d = 2048), plus
# the hardware exp/reciprocal used in SiLU (~1e-6 relative); 2e-3 + 1e-3 relative is the bar.
G_ATOL = 1e-2
ATTN_MAX_ABS = 2e-2
ATTN_MEAN_REL = 1e-2
S_ATOL = 2e-3
S_RTOL = 1e-3


def dev(a, dtype=None):
    """numpy -> CUDA tensor (uint16 bf16 bits become torch.int16 with the same bytes)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a).cuda()
    return t if dtype is None else t.to(dtype)


def host(t):
    a = t.cpu().numpy()
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    return a


def bf16_dev_to_f64(t):
    return I.bf16_bits_to_f64(host(t))


def zeros_i32(n):
    return torch.zeros(n, dtype=torch.int32, device="cuda")


def status_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def attention_close(got, ref):
    """(max-abs error, mean-relative error) of got vs ref."""
    err = np.abs(got - ref)
    return float(err.max()) if err.size else 0.0, float(err.mean() / max(np.abs(ref).mean(), 1e-30)) if err.size else 0.0


def sampled_rows(cu, instr_rows, n_random, seed, extra=()):
    """Query rows for sampled parity: first/last rows of every sequence, rows around
    instruction tokens, plus seeded random rows."""
    rows = set(extra)
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        if e > a:
            rows.update([a, min(a + 1, e - 1), e - 1, max(a, e - 2), max(a, e - 129), min(e - 1, a + 127),
                         min(e - 1, a + 128)])
    for r in instr_rows[:: max(1, len(instr_rows) // 64)]:
        rows.update([max(0, r - 1), r, min(int(cu[-1]) - 1, r + 1)])
    rng = np.random.default_rng(seed)
    if int(cu[-1]) > 0:
        rows.update(rng.integers(0, int(cu[-1]), n_random).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < int(cu[-1])), dtype=np.int64)
