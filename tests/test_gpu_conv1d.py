"""Depthwise causal conv1d against the oracle (Helion hackathon gallery,
"Causal Conv1d": out[b, d, t] = bias[d] + sum_k weight[d, k] x[b, d, t - W + 1 + k])."""
import numpy as np
import pytest
import torch

import oracle
import state_space_sequence_chunk_gb300 as ssd
from harness import TOL, rel_err

pytestmark = pytest.mark.gpu


def _inputs(b, d, L, W, dtype, seed, with_bias=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((b, d, L)).astype(np.float32)
    w = (rng.standard_normal((d, W)) / np.sqrt(W)).astype(np.float32)
    bias = rng.standard_normal(d).astype(np.float32) if with_bias else None
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    xt = torch.from_numpy(x).to(tdt)
    # the oracle sees exactly the values the kernel reads
    x_used = xt.float().numpy()
    return (xt.cuda(), torch.from_numpy(w).cuda(), None if bias is None else torch.from_numpy(bias).cuda(),
            x_used, w, bias)


@pytest.mark.parametrize("dtype,b,d,L,W,with_bias", [
    ("bf16", 2, 7, 4096, 4, True),    # vector path, the Mamba-2 width
    ("bf16", 2, 5, 1000, 3, True),    # vector path, 1000 % 8 == 0
    ("bf16", 3, 4, 1001, 4, True),    # ragged row length: one output per thread
    ("f32", 2, 6, 512, 5, False),     # fp32 vector path, widest halo from one lane
    ("f32", 1, 3, 300, 8, True),      # fp32 width 8: scalar path
    ("bf16", 1, 2, 3, 4, True),       # shorter than the filter
    ("f32", 2, 3, 64, 1, True),       # width 1: a per-channel scale
])
def test_conv1d_matches_oracle(dtype, b, d, L, W, with_bias):
    x, w, bias, x_used, w_np, b_np = _inputs(b, d, L, W, dtype, seed=L + W)
    out = ssd.causal_conv1d(x, w, bias)
    torch.cuda.synchronize()
    ref = oracle.causal_conv1d(x_used, w_np, b_np)
    assert np.all(np.isfinite(out.float().cpu().numpy()))
    assert rel_err(out.float().cpu().numpy(), ref) < TOL[dtype]


def test_conv1d_fp32_is_near_exact():
    """fp32 in and out: W fused multiply-adds per output, so the result is within
    a few ulps of the fp64 oracle (a much tighter check than the bound)."""
    x, w, bias, x_used, w_np, b_np = _inputs(2, 9, 2048, 4, "f32", seed=5)
    out = ssd.causal_conv1d(x, w, bias)
    torch.cuda.synchronize()
    ref = oracle.causal_conv1d(x_used, w_np, b_np)
    assert np.max(np.abs(out.cpu().numpy() - ref)) < 1e-5 * max(1.0, np.max(np.abs(ref)))


def test_conv1d_empty():
    x = torch.empty((2, 3, 0), dtype=torch.bfloat16, device="cuda")
    w = torch.ones((3, 4), device="cuda")
    out = ssd.causal_conv1d(x, w, None)
    assert out.shape == x.shape
