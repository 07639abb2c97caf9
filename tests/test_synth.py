"""The seeded input generator: deterministic, with the stated distributions."""
import math

import numpy as np
import pytest
import torch

from state_space_sequence_chunk_gb300 import synth


def test_splitmix_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    # (state += 0x9E3779B97F4A7C15, then the mix function).
    out = synth.raw64(np.uint64(0), 0, 3)
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_distinct_streams():
    w = synth.WORKLOADS["tiny_fp32"]
    a, b = synth.make_inputs(w), synth.make_inputs(w)
    for k in a:
        if a[k] is not None:
            assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["B"], a["C"])


def test_distributions():
    w = synth.WORKLOADS["small_fp32"]
    inp = synth.make_inputs(w)
    x = inp["x"].ravel()
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert np.all(inp["dt"] > 0)
    z = np.log(np.expm1(inp["dt"].astype(np.float64)))   # inverse softplus
    assert abs(z.mean() + 3.0) < 0.02 and abs(z.std() - 0.5) < 0.02
    assert np.all(inp["A"] < -1.0 + 1e-6) and np.all(inp["A"] >= -16.0)
    assert abs(inp["init_state"].std() - 0.1) < 0.002


@pytest.mark.parametrize("seed", [0, 1])
def test_bf16_rounding_matches_torch(seed):
    v = np.random.default_rng(seed).standard_normal(100000).astype(np.float32) * 3
    ours = synth.round_to_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, ref)
    bits = synth.bf16_bits(ours)
    assert np.array_equal(bits, torch.from_numpy(ours).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def test_workload_table():
    w = synth.WORKLOADS
    assert [k for k in w] == ["tiny_fp32", "small_fp32", "mamba2_layer_bf16",
                              "long_context_bf16", "short_streams_bf16"]
    assert w["mamba2_layer_bf16"].tokens == 16384
    assert w["short_streams_bf16"].ngroups == 8
