"""ssd_fwd_host -- the forward pass on host buffers, batch slices pipelined
against their copies -- against ssd_fwd on the device and against the oracle.

Each batch element is an independent recurrence ("The Mamba-2 Recurrence"),
so a slice of the batch is a problem of its own: with single-pass chains the
arithmetic per (batch, head) is the same as in one ssd_fwd call over the whole
batch, and the host results are bit-identical to it.
"""
import numpy as np
import pytest
import torch

import state_space_sequence_chunk_gb300 as ssd
from state_space_sequence_chunk_gb300 import synth
from harness import TOL, gpu_fwd, oracle_fwd, rel_err, small, to_device

pytestmark = pytest.mark.gpu


def _host(inp, dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        else:
            t = torch.from_numpy(v)
            out[k] = (t.to(tdt) if k in ("x", "B", "C") else t.float()).contiguous().pin_memory()
    return out


def _run_host(h, chunk, nslices, **kw):
    y, fin = ssd.ssd_fwd_host(h["x"], h["dt"], h["A"], h["B"], h["C"], h["D"], h["init_state"],
                              chunk_size=chunk, nslices=nslices, **kw)
    torch.cuda.synchronize()
    assert ssd.ssd_take_device_errors() == 0
    return y, fin


@pytest.mark.parametrize("dtype,nslices", [("bf16", 1), ("bf16", 2), ("bf16", 3), ("bf16", 5),
                                           ("f32", 2)])
def test_host_equals_device(dtype, nslices):
    w = small(seqlen=300, nheads=4, ngroups=2, headdim=64 if dtype == "bf16" else 32,
              dstate=128 if dtype == "bf16" else 16, chunk=128, dtype=dtype, batch=5,
              init_std=0.2)
    inp = synth.make_inputs(w)
    h = _host(inp, dtype)
    y, fin = _run_host(h, 128, nslices)
    y_dev, fin_dev = gpu_fwd(to_device(inp, dtype), 128)
    assert np.array_equal(y.float().numpy(), y_dev)
    assert np.array_equal(fin.numpy(), fin_dev)


def test_host_state_in_place_and_no_D():
    w = small(seqlen=200, nheads=4, ngroups=1, headdim=64, dstate=128, chunk=64, dtype="bf16",
              batch=4, init_std=0.3, with_D=False)
    inp = synth.make_inputs(w)
    h = _host(inp, "bf16")
    state = h["init_state"].clone().pin_memory()
    h["init_state"] = state
    y, fin = _run_host(h, 64, 4, final_out=state)
    assert fin.data_ptr() == state.data_ptr()
    y_ref, f_ref = oracle_fwd(inp)
    assert rel_err(y.float().numpy(), y_ref) < TOL["bf16"]
    assert rel_err(state.numpy(), f_ref) < TOL["bf16"]


def test_host_long_chains_against_the_oracle():
    """Long chains (64 chunks: the two-pass form of fwd_pass_state) per slice."""
    w = small(seqlen=64 * 64, nheads=2, ngroups=1, headdim=64, dstate=128, chunk=64,
              dtype="bf16", batch=2, init_std=0.1)
    inp = synth.make_inputs(w)
    y, fin = _run_host(_host(inp, "bf16"), 64, 2)
    y_ref, f_ref = oracle_fwd(inp)
    assert rel_err(y.float().numpy(), y_ref) < TOL["bf16"]
    assert rel_err(fin.numpy(), f_ref) < TOL["bf16"]


def test_host_empty_sequence_passes_the_state():
    w = small(seqlen=0, nheads=2, ngroups=1, headdim=32, dstate=16, dtype="bf16", batch=3,
              init_std=0.5)
    inp = synth.make_inputs(w)
    h = _host(inp, "bf16")
    y, fin = _run_host(h, 64, 3)
    assert y.numel() == 0
    assert np.array_equal(fin.numpy(), inp["init_state"])
