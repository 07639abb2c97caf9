"""ssd_fwd_noalloc: the forward pass for callers that cannot allocate device
memory (a framework that hands out only fixed buffers, a loop that must not
call cudaMalloc/cudaFree).  Its scratch is a fixed device array inside the
library; these tests call it through the C ABI and check it against ssd_fwd
with a caller-owned workspace, on two calls in a row (the array keeps the
previous call's contents, which must not leak into the next result).  Both
paths run the same kernels on the same inputs, so the results must be equal
bit for bit."""
import ctypes

import pytest
import torch

import state_space_sequence_chunk_gb300 as ssd
from state_space_sequence_chunk_gb300 import build as ssd_build
from state_space_sequence_chunk_gb300 import synth
from harness import small, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ssd_build.build()
    return ssd.load_library()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("dtype,Q", [("bf16", 128), ("f32", 64)])
def test_noalloc_matches_ssd_fwd_twice(lib, dtype, Q):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed, L in ((21, 700), (22, 333)):   # two calls in a row, different inputs
        w = small(seqlen=L, nheads=4, ngroups=2, headdim=64, dstate=128, chunk=Q, dtype=dtype,
                  seed=seed)
        dev = to_device(synth.make_inputs(w), dtype)
        y_ref, f_ref = ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                                   dev["init_state"], chunk_size=Q)
        y = torch.empty_like(dev["x"])
        fin = torch.empty_like(f_ref)
        dims = ssd.dims_for(dev["x"], dev["B"], Q)
        rc = lib.ssd_fwd_noalloc(ctypes.byref(dims), _p(dev["x"]), _p(dev["dt"]), _p(dev["A"]),
                                 _p(dev["B"]), _p(dev["C"]), _p(dev["D"]), _p(dev["init_state"]),
                                 _p(y), _p(fin), stream)
        assert rc == 0, lib.ssd_status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)
        assert torch.equal(fin, f_ref)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    w = synth.WORKLOADS["mamba2_layer_bf16"]
    dims = ssd.Dims(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk,
                    ssd.SSD_BF16, 0)
    assert ssd.ssd_fwd_workspace_bytes(dims) > 32 << 20
    x = torch.empty(16, device="cuda")
    args = [_p(x)] * 9
    rc = lib.ssd_fwd_noalloc(ctypes.byref(dims), *args,
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 5   # SSD_ERR_WORKSPACE, nothing enqueued
