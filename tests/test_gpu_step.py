"""ssd_step -- the token-by-token recurrence for decoding -- against the oracle.

The oracle's recurrence run from the same initial state over the same tokens
is the definition the step follows ("The Mamba-2 Recurrence"); the chunked
ssd_fwd computes the same result another way, and a sequence fed through the
step one token per call must continue exactly as one call over all of it.
"""
import numpy as np
import pytest
import torch

import state_space_sequence_chunk_gb300 as ssd
from state_space_sequence_chunk_gb300 import synth
from harness import TOL, gpu_fwd, oracle_fwd, rel_err, small, to_device

pytestmark = pytest.mark.gpu


def _step(dev, state):
    y = ssd.ssd_step(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], state)
    torch.cuda.synchronize()
    return y.float().cpu().numpy()


@pytest.mark.parametrize("dtype,L,H,G,P,N,with_D", [
    ("bf16", 1, 6, 2, 64, 128, True),     # one decode step, Mamba-2 head shape
    ("f32", 5, 4, 1, 32, 16, True),       # a few tokens in one call
    ("bf16", 3, 2, 2, 128, 256, False),   # largest P and N, no D
    ("f32", 1, 8, 4, 16, 48, True),       # N not a multiple of 128
])
def test_step_matches_oracle(dtype, L, H, G, P, N, with_D):
    w = small(seqlen=L, nheads=H, ngroups=G, headdim=P, dstate=N, chunk=64, dtype=dtype,
              init_std=0.3, with_D=with_D, batch=3)
    inp = synth.make_inputs(w)
    dev = to_device(inp, dtype)
    state = dev["init_state"].clone()
    y = _step(dev, state)
    y_ref, f_ref = oracle_fwd(inp)
    assert np.all(np.isfinite(y))
    assert rel_err(y, y_ref) < TOL[dtype]
    assert rel_err(state.cpu().numpy(), f_ref) < TOL[dtype]


def test_step_by_step_equals_one_call_and_ssd_fwd():
    """T one-token calls == one T-token call (bit for bit: the state is fp32 either
    way), and both agree with the chunked ssd_fwd over the same tokens."""
    T = 9
    w = small(seqlen=T, nheads=4, ngroups=2, headdim=64, dstate=128, chunk=64, dtype="bf16",
              init_std=0.2, batch=2)
    inp = synth.make_inputs(w)
    dev = to_device(inp, "bf16")
    s_all = dev["init_state"].clone()
    y_all = _step(dev, s_all)
    s_one = dev["init_state"].clone()
    ys = []
    for t in range(T):
        tok = {k: (v[:, t:t + 1].contiguous() if k in ("x", "dt", "B", "C") else v)
               for k, v in dev.items()}
        ys.append(_step(tok, s_one))
    assert np.array_equal(np.concatenate(ys, axis=1), y_all)
    assert torch.equal(s_one, s_all)
    y_fwd, f_fwd = gpu_fwd(dev, 64)
    assert rel_err(y_all, y_fwd) < TOL["bf16"]
    assert rel_err(s_all.cpu().numpy(), f_fwd) < TOL["bf16"]


def test_step_continues_a_chunked_prefix():
    """Streaming use: ssd_fwd over a prompt, then decode steps from its final
    state, against the oracle over the whole sequence."""
    L0, T = 300, 4
    w = small(seqlen=L0 + T, nheads=4, ngroups=1, headdim=64, dstate=128, chunk=128,
              dtype="bf16", init_std=0.1, batch=2)
    inp = synth.make_inputs(w)
    dev = to_device(inp, "bf16")
    pre = {k: (v[:, :L0].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in dev.items()}
    _, f0 = gpu_fwd(pre, 128)
    state = torch.from_numpy(f0).cuda()
    post = {k: (v[:, L0:].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in dev.items()}
    y = _step(post, state)
    y_ref, f_ref = oracle_fwd(inp)
    assert rel_err(y, y_ref[:, L0:]) < TOL["bf16"]
    assert rel_err(state.cpu().numpy(), f_ref) < TOL["bf16"]


def test_step_empty_is_a_no_op():
    w = small(seqlen=0, nheads=2, ngroups=1, headdim=32, dstate=16, dtype="bf16", init_std=0.1)
    inp = synth.make_inputs(w)
    dev = to_device(inp, "bf16")
    state = dev["init_state"].clone()
    y = ssd.ssd_step(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], state)
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert torch.equal(state, dev["init_state"])
