"""Failure detection without a GPU fault.

fwd_pass_state hands the running state from one CTA's work range to the next
through a flag in global memory; the receiving CTA's wait is bounded (about
1 s of SM clock).  Here a test hook makes every range withhold its hand-off: the
waits must give up, the launch must end with the error bit set (no hang, no
fault), and the same context must then produce correct results again.  The
next launching call reports the failure as SSD_ERR_TIMEOUT.
"""
import time

import numpy as np
import pytest

import state_space_sequence_chunk_gb300 as ssd
from state_space_sequence_chunk_gb300 import synth
from harness import TOL, gpu_fwd, oracle_fwd, rel_err, small, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("init_std,ngroups", [(0.1, 2), (0.0, 1), (0.1, 1)],
                         ids=["per-head", "paired-heads", "paired-heads-init"])
def test_withheld_handoff_times_out_and_is_reported(init_std, ngroups):
    # 2 heads x 16 chunks: far fewer units than CTAs, so every CTA takes one
    # chunk and each chain crosses 15 range boundaries.  With both heads in one
    # group they walk as one pair-chain; one head per group takes the one-head
    # kernel.
    w = small(seqlen=4096, nheads=2, ngroups=ngroups, headdim=64, dstate=128, chunk=256,
              dtype="bf16", init_std=init_std, batch=1)
    inp = synth.make_inputs(w)
    dev = to_device(inp, "bf16")
    assert ssd.ssd_take_device_errors() == 0
    t0 = time.time()
    try:
        ssd.ssd_debug_withhold_handoffs(True)
        ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                    dev["init_state"], chunk_size=256)
        errs = ssd.ssd_take_device_errors()   # synchronises
    finally:
        ssd.ssd_debug_withhold_handoffs(False)
    elapsed = time.time() - t0
    assert errs & 1, "the bounded hand-off wait should have given up"
    assert elapsed < 60
    # the context is still usable, and the next call is exact again
    y, fin = gpu_fwd(dev, 256)
    y_ref, fin_ref = oracle_fwd(inp)
    assert rel_err(y, y_ref) < TOL["bf16"] and rel_err(fin, fin_ref) < TOL["bf16"]


@pytest.mark.parametrize("ngroups", [1, 2], ids=["paired-heads", "per-head"])
def test_timeout_is_returned_by_the_next_call(ngroups):
    """A wait that gave up cannot be returned by the asynchronous call that
    enqueued it: the kernel raises a page-locked host word at its end, and the
    next launching call returns SSD_ERR_TIMEOUT without enqueuing anything.
    The report clears the record, so the call after that is exact again."""
    import torch
    w = small(seqlen=4096, nheads=2, ngroups=ngroups, headdim=64, dstate=128, chunk=256,
              dtype="bf16", init_std=0.1, batch=1)
    inp = synth.make_inputs(w)
    dev = to_device(inp, "bf16")
    assert ssd.ssd_take_device_errors() == 0
    try:
        ssd.ssd_debug_withhold_handoffs(True)
        ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                    dev["init_state"], chunk_size=256)     # enqueued: returns SSD_OK
        torch.cuda.synchronize()
    finally:
        ssd.ssd_debug_withhold_handoffs(False)
    y_sentinel = torch.full_like(dev["x"], 7.0)
    with pytest.raises(ssd.SSDError, match="SSD_ERR_TIMEOUT") as e:
        ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                    dev["init_state"], chunk_size=256, out=y_sentinel)
    assert e.value.code == 9
    torch.cuda.synchronize()
    assert bool((y_sentinel == 7.0).all()), "the reporting call must enqueue nothing"
    assert ssd.ssd_take_device_errors() == 0   # reported once, then cleared
    y, fin = gpu_fwd(dev, 256)
    y_ref, fin_ref = oracle_fwd(inp)
    assert rel_err(y, y_ref) < TOL["bf16"] and rel_err(fin, fin_ref) < TOL["bf16"]
