"""Shared helpers of the GPU tests: inputs from the seeded generator, the CUDA
path through the binding, the oracle on the same inputs, and the error metric
max|out - ref| / max|ref| with the tolerances the tests enforce."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import state_space_sequence_chunk_gb300 as ssd
from state_space_sequence_chunk_gb300 import synth

# max|out - ref| / max|ref| bounds: fp32 inputs (TF32-class tensor-core products)
# and bf16 inputs; the same bound applies to y, final_state and the chunk-start
# states.
TOL = {"f32": 1e-3, "bf16": 1e-2}


def rel_err(out, ref) -> float:
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref))
    if den == 0:
        return float(np.max(np.abs(out)))
    return float(np.max(np.abs(out - ref)) / den)


def small(name="small", batch=1, seqlen=300, nheads=4, headdim=64, dstate=64, ngroups=2,
          chunk=64, dtype="bf16", init_std=0.1, with_D=True, seed=7, **kw) -> synth.Workload:
    return synth.Workload(name, batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype,
                          init_std=init_std, with_D=with_D, seed=seed, **kw)


def to_device(inp: dict, dtype: str, device="cuda"):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        elif k in ("x", "B", "C"):
            out[k] = torch.from_numpy(v).to(device=device).to(tdt).contiguous()
        else:
            out[k] = torch.from_numpy(v).to(device=device).contiguous()
    return out


def gpu_fwd(dev: dict, chunk: int, **kw):
    y, fin = ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                         dev["init_state"], chunk_size=chunk, **kw)
    torch.cuda.synchronize()
    assert ssd.ssd_take_device_errors() == 0, "a bounded wait in a kernel gave up"
    return y.float().cpu().numpy(), (None if fin is None else fin.cpu().numpy())


def _slice_inputs(inp: dict, b: int, h: int, T: int | None = None) -> dict:
    """The inputs of one (batch, head) recurrence, optionally its first T tokens."""
    H, G = inp["x"].shape[2], inp["B"].shape[2]
    g = h // (H // G)
    t = slice(0, T)
    return dict(x=inp["x"][b:b + 1, t, h:h + 1], dt=inp["dt"][b:b + 1, t, h:h + 1],
                A=inp["A"][h:h + 1], B=inp["B"][b:b + 1, t, g:g + 1],
                C=inp["C"][b:b + 1, t, g:g + 1],
                D=None if inp["D"] is None else inp["D"][h:h + 1],
                init_state=None if inp["init_state"] is None else inp["init_state"][b:b + 1, h:h + 1])


def whole_tensor_errors(inp: dict, y, fin, hid=None, chunk: int = 0, threads: int | None = None):
    """max|out - ref| / max|ref| over the WHOLE y, final_state (and, with `hid`
    and `chunk`, the chunk-start states) of a problem.

    Every (batch, head) slice is an independent recurrence, so the oracle runs
    slice by slice on one thread per host core (the C oracle releases the
    interpreter lock); each slice's largest |difference| and |reference| are
    folded into global maxima, so the result is exactly the global metric
    without holding the fp64 reference of the whole tensor.  `y` is
    [b, L, H, P], `fin` [b, H, P, N] and `hid` [b, H, nc, N, P] (the GPU's
    transposed layout), all numpy.  Returns a dict of relative errors.
    """
    import concurrent.futures as cf
    import os
    import threading

    b, L, H, P = inp["x"].shape
    lib = oracle.load()
    acc = {"y": [0.0, 0.0], "final_state": [0.0, 0.0], "hiddens": [0.0, 0.0]}
    lock = threading.Lock()

    def fold(key, out, ref):
        d = float(np.max(np.abs(np.asarray(out, np.float64) - ref))) if ref.size else 0.0
        m = float(np.max(np.abs(ref))) if ref.size else 0.0
        with lock:
            acc[key][0] = max(acc[key][0], d)
            acc[key][1] = max(acc[key][1], m)

    def run(bh):
        bi, h = bh
        s = _slice_inputs(inp, bi, h)
        if hid is not None:
            yr, fr, ck = oracle.recurrence(**s, ckpt_every=chunk, lib=lib)
            fold("hiddens", np.swapaxes(hid[bi, h], -1, -2), ck[0, 0])
        else:
            yr, fr = oracle.recurrence(**s, lib=lib)
        fold("y", y[bi, :, h], yr[0, :, 0])
        fold("final_state", fin[bi, h], fr[0, 0])

    pairs = [(bi, h) for bi in range(b) for h in range(H)]
    with cf.ThreadPoolExecutor(max_workers=threads or os.cpu_count() or 1) as ex:
        list(ex.map(run, pairs))
    keys = ["y", "final_state"] + (["hiddens"] if hid is not None else [])
    return {k: (acc[k][0] / acc[k][1] if acc[k][1] > 0 else acc[k][0]) for k in keys}


def oracle_fwd(inp: dict, bh=None, ckpt_every: int = 0):
    """Oracle on all (b, h) or only on the listed (b, h) pairs (each pair is an
    independent recurrence, so a subset is computed exactly)."""
    if bh is None:
        return oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                 inp["init_state"], ckpt_every=ckpt_every)
    H, G = inp["x"].shape[2], inp["B"].shape[2]
    res = []
    for b, h in bh:
        g = h // (H // G)
        r = oracle.recurrence(
            inp["x"][b:b + 1, :, h:h + 1], inp["dt"][b:b + 1, :, h:h + 1], inp["A"][h:h + 1],
            inp["B"][b:b + 1, :, g:g + 1], inp["C"][b:b + 1, :, g:g + 1],
            None if inp["D"] is None else inp["D"][h:h + 1],
            None if inp["init_state"] is None else inp["init_state"][b:b + 1, h:h + 1],
            ckpt_every=ckpt_every)
        res.append(r)
    return res
