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
