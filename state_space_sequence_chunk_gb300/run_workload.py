"""Run the forward pass on one of the synthetic workloads a few times.

A minimal driver for profilers (ncu) and quick manual checks:

    python -m state_space_sequence_chunk_gb300.run_workload --workload mamba2_layer_bf16 --iters 3

Each iteration is one ``ssd_fwd`` call (chunk_cumsum, fwd_pass_state,
compute_out); the device is synchronised at the end and the kernels' device
error bits are checked.
"""
from __future__ import annotations

import argparse
import sys

import torch

import state_space_sequence_chunk_gb300 as ssd
from state_space_sequence_chunk_gb300 import synth


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="mamba2_layer_bf16",
                    choices=list(synth.WORKLOADS) + list(synth.CONTEXT_WORKLOADS))
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--chunk", type=int, default=0, help="override the chunk size")
    args = ap.parse_args(argv)
    w = synth.workload(args.workload)
    Q = args.chunk or w.chunk
    inp = synth.make_inputs(w)
    dev = torch.device("cuda")
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    t = {k: (None if v is None else torch.from_numpy(v).to(dev)) for k, v in inp.items()}
    for k in ("x", "B", "C"):
        t[k] = t[k].to(tdt)
    dims = ssd.dims_for(t["x"], t["B"], Q)
    ws = torch.empty(ssd.ssd_fwd_workspace_bytes(dims), dtype=torch.uint8, device=dev)
    y = torch.empty_like(t["x"])
    fin = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device=dev)
    for _ in range(args.iters):
        ssd.ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                    chunk_size=Q, workspace=ws, out=y, final_out=fin)
    torch.cuda.synchronize()
    errs = ssd.ssd_take_device_errors()
    if errs:
        print(f"device error bits {errs:#x}", file=sys.stderr)
        return 1
    print(f"{w.name}: {args.iters} forward passes ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
