"""The whole-tensor parity metric of the GPU tests, checked on the CPU.

``harness.whole_tensor_errors`` runs the oracle slice by slice on several
threads and folds each slice's maxima into global ones.  Given the oracle's
own outputs it must report exactly zero, and a single planted difference
anywhere in y or the chunk-start states must come back at its exact size
relative to the global maximum of the reference.
"""
import numpy as np

import oracle
from harness import rel_err, small, whole_tensor_errors
from state_space_sequence_chunk_gb300 import synth


def _case():
    w = small(seqlen=300, nheads=4, ngroups=2, headdim=16, dstate=8, chunk=64, dtype="bf16",
              batch=2)
    inp = synth.make_inputs(w)
    y, fin, ck = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["init_state"], ckpt_every=64)
    return inp, y, fin, ck


def test_exact_outputs_give_zero():
    inp, y, fin, ck = _case()
    err = whole_tensor_errors(inp, y, fin, np.swapaxes(ck, -1, -2), 64, threads=3)
    assert err == {"y": 0.0, "final_state": 0.0, "hiddens": 0.0}


def test_planted_differences_are_found_at_their_size():
    inp, y, fin, ck = _case()
    y2 = y.copy()
    y2[1, 123, 3, 5] += 0.5 * np.abs(y).max()
    f2 = fin.copy()
    f2[0, 2, 7, 1] -= 0.125 * np.abs(fin).max()
    hid = np.swapaxes(ck, -1, -2).copy()
    hid[0, 1, 2, 3, 4] += 0.25 * np.abs(ck).max()
    err = whole_tensor_errors(inp, y2, f2, hid, 64, threads=4)
    assert np.isclose(err["y"], 0.5) and np.isclose(err["y"], rel_err(y2, y))
    assert np.isclose(err["final_state"], 0.125)
    assert np.isclose(err["hiddens"], 0.25)
