"""The algorithmic byte counts behind bench.py's roofline figures, checked
against the sizes of the tensors each kernel reads and writes, listed here one
by one (host logic, no GPU)."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from state_space_sequence_chunk_gb300 import synth  # noqa: E402


def _tensor_bytes(shape, itemsize):
    n = 1
    for d in shape:
        n *= d
    return n * itemsize


@pytest.mark.parametrize("B,T,H,K,V,C", [(4, 4096, 16, 128, 128, 64), (1, 300, 3, 64, 32, 64),
                                          (2, 128, 2, 16, 48, 32)])
def test_gdn_step_bytes(B, T, H, K, V, C):
    NT = -(-T // C)
    f = 4
    reads_h = [(B, T, H, K), (B, T, H, K), (B, T, H, V), (B, T, H), (B, H, K, V)]      # k, w, u, g, h0
    writes_h = [(B, H, NT, K, V), (B, T, H, V), (B, H, K, V)]                          # h, v_new, final
    reads_o = [(B, T, H, K), (B, T, H, K), (B, T, H, V), (B, H, NT, K, V), (B, T, H)]  # q, k, v_new, h, g
    writes_o = [(B, T, H, V)]                                                          # o
    want = sum(_tensor_bytes(s, f) for s in reads_h + writes_h + reads_o + writes_o)
    assert bench.gdn_bytes(B, T, H, K, V, C) == want


def test_gdn_bench_shape_is_hbm_bound():
    # the bench shape moves 1.62 GB against 30.1 GFLOP: at any GB300 peak pair
    # (6.8-8 TB/s, 0.9-1.1 PFLOP/s TF32) the bytes take longer than the FLOPs
    g = bench.GDN
    nbytes = bench.gdn_bytes(g["B"], g["T"], g["H"], g["K"], g["V"], g["chunk"])
    assert 1.60e9 < nbytes < 1.64e9
    assert nbytes / 8.0e12 > 30.2e9 / 0.9e15


def test_ssd_byte_model_mamba2_layer():
    w = synth.workload("mamba2_layer_bf16")
    b, L, H, P, N, G, Q = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk
    nc = -(-L // Q)
    x = _tensor_bytes((b, L, H, P), 2)
    bc = _tensor_bytes((b, L, G, N), 2)
    g_rows = _tensor_bytes((b, H, nc * Q), 4)              # Gcs or dtT, token-contiguous
    hid = _tensor_bytes((b, H, nc, P, N), 2)
    fin = _tensor_bytes((b, H, P, N), 4)
    d = _tensor_bytes((H,), 4) if w.with_D else 0
    assert w.init_std == 0                                  # no initial state in this workload
    m = bench.byte_model(w)
    assert m["chunk_cumsum"] == _tensor_bytes((b, L, H), 4) + H * 4 + 2 * g_rows
    assert m["fwd_pass_state"] == x + bc + 2 * g_rows + hid + fin
    assert m["compute_out"] == x + 2 * bc + 2 * g_rows + hid + d + x
