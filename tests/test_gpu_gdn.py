"""Gated DeltaNet chunk kernels (Helion hackathon gallery, "GDN chunk_fwd_h" /
"GDN chunk_fwd_o") against the step-by-step fp64 oracle: shapes with K and V
multiples of 16 run on the TF32 tensor cores, the others on the CUDA cores."""
import numpy as np
import pytest
import torch

import oracle
import state_space_sequence_chunk_gb300 as ssd
from harness import TOL, rel_err

pytestmark = pytest.mark.gpu


def gdn_inputs(B, T, H, K, V, chunk, seed, with_h0=True):
    """Seeded inputs with the pages' conventions: per-token log gates <= 0 summed
    within each chunk (inclusive), keys and WY rows scaled so the state stays O(1)."""
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((B, T, H, K)) / np.sqrt(K)).astype(np.float32)
    k = (rng.standard_normal((B, T, H, K)) / np.sqrt(K)).astype(np.float32)
    w = (rng.standard_normal((B, T, H, K)) / np.sqrt(K) * 0.5).astype(np.float32)
    u = rng.standard_normal((B, T, H, V)).astype(np.float32)
    gamma = -np.abs(rng.normal(0.05, 0.03, (B, T, H)))
    g = np.zeros_like(gamma)
    for t in range(T):
        g[:, t] = gamma[:, t] + (g[:, t - 1] if t % chunk else 0.0)
    g = g.astype(np.float32)
    h0 = rng.standard_normal((B, H, K, V)).astype(np.float32) * 0.1 if with_h0 else None
    return q, k, w, u, g, h0


@pytest.mark.parametrize("B,T,H,K,V,chunk,with_h0", [
    (2, 300, 3, 128, 128, 64, True),    # ragged last chunk, full K and V tiles
    (1, 256, 2, 64, 32, 32, False),     # no initial state
    (2, 100, 2, 16, 48, 16, True),      # V not a multiple of the 32-column tile
    (1, 7, 1, 32, 64, 64, True),        # shorter than one chunk
    (1, 130, 2, 32, 37, 32, True),      # V not a multiple of 4 (scalar loads and stores)
    (1, 200, 2, 128, 100, 64, False),   # two V halves of chunk_fwd_o, the second partial
    # K and V multiples of 16: the tensor-core kernels
    (2, 333, 2, 64, 128, 64, True),     # two 64-column V tiles of chunk_fwd_h, ragged
    (1, 500, 3, 128, 16, 32, True),     # smallest V, chunk 32
    (1, 90, 2, 16, 128, 16, False),     # smallest K and chunk
])
def test_gdn_matches_oracle(B, T, H, K, V, chunk, with_h0):
    q, k, w, u, g, h0 = gdn_inputs(B, T, H, K, V, chunk, seed=T + K)
    dev = lambda a: None if a is None else torch.from_numpy(a).cuda()
    h, v_new, fin = ssd.gdn_chunk_fwd_h(dev(k), dev(w), dev(u), dev(g), dev(h0), chunk=chunk)
    o = ssd.gdn_chunk_fwd_o(dev(q), dev(k), v_new, h, dev(g), chunk=chunk)
    torch.cuda.synchronize()
    h_ref, vn_ref, fin_ref = oracle.gdn_fwd_h(k, w, u, g, h0, chunk=chunk)
    o_ref = oracle.gdn_fwd_o(q, k, vn_ref, h_ref, g, chunk=chunk)
    assert rel_err(h.cpu().numpy(), h_ref) < TOL["f32"]
    assert rel_err(v_new.cpu().numpy(), vn_ref) < TOL["f32"]
    assert rel_err(fin.cpu().numpy(), fin_ref) < TOL["f32"]
    assert rel_err(o.cpu().numpy(), o_ref) < TOL["f32"]


def test_gdn_binding_rejects_other_dtypes():
    q, k, w, u, g, h0 = gdn_inputs(1, 64, 1, 16, 16, 64, seed=4)
    dev = lambda a: torch.from_numpy(a).cuda()
    with pytest.raises(TypeError):
        ssd.gdn_chunk_fwd_h(dev(k), dev(w).double(), dev(u), dev(g), dev(h0), chunk=64)


def test_gdn_empty_sequence_passes_the_state():
    q, k, w, u, g, h0 = gdn_inputs(1, 0, 2, 32, 32, 64, seed=3)
    dev = lambda a: torch.from_numpy(a).cuda()
    h, v_new, fin = ssd.gdn_chunk_fwd_h(dev(k), dev(w), dev(u), dev(g), dev(h0), chunk=64)
    torch.cuda.synchronize()
    assert h.numel() == 0 and v_new.numel() == 0
    assert torch.equal(fin.cpu(), torch.from_numpy(h0))


def test_gdn_bench_shape_whole_tensors():
    """The benchmark's shape (B4, T4096, H16, K = V = 128, chunk 64: each CTA
    walks 64 chunks on the tensor cores) against the oracle on every output
    element: h, v_new, final_state and o.  Each (batch, head) is an independent
    recurrence, so the oracle runs slice by slice on all host cores and the
    maxima are folded into global ones."""
    import concurrent.futures as cf
    import os
    import threading
    B, T, H, K, V, C = 4, 4096, 16, 128, 128, 64
    q, k, w, u, g, h0 = gdn_inputs(B, T, H, K, V, C, seed=4096 + 128)
    dev = lambda a: torch.from_numpy(a).cuda()
    h, v_new, fin = ssd.gdn_chunk_fwd_h(dev(k), dev(w), dev(u), dev(g), dev(h0), chunk=C)
    o = ssd.gdn_chunk_fwd_o(dev(q), dev(k), v_new, h, dev(g), chunk=C)
    torch.cuda.synchronize()
    assert ssd.ssd_take_device_errors() == 0
    h, v_new, fin, o = (t.cpu().numpy() for t in (h, v_new, fin, o))
    acc = {n: [0.0, 0.0] for n in ("h", "v_new", "final_state", "o")}
    lock = threading.Lock()
    lib = oracle.load()

    def fold(name, out, ref):
        d, m = float(np.max(np.abs(out - ref))), float(np.max(np.abs(ref)))
        with lock:
            acc[name][0] = max(acc[name][0], d)
            acc[name][1] = max(acc[name][1], m)

    def run(bh):
        b, hh = bh
        sl = lambda a: a[b:b + 1, :, hh:hh + 1]
        hr, vr, fr = oracle.gdn_fwd_h(sl(k), sl(w), sl(u), sl(g), h0[b:b + 1, hh:hh + 1],
                                      chunk=C, lib=lib)
        orf = oracle.gdn_fwd_o(sl(q), sl(k), vr, hr, sl(g), chunk=C, lib=lib)
        fold("h", h[b, hh], hr[0, 0])
        fold("v_new", v_new[b, :, hh], vr[0, :, 0])
        fold("final_state", fin[b, hh], fr[0, 0])
        fold("o", o[b, :, hh], orf[0, :, 0])

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        list(ex.map(run, [(b, hh) for b in range(B) for hh in range(H)]))
    errs = {n: a[0] / a[1] for n, a in acc.items()}
    print("\ngdn bench shape whole-tensor rel err " +
          ", ".join(f"{n} {e:.3e}" for n, e in errs.items()))
    for n, e in errs.items():
        assert e < TOL["f32"], (n, e)


def test_gdn_repeatable_at_bench_shape():
    """Twenty calls of both kernels at the benchmark's shape give bit-identical
    h, v_new, final_state and o (the chunk walk's warps hand TMEM columns and
    shared tiles to one another: a missing ordering shows up as a call that
    differs)."""
    B, T, H, K, V, C = 4, 4096, 16, 128, 128, 64
    q, k, w, u, g, h0 = gdn_inputs(B, T, H, K, V, C, seed=11)
    dev = lambda a: torch.from_numpy(a).cuda()
    tq, tk, tw, tu, tg, th = dev(q), dev(k), dev(w), dev(u), dev(g), dev(h0)

    def run():
        h, v_new, fin = ssd.gdn_chunk_fwd_h(tk, tw, tu, tg, th, chunk=C)
        return h, v_new, fin, ssd.gdn_chunk_fwd_o(tq, tk, v_new, h, tg, chunk=C)

    first = run()
    differ = []
    for i in range(20):
        out = run()
        if not all(torch.equal(a, b) for a, b in zip(out, first)):
            differ.append(i)
    torch.cuda.synchronize()
    assert ssd.ssd_take_device_errors() == 0
    assert not differ, f"calls {differ} differ from the first"
