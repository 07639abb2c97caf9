"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Every comparison is element by element on the same seeded inputs, with the
bound max|out - ref| / max|ref| <= 1e-3 (fp32 inputs) or 1e-2 (bf16 inputs).
Every problem, the full-size workloads included, is compared in full: the
oracle runs on every (batch, head) slice (each an exact, independent
recurrence) and the maxima are taken over the whole tensor.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import state_space_sequence_chunk_gb300 as ssd
from state_space_sequence_chunk_gb300 import build as ssd_build
from state_space_sequence_chunk_gb300 import synth
from harness import TOL, gpu_fwd, oracle_fwd, rel_err, small, to_device, whole_tensor_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ssd_build.build()
    ssd.load_library()


# --- step 1: chunk_cumsum ---------------------------------------------------

@pytest.mark.parametrize("Q,L", [(64, 64), (64, 301), (128, 1000), (256, 257), (256, 4096)])
def test_chunk_cumsum(Q, L):
    w = small(seqlen=L, nheads=37, chunk=Q, batch=2)
    inp = synth.make_inputs(w)
    dev = to_device(inp, w.dtype)
    Gcs, dtT = ssd.ssd_chunk_cumsum(dev["dt"], dev["A"], Q)
    torch.cuda.synchronize()
    Gcs, dtT = Gcs.cpu().numpy(), dtT.cpu().numpy()
    ref = oracle.chunk_cumsum(inp["dt"], inp["A"], Q)
    assert rel_err(Gcs[:, :, :L], ref) < 2e-5
    assert np.array_equal(dtT[:, :, :L], np.moveaxis(inp["dt"], 1, 2))
    # padded tail: dt reads as 0, so G repeats the value at the last real token
    assert not np.any(dtT[:, :, L:])
    if Gcs.shape[2] > L:
        assert np.array_equal(Gcs[:, :, L:], np.repeat(Gcs[:, :, L - 1:L], Gcs.shape[2] - L, 2))
    # decay-mask invariant: G never increases inside a chunk, so every kept
    # entry 2^{g_i - g_j} (i >= j) is at most 1
    d = np.diff(Gcs.reshape(2, 37, -1, Q), axis=3)
    assert np.all(d <= 0)


# --- step 2: fwd_pass_state -------------------------------------------------

@pytest.mark.parametrize("dtype,Q,L,P,N", [("f32", 64, 300, 32, 16), ("f32", 128, 700, 64, 64),
                                           ("bf16", 256, 600, 64, 128), ("bf16", 128, 128, 16, 256),
                                           ("bf16", 64, 1000, 128, 32)])
def test_fwd_pass_state(dtype, Q, L, P, N):
    w = small(seqlen=L, headdim=P, dstate=N, chunk=Q, dtype=dtype, nheads=4, ngroups=2, batch=2)
    inp = synth.make_inputs(w)
    dev = to_device(inp, dtype)
    Gcs, dtT = ssd.ssd_chunk_cumsum(dev["dt"], dev["A"], Q)
    hid, fin = ssd.ssd_fwd_pass_state(dev["x"], dev["B"], Gcs, dtT, dev["init_state"], Q)
    torch.cuda.synchronize()
    _, fin_ref, ck_ref = oracle_fwd(inp, ckpt_every=Q)
    # hiddens is stored transposed, [b, H, nc, N, P]
    assert rel_err(hid.float().permute(0, 1, 2, 4, 3).cpu().numpy(), ck_ref) < TOL[dtype]
    assert rel_err(fin.cpu().numpy(), fin_ref) < TOL[dtype]


# --- the whole pass on small and edge-case problems --------------------------

CASES = [
    # dtype, Q, L, H, G, P, N, init, D
    ("f32", 64, 256, 2, 1, 32, 16, False, True),      # tiny workload shape
    ("f32", 64, 1, 2, 1, 32, 16, True, True),         # one token
    ("f32", 64, 63, 3, 3, 16, 32, True, False),       # shorter than a chunk, G = H
    ("f32", 128, 389, 4, 2, 64, 64, True, True),      # ragged tail
    # fp32 on the TF32 tensor-core kernels
    ("f32", 256, 700, 4, 2, 64, 128, True, True),     # two query blocks per chunk, ragged
    ("f32", 128, 333, 2, 1, 128, 128, True, True),    # largest TF32 P and N
    ("f32", 64, 450, 4, 2, 64, 128, True, True),      # C h^T, C B^T in two passes over N, Q = 64
    ("f32", 64, 300, 4, 4, 48, 48, False, True),      # P, N not multiples of 32
    ("bf16", 256, 511, 4, 1, 64, 128, False, True),   # ragged, Q = 256
    ("bf16", 256, 4096, 2, 1, 64, 128, True, True),
    ("bf16", 128, 130, 8, 2, 64, 128, True, True),    # 4 heads per group
    ("bf16", 64, 200, 2, 2, 128, 256, True, True),    # P = 128 with the largest N
    ("bf16", 128, 300, 2, 1, 256, 256, True, True),   # largest P and N
    # N = 256 on the tensor-core compute_out (Q <= 128)
    ("bf16", 128, 777, 4, 2, 64, 256, True, True),    # Q = 128, ragged
    ("bf16", 64, 500, 6, 2, 32, 256, False, True),    # Q = 64, P = 32
    ("bf16", 128, 400, 2, 1, 64, 192, True, False),   # N = 192: padded to 256 by the TMA
    ("bf16", 256, 333, 4, 2, 256, 64, False, True),   # largest P, ragged, Q = 256
    ("f32", 64, 200, 2, 1, 256, 128, True, True),     # largest P, fp32
    ("bf16", 128, 333, 2, 1, 16, 16, True, True),     # smallest P and N
    ("bf16", 64, 150, 2, 1, 48, 48, True, True),      # N splits a warp's state rows
    # no initial state: heads 2k, 2k+1 of one group walk together, sharing B
    ("bf16", 128, 1000, 6, 3, 32, 64, False, True),   # paired heads, ragged tail
    ("bf16", 256, 4096, 4, 1, 64, 128, False, False), # paired, one chunk per CTA
    ("bf16", 64, 700, 6, 2, 64, 128, False, True),    # odd heads per group: unpaired
    ("bf16", 128, 1000, 3, 3, 64, 128, True, True),   # unpaired, with an initial state
    ("bf16", 64, 300, 4, 2, 64, 48, False, True),     # paired, TMA-stored 48-row states
    # long chains: local pass, scan over each chain's ranges, apply pass
    ("bf16", 128, 15999, 4, 2, 64, 128, True, True),  # with an initial state, ragged
    ("bf16", 256, 20000, 2, 1, 32, 64, False, True),  # ~76 ranges per chain, P = 32
    # long chains on the one-head kernel (unpaired heads, P > 64 or N > 128)
    ("bf16", 64, 4096, 3, 3, 64, 128, True, True),    # odd heads: ranges of one or two chunks
    ("bf16", 128, 9000, 2, 1, 128, 64, False, True),  # two 64-column blocks of P, ragged
    ("bf16", 128, 8300, 2, 1, 64, 256, True, False),  # two 128-row blocks of N, ragged
    ("bf16", 64, 40000, 1, 1, 64, 192, True, True),   # N = 192 (padded rows), ~8 chunks per range
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-Q{c[1]}-L{c[2]}-H{c[3]}G{c[4]}-P{c[5]}N{c[6]}"
                                              for c in CASES])
def test_fwd_small(case):
    dtype, Q, L, H, G, P, N, with_init, with_D = case
    w = small(seqlen=L, nheads=H, ngroups=G, headdim=P, dstate=N, chunk=Q, dtype=dtype,
              init_std=0.1 if with_init else 0.0, with_D=with_D, batch=2)
    inp = synth.make_inputs(w)
    y, fin = gpu_fwd(to_device(inp, dtype), Q)
    y_ref, fin_ref = oracle_fwd(inp)
    assert np.all(np.isfinite(y))
    assert rel_err(y, y_ref) < TOL[dtype]
    assert rel_err(fin, fin_ref) < TOL[dtype]


def _random_cases(n=48, seed=20261202):
    """Seeded random shapes across the whole size contract (dtype, chunk, ragged
    length, heads and groups, P and N multiples of 16 up to 256, initial state
    and D on or off), with the oracle's work kept to a few seconds per case."""
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        dtype = ["f32", "bf16"][rng.integers(2)]
        Q = int(rng.choice([64, 128, 256]))
        L = int(rng.integers(1, 1500))
        G = int(rng.choice([1, 2, 3]))
        H = G * int(rng.integers(1, 4))
        P = 16 * int(rng.integers(1, 17))
        N = 16 * int(rng.integers(1, 17))
        b = int(rng.integers(1, 3))
        if b * L * H * P * N > 6e8:       # oracle budget
            continue
        cases.append((dtype, Q, L, H, G, P, N, bool(rng.integers(2)), bool(rng.integers(2)), b))
    return cases


RANDOM_CASES = _random_cases()


@pytest.mark.parametrize("case", RANDOM_CASES,
                         ids=[f"{c[0]}-Q{c[1]}-L{c[2]}-H{c[3]}G{c[4]}-P{c[5]}N{c[6]}-b{c[9]}"
                              for c in RANDOM_CASES])
def test_random_shapes(case):
    dtype, Q, L, H, G, P, N, with_init, with_D, b = case
    w = small(seqlen=L, nheads=H, ngroups=G, headdim=P, dstate=N, chunk=Q, dtype=dtype,
              init_std=0.1 if with_init else 0.0, with_D=with_D, batch=b)
    inp = synth.make_inputs(w)
    y, fin = gpu_fwd(to_device(inp, dtype), Q)
    y_ref, fin_ref = oracle_fwd(inp)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(fin))
    assert rel_err(y, y_ref) < TOL[dtype]
    assert rel_err(fin, fin_ref) < TOL[dtype]
    assert ssd.ssd_take_device_errors() == 0


# --- the five workloads -------------------------------------------------------

def fwd_with_hiddens(w, dev):
    """ssd_fwd with an explicit workspace (the launch chain bench.py times),
    returning y, final_state and the chunk-start states it left in the
    workspace ([b, H, nc, N, P], the x dtype)."""
    dims = ssd.dims_for(dev["x"], dev["B"], w.chunk)
    ws = torch.empty(ssd.ssd_fwd_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    y, fin = ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                         dev["init_state"], chunk_size=w.chunk, workspace=ws)
    torch.cuda.synchronize()
    assert ssd.ssd_take_device_errors() == 0, "a bounded wait in a kernel gave up"
    gb, hb = ssd.ssd_intermediate_bytes(dims)
    off = 2 * ((gb + 255) // 256 * 256)
    nc = -(-w.seqlen // w.chunk)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    hid = ws[off:off + hb].view(tdt).view(w.batch, w.nheads, nc, w.dstate, w.headdim)
    return (y.float().cpu().numpy(), fin.cpu().numpy(), hid.float().cpu().numpy())


def check_whole(name, w, inp, dev):
    """The whole output tensors of one workload against the oracle (every
    (batch, head) slice, one thread per host core), with global maxima."""
    y, fin, hid = fwd_with_hiddens(w, dev)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(fin))
    err = whole_tensor_errors(inp, y, fin, hid, w.chunk)
    print(f"\n{name}: whole-tensor rel err y {err['y']:.3e}, final_state "
          f"{err['final_state']:.3e}, chunk-start states {err['hiddens']:.3e} "
          f"(bound {TOL[w.dtype]})")
    for k, v in err.items():
        assert v < TOL[w.dtype], (k, v)


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload(name):
    """Every output of the five workloads, compared in full: y, final_state and
    the chunk-start states, max|out - ref| / max|ref| over the whole tensor."""
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w)
    check_whole(name, w, inp, to_device(inp, w.dtype))


@pytest.mark.parametrize("name", list(synth.CONTEXT_WORKLOADS))
def test_pages_example_shape(name):
    """The pages' own example problem (b4, 16384 tokens, H8, P64, G1, chunk
    128, bf16) at state sizes 64, 128 and 256: 128 chunks per chain, so
    fwd_pass_state takes its two-pass form where the paired geometry allows
    (N <= 128); every output compared in full against the oracle."""
    w = synth.CONTEXT_WORKLOADS[name]
    inp = synth.make_inputs(w)
    check_whole(name, w, inp, to_device(inp, w.dtype))


# --- properties -----------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_size_invariance(dtype):
    """The recurrence has no chunk parameter: every chunk size meets the bound
    against one oracle run."""
    w = small(seqlen=777, nheads=4, ngroups=2, headdim=64, dstate=64, dtype=dtype)
    inp = synth.make_inputs(w)
    y_ref, fin_ref = oracle_fwd(inp)
    dev = to_device(inp, dtype)
    for Q in (64, 128, 256):
        y, fin = gpu_fwd(dev, Q)
        assert rel_err(y, y_ref) < TOL[dtype], Q
        assert rel_err(fin, fin_ref) < TOL[dtype], Q


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_composition(dtype):
    """final_state fed back as init_state continues the sequence: two calls
    split at a token that is not a chunk boundary give, joined, the oracle's
    result for the whole sequence (the split chunks the tokens differently, so
    the two GPU results differ from one whole run at the rounding level of the
    products; each must meet the bound)."""
    w = small(seqlen=700, dtype=dtype, headdim=32, dstate=32)
    inp = synth.make_inputs(w)
    dev = to_device(inp, dtype)
    y_ref, f_ref = oracle_fwd(inp)
    L1 = 300
    d1 = {k: (v[:, :L1].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in dev.items()}
    y1, f1 = gpu_fwd(d1, 64)
    d2 = {k: (v[:, L1:].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in dev.items()}
    d2["init_state"] = torch.from_numpy(f1).cuda()
    y2, f2 = gpu_fwd(d2, 64)
    assert rel_err(np.concatenate([y1, y2], axis=1), y_ref) < TOL[dtype]
    assert rel_err(f2, f_ref) < TOL[dtype]


@pytest.mark.parametrize("dtype,Q", [("f32", 128), ("bf16", 256)])
def test_strong_decay_never_overflows(dtype, Q):
    """Decays of up to -46 per token (log2 units): above the diagonal 2^{g_i - g_j}
    overflows to inf, and the mask must discard it (a select, not a product)."""
    w = small(seqlen=600, dtype=dtype, chunk=Q, headdim=32, dstate=32)
    inp = synth.make_inputs(w)
    inp["A"] = np.full_like(inp["A"], -16.0)
    inp["dt"] = np.full_like(inp["dt"], 2.0)
    y, fin = gpu_fwd(to_device(inp, dtype), Q)
    y_ref, fin_ref = oracle_fwd(inp)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(fin))
    assert rel_err(y, y_ref) < TOL[dtype]
    assert rel_err(fin, fin_ref) < TOL[dtype]


def test_inplace_state_update():
    w = small(seqlen=300, dtype="bf16", chunk=128, headdim=64, dstate=128)
    inp = synth.make_inputs(w)
    dev = to_device(inp, "bf16")
    y_ref, f_ref = gpu_fwd(dev, 128)
    state = dev["init_state"].clone()
    y, f = ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], state,
                       chunk_size=128, final_out=state)
    torch.cuda.synchronize()
    assert np.array_equal(state.cpu().numpy(), f_ref)
    assert np.array_equal(y.float().cpu().numpy(), y_ref)


def test_empty_inputs():
    w = small(seqlen=0, dtype="bf16", chunk=64)
    inp = synth.make_inputs(w)
    dev = to_device(inp, "bf16")
    y, fin = ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                         dev["init_state"], chunk_size=64)
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert np.array_equal(fin.cpu().numpy(), inp["init_state"])
    w0 = small(seqlen=10, batch=0, dtype="bf16")
    d0 = to_device(synth.make_inputs(w0), "bf16")
    y0, f0 = ssd.ssd_fwd(d0["x"], d0["dt"], d0["A"], d0["B"], d0["C"], d0["D"], d0["init_state"],
                         chunk_size=64)
    assert y0.numel() == 0 and f0.numel() == 0


def test_deterministic_and_stream_ordered():
    w = small(seqlen=1000, dtype="bf16", chunk=256, headdim=64, dstate=128)
    inp = synth.make_inputs(w)
    dev = to_device(inp, "bf16")
    y1, f1 = gpu_fwd(dev, 256)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y2, f2 = ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                             dev["init_state"], chunk_size=256)
    s.synchronize()
    assert np.array_equal(y1, y2.float().cpu().numpy())
    assert np.array_equal(f1, f2.cpu().numpy())


def test_repeatable_across_group_switches():
    """The pages' example shape at chunk 256 (b4, 16384 tokens, H8 in one group:
    a group switch every 8 units of compute_out) run 60 times, L2 flushed
    between calls: every y and final_state bit-identical to the first call's,
    and the first compared in full with the oracle.  A stage handed back before
    the loads from it had completed showed here as the next unit's x in the
    D x term of the group's last head, in a few calls out of a hundred."""
    w = synth.CONTEXT_WORKLOADS["pages_example_bf16"].replace(chunk=256)
    inp = synth.make_inputs(w)
    dev = to_device(inp, w.dtype)
    dims = ssd.dims_for(dev["x"], dev["B"], w.chunk)
    ws = torch.empty(ssd.ssd_fwd_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(dev["x"])
    fin = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def run():
        flush.fill_(1)
        ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["init_state"],
                    chunk_size=w.chunk, workspace=ws, out=y, final_out=fin)

    run()
    torch.cuda.synchronize()
    y0, f0 = y.clone(), fin.clone()
    differ = []
    for i in range(60):
        run()
        torch.cuda.synchronize()
        if not (torch.equal(y, y0) and torch.equal(fin, f0)):
            differ.append(i)
    assert ssd.ssd_take_device_errors() == 0
    assert not differ, f"calls {differ} differ from the first"
    err = whole_tensor_errors(inp, y0.float().cpu().numpy(), f0.cpu().numpy())
    assert err["y"] < TOL["bf16"] and err["final_state"] < TOL["bf16"], err


@pytest.mark.parametrize("name,chunk", [
    ("mamba2_layer_bf16", 256),        # paired fwd_pass_state with hand-offs, Q = 256
    ("long_context_bf16", 256),        # paired two-pass form, initial state
    ("short_streams_bf16", 128),       # paired, initial state, 4 heads per group
    ("pages_example_n256_bf16", 128),  # one-head two-pass form, N = 256 compute_out
    ("small_fp32", 64),                # TF32 kernels
])
def test_repeatable_full_size(name, chunk):
    """Twenty calls of ssd_fwd on a full-size workload, L2 flushed between them,
    all bit-identical to the first (every kernel here reduces in a fixed order,
    so a call that differs exposes a missing ordering between warps or CTAs)."""
    w = synth.workload(name).replace(chunk=chunk)
    dev = to_device(synth.make_inputs(w), w.dtype)
    dims = ssd.dims_for(dev["x"], dev["B"], w.chunk)
    ws = torch.empty(ssd.ssd_fwd_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(dev["x"])
    fin = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def run():
        flush.fill_(1)
        ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["init_state"],
                    chunk_size=w.chunk, workspace=ws, out=y, final_out=fin)

    run()
    torch.cuda.synchronize()
    y0, f0 = y.clone(), fin.clone()
    differ = []
    for i in range(20):
        run()
        torch.cuda.synchronize()
        if not (torch.equal(y, y0) and torch.equal(fin, f0)):
            differ.append(i)
    assert ssd.ssd_take_device_errors() == 0
    assert not differ, f"calls {differ} differ from the first"


def test_workspace_contents_do_not_matter():
    """The workspace (and its fwd_pass_state control block) may hold anything
    on entry: fill it with 0xFF bytes, run twice through the same buffer, and
    compare with a fresh run and with the oracle.  Also the step entry point
    with a garbage scratch buffer."""
    w = small(seqlen=700, nheads=6, dtype="bf16", chunk=128, headdim=64, dstate=128,
              init_std=0.1, batch=2)
    inp = synth.make_inputs(w)
    dev = to_device(inp, "bf16")
    y_ref, f_ref = oracle_fwd(inp)
    dims = ssd.dims_for(dev["x"], dev["B"], 128)
    ws = torch.full((ssd.ssd_fwd_workspace_bytes(dims),), 0xFF, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        y, f = ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                           dev["init_state"], chunk_size=128, workspace=ws)
        torch.cuda.synchronize()
        outs.append((y.float().cpu().numpy(), f.cpu().numpy()))
    assert ssd.ssd_take_device_errors() == 0
    for y, f in outs:
        assert rel_err(y, y_ref) < TOL["bf16"] and rel_err(f, f_ref) < TOL["bf16"]
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    Gcs, dtT = ssd.ssd_chunk_cumsum(dev["dt"], dev["A"], chunk_size=128)
    scr = torch.full((int(ssd.load_library().ssd_fwd_pass_state_scratch_bytes(
        ctypes.byref(dims))),), 0xA5, dtype=torch.uint8, device="cuda")
    hid1, fin1 = ssd.ssd_fwd_pass_state(dev["x"], dev["B"], Gcs, dtT, dev["init_state"],
                                        chunk_size=128, scratch=scr)
    hid2, fin2 = ssd.ssd_fwd_pass_state(dev["x"], dev["B"], Gcs, dtT, dev["init_state"],
                                        chunk_size=128, scratch=scr)
    torch.cuda.synchronize()
    assert ssd.ssd_take_device_errors() == 0
    assert torch.equal(hid1, hid2) and torch.equal(fin1, fin2)
    assert np.array_equal(fin1.cpu().numpy(), outs[0][1])


def test_errors_are_raised():
    w = small(seqlen=100, dtype="bf16", chunk=64)
    dev = to_device(synth.make_inputs(w), "bf16")
    small_ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ssd.SSDError, match="SSD_ERR_WORKSPACE"):
        ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], workspace=small_ws,
                    chunk_size=64)
    with pytest.raises(ssd.SSDError, match="SSD_ERR_SHAPE"):
        ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], chunk_size=96)
    with pytest.raises(ssd.SSDError, match="SSD_ERR_ALIAS"):
        ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], chunk_size=64,
                    out=dev["x"])


@pytest.mark.parametrize("headdim", [64, 16])
def test_output_at_16_byte_offset(headdim):
    """y may start on any 16-byte boundary: an output 16 bytes past a 32-byte
    boundary (where the 32-byte row stores cannot be used) holds exactly the
    values of an aligned one."""
    w = small(seqlen=300, nheads=4, ngroups=2, headdim=headdim, dstate=128, chunk=128,
              dtype="bf16", batch=2)
    dev = to_device(synth.make_inputs(w), "bf16")
    y_ref, _ = ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                           chunk_size=128, return_final_state=False)
    n = dev["x"].numel()
    flat = torch.full((n + 16,), float("nan"), dtype=torch.bfloat16, device="cuda")
    y_off = flat[8:8 + n].view(dev["x"].shape)
    assert y_off.data_ptr() % 32 == 16
    ssd.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], chunk_size=128,
                return_final_state=False, out=y_off)
    torch.cuda.synchronize()
    assert torch.equal(y_off, y_ref)
    assert torch.isnan(flat[:8]).all() and torch.isnan(flat[8 + n:]).all()
