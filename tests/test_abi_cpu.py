"""The C ABI on the host: the library loads, exports every entry point that
include/*.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import glob
import os
import re

import pytest

import state_space_sequence_chunk_gb300 as ssd
from state_space_sequence_chunk_gb300 import build as ssd_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ssd_build.build()
    return ssd.load_library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(ssd_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_binding_exports():
    assert set(ssd.EXPORTS) <= set(declared_functions())


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert lib.ssd_abi_version() == 5
    for code in range(0, 10):
        s = lib.ssd_status_string(code)
        assert s and s != b"unknown status"
    assert lib.ssd_status_string(99) == b"unknown status"


def dims(**kw):
    base = dict(batch=2, seqlen=300, nheads=4, headdim=64, dstate=128, ngroups=2,
                chunk_size=128, dtype=ssd.SSD_BF16, reserved=0)
    base.update(kw)
    return ssd.Dims(*[base[k] for k, _ in ssd.Dims._fields_])


def test_workspace_bytes(lib):
    d = dims()
    nc = 3
    gcs = 2 * 4 * nc * 128 * 4
    hid = 2 * 4 * nc * 64 * 128 * 2
    ru = lambda v: (v + 255) // 256 * 256
    # fwd_pass_state scratch (bf16): a two-slot fp32 state ring of 128 rows x 64
    # (P padded) per (batch, head, 128-row block of N), then 32 + chains words
    chains = 2 * 4 * 1
    scratch = ru(chains * 2 * 128 * 64 * 4) + ru((32 + chains) * 4)
    assert lib.ssd_fwd_pass_state_scratch_bytes(ctypes.byref(d)) == scratch
    assert ssd.ssd_fwd_workspace_bytes(d) == 2 * ru(gcs) + ru(hid) + scratch
    assert ssd.ssd_intermediate_bytes(d) == (gcs, hid)
    d32 = dims(dtype=ssd.SSD_F32)
    assert lib.ssd_fwd_pass_state_scratch_bytes(ctypes.byref(d32)) == 0
    assert ssd.ssd_fwd_workspace_bytes(d32) == 2 * ru(gcs) + ru(2 * hid)
    d2 = dims(dstate=256, headdim=96)   # two row blocks per head, P padded to 128
    chains2 = 2 * 4 * 2
    assert lib.ssd_fwd_pass_state_scratch_bytes(ctypes.byref(d2)) == (
        ru(chains2 * 2 * 128 * 128 * 4) + ru((32 + chains2) * 4))
    # long chains (nc >= 64, either kernel): + 1024 aggregate slots (fp32 states
    # of 128 x 64: four per range of the paired kernel, two per range of the
    # one-head kernel) and their log2 decay sums
    dl = dims(seqlen=64 * 128)
    chains_l = 2 * 4
    agg = ru(1024 * 128 * 64 * 4) + ru(1024 * 4)
    assert lib.ssd_fwd_pass_state_scratch_bytes(ctypes.byref(dl)) == (
        ru(chains_l * 2 * 128 * 64 * 4) + ru((32 + chains_l) * 4) + agg)
    dodd = dims(seqlen=64 * 128, ngroups=4)   # one head per group: the one-head kernel
    assert lib.ssd_fwd_pass_state_scratch_bytes(ctypes.byref(dodd)) == (
        ru(chains_l * 2 * 128 * 64 * 4) + ru((32 + chains_l) * 4) + agg)
    dshort = dims(seqlen=63 * 128, ngroups=4)   # 63 chunks: no two-pass form
    assert lib.ssd_fwd_pass_state_scratch_bytes(ctypes.byref(dshort)) == (
        ru(chains_l * 2 * 128 * 64 * 4) + ru((32 + chains_l) * 4))
    # the largest head and state sizes are accepted (P, N up to 256)
    assert ssd.ssd_fwd_workspace_bytes(dims(headdim=256, dstate=256)) > 0
    assert ssd.ssd_fwd_workspace_bytes(dims(seqlen=0)) == 0
    assert ssd.ssd_fwd_workspace_bytes(dims(chunk_size=100)) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(chunk_size=96), 2), (dict(headdim=40), 2), (dict(headdim=272), 2),
    (dict(dstate=8), 2), (dict(dstate=272), 2), (dict(ngroups=3), 2), (dict(nheads=0), 2),
    (dict(batch=-1), 2), (dict(dtype=5), 3), (dict(reserved=1), 2)])
def test_bad_shapes_rejected(lib, kw, code):
    d = dims(**kw)
    P = ctypes.c_void_p
    a = [P(0x100000 * (i + 1)) for i in range(10)]
    rc = lib.ssd_fwd(ctypes.byref(d), *a, ctypes.c_size_t(1 << 40), None)
    assert rc == code


def _fwd_args(n=10):
    # distinct, 16-byte aligned, far-apart fake device addresses (never dereferenced:
    # every call below fails validation before anything is enqueued)
    return [ctypes.c_void_p(0x10000000000 * (i + 1)) for i in range(n)]


def test_null_misaligned_alias_workspace(lib):
    d = dims()
    big = ctypes.c_size_t(1 << 40)
    a = _fwd_args()
    # x, dt, A, B, C, D, init, y, final, workspace
    null_x = list(a); null_x[0] = None
    assert lib.ssd_fwd(ctypes.byref(d), *null_x, big, None) == 1
    null_ws = list(a); null_ws[9] = None
    assert lib.ssd_fwd(ctypes.byref(d), *null_ws, big, None) == 1
    mis = list(a); mis[3] = ctypes.c_void_p(a[3].value + 8)
    assert lib.ssd_fwd(ctypes.byref(d), *mis, big, None) == 4
    assert lib.ssd_fwd(ctypes.byref(d), *a, ctypes.c_size_t(100), None) == 5
    alias = list(a); alias[7] = ctypes.c_void_p(a[0].value + 4096)   # y inside x
    assert lib.ssd_fwd(ctypes.byref(d), *alias, big, None) == 8
    alias = list(a); alias[9] = ctypes.c_void_p(a[4].value + 256)    # workspace inside C
    assert lib.ssd_fwd(ctypes.byref(d), *alias, big, None) == 8
    # D and init_state are optional: NULL passes validation and only fails at the
    # device check (no GPU here) -- never with a validation code
    opt = list(a); opt[5] = None; opt[6] = None; opt[8] = None
    rc = lib.ssd_fwd(ctypes.byref(d), *opt, big, None)
    assert rc in (0, 6, 7)


def test_per_step_validation(lib):
    d = dims()
    a = _fwd_args()
    assert lib.ssd_chunk_cumsum(ctypes.byref(d), a[0], None, a[2], a[3], None) == 1
    assert lib.ssd_chunk_cumsum(ctypes.byref(d), a[0], a[1], a[2], a[2], None) == 8
    big = ctypes.c_size_t(1 << 40)
    fps = lambda *args: lib.ssd_fwd_pass_state(ctypes.byref(d), *args)
    assert fps(a[0], a[1], a[2], a[3], a[4], None, a[6], a[7], big, None) == 1
    hid_in_x = ctypes.c_void_p(a[0].value + 1024)
    assert fps(a[0], a[1], a[2], a[3], a[4], hid_in_x, a[6], a[7], big, None) == 8
    # the bf16 path needs its scratch: NULL, too small, misaligned, overlapping
    assert fps(a[0], a[1], a[2], a[3], a[4], a[5], a[6], None, big, None) == 1
    assert fps(a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7], ctypes.c_size_t(64), None) == 5
    assert fps(a[0], a[1], a[2], a[3], a[4], a[5], a[6], ctypes.c_void_p(a[7].value + 4), big,
               None) == 4
    assert fps(a[0], a[1], a[2], a[3], a[4], a[5], a[6], ctypes.c_void_p(a[1].value + 512), big,
               None) == 8
    assert lib.ssd_compute_out(ctypes.byref(d), a[0], a[1], a[2], a[3], a[4], a[5], None,
                               ctypes.c_void_p(a[0].value), None) == 8


def test_step_validation(lib):
    # ssd_step(d, x, dt, A, B, C, D, state, y, stream); chunk_size is not used
    a = _fwd_args()
    step = lambda d, *args: lib.ssd_step(ctypes.byref(d), *args, None)
    d = dims(seqlen=2, chunk_size=100)
    assert step(d, None, a[1], a[2], a[3], a[4], a[5], a[6], a[7]) == 1
    assert step(d, a[0], a[1], a[2], a[3], a[4], a[5], None, a[7]) == 1   # state required
    assert step(d, a[0], a[1], a[2], a[3], a[4], a[5], a[6], None) == 1   # y required
    assert step(d, a[0], a[1], a[2], ctypes.c_void_p(a[3].value + 8), a[4], a[5], a[6],
                a[7]) == 4
    assert step(d, a[0], a[1], a[2], a[3], a[4], a[5], a[6],
                ctypes.c_void_p(a[0].value + 64)) == 8                      # y inside x
    assert step(d, a[0], a[1], a[2], a[3], a[4], a[5], ctypes.c_void_p(a[4].value + 256),
                a[7]) == 8                                                  # state inside C
    assert step(dims(seqlen=2, headdim=40), *a[:8]) == 2
    assert step(dims(seqlen=0), *a[:8]) == 0                                # nothing to do
    # D is optional: NULL passes validation and fails only at the device check
    assert step(d, a[0], a[1], a[2], a[3], a[4], None, a[6], a[7]) in (0, 6, 7)


def test_conv1d_validation(lib):
    a = _fwd_args(4)
    conv = lambda d, *args: lib.ssd_causal_conv1d(ctypes.byref(d), *args, None)
    cd = lambda **kw: ssd.ConvDims(*[dict(batch=2, dim=8, seqlen=64, width=4, dtype=ssd.SSD_BF16,
                                            reserved=0, **{})[k] if k not in kw else kw[k]
                                       for k, _ in ssd.ConvDims._fields_])
    assert conv(cd(width=0), *a) == 2
    assert conv(cd(width=9), *a) == 2
    assert conv(cd(dim=0), *a) == 2
    assert conv(cd(dtype=7), *a) == 3
    assert conv(cd(reserved=1), *a) == 2
    assert conv(cd(), None, a[1], a[2], a[3]) == 1
    assert conv(cd(), a[0], None, a[2], a[3]) == 1
    assert conv(cd(), a[0], a[1], a[2], ctypes.c_void_p(a[3].value + 4)) == 4
    assert conv(cd(), a[0], a[1], a[2], ctypes.c_void_p(a[0].value + 256)) == 8   # out inside x
    assert conv(cd(seqlen=0), *a) == 0
    # bias is optional: NULL passes validation and fails only at the device check
    assert conv(cd(), a[0], a[1], None, a[3]) in (0, 6, 7)


def test_gdn_validation(lib):
    a = _fwd_args(9)
    gd = lambda **kw: ssd.GdnDims(*[dict(batch=1, seqlen=128, nheads=2, kdim=64, vdim=64, chunk=64,
                                          dtype=ssd.SSD_F32, reserved=0)[k] if k not in kw else kw[k]
                                     for k, _ in ssd.GdnDims._fields_])
    fh = lambda d, *args: lib.ssd_gdn_chunk_fwd_h(ctypes.byref(d), *args, None)
    fo = lambda d, *args: lib.ssd_gdn_chunk_fwd_o(ctypes.byref(d), *args, None)
    assert fh(gd(dtype=ssd.SSD_BF16), *a[:8]) == 3
    assert fh(gd(chunk=48), *a[:8]) == 2
    assert fh(gd(kdim=129), *a[:8]) == 2
    assert fh(gd(), None, *a[1:8]) == 1
    assert fh(gd(), *a[:5], ctypes.c_void_p(a[0].value + 64), *a[6:8]) == 8   # h inside k
    assert fh(gd(), *a[:2], ctypes.c_void_p(a[2].value + 4), *a[3:8]) == 4
    assert fo(gd(), *a[:5], ctypes.c_void_p(a[2].value)) == 8                  # o over v_new
    assert fo(gd(), None, *a[1:6]) == 1
    assert fo(gd(batch=0), *a[:6]) == 0


def test_binding_raises_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="CUDA library not found"):
        saved = ssd._lib
        ssd._lib = None
        try:
            ssd.load_library(str(tmp_path / "nope.so"))
        finally:
            ssd._lib = saved


def test_fwd_host_validation(lib):
    """ssd_fwd_host rejects bad slices, buffers and overlaps before anything is
    enqueued (host pointers here are fake and never dereferenced)."""
    d = dims()
    b = d.batch
    a = _fwd_args(10)
    streams = (ctypes.c_void_p * 3)(None, None, None)
    need = lib.ssd_fwd_host_staging_bytes(ctypes.byref(d), min(b, 2))
    assert need > 0
    assert lib.ssd_fwd_host_staging_bytes(ctypes.byref(d), 0) == 0
    assert lib.ssd_fwd_host_staging_bytes(ctypes.byref(d), b + 1) == 0
    assert lib.ssd_fwd_host_staging_bytes(ctypes.byref(d), 65) == 0
    args = a[:9] + [a[9], ctypes.c_size_t(need)]
    host = lambda *v: lib.ssd_fwd_host(ctypes.byref(d), *v)
    assert host(*args, 0, streams) == 2                     # nslices < 1
    assert host(*args, b + 1, streams) == 2                 # more slices than batch elements
    assert host(*args, 1, None) == 1                        # no streams
    small = a[:9] + [a[9], ctypes.c_size_t(need - 1)]
    assert host(*small, min(b, 2), streams) == 5            # staging too small
    odd = a[:9] + [ctypes.c_void_p(a[9].value + 16), ctypes.c_size_t(need)]
    assert host(*odd, min(b, 2), streams) == 4              # staging not 256-byte aligned
    over = list(args); over[7] = ctypes.c_void_p(a[0].value + 64)   # y inside x
    assert host(*over, min(b, 2), streams) == 8
    # the last slice may hold fewer batch elements: its workspace fits the slot's
    for L in (300, 64 * 128):          # single pass, and a two-pass candidate
        for bb in range(1, 9):
            for nb in range(1, bb):
                lo, hi = dims(seqlen=L), dims(seqlen=L)
                lo.batch, hi.batch = nb, bb
                assert lib.ssd_fwd_workspace_bytes(ctypes.byref(lo)) <= \
                    lib.ssd_fwd_workspace_bytes(ctypes.byref(hi))
