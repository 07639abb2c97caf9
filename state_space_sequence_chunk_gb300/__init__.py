"""GB300-native (sm_103a) Mamba-2 SSD chunked-scan forward pass.

A thin ctypes binding over the C ABI in ``include/ssd.h`` (``_lib/libssd.so``,
built in-tree by :mod:`state_space_sequence_chunk_gb300.build`).  The Python
side only marshals arguments: it allocates outputs and workspace with torch,
passes raw device pointers and torch's current CUDA stream, and turns status
codes into exceptions.  Every step of the computation runs in the library's
CUDA kernels; there is no CPU or PyTorch fallback -- if the library is missing,
the calls raise.

Entry points (same names as the C ABI):

* :func:`ssd_fwd` -- the whole forward pass, ``(y, final_state)``.
* :func:`ssd_chunk_cumsum`, :func:`ssd_fwd_pass_state`,
  :func:`ssd_compute_out` -- the three steps one at a time.
* :func:`ssd_fwd_workspace_bytes`, :func:`ssd_intermediate_bytes`.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libssd.so")

SSD_F32, SSD_BF16 = 0, 1
STATUS = {0: "SSD_OK", 1: "SSD_ERR_NULL", 2: "SSD_ERR_SHAPE", 3: "SSD_ERR_DTYPE",
          4: "SSD_ERR_ALIGN", 5: "SSD_ERR_WORKSPACE", 6: "SSD_ERR_ARCH", 7: "SSD_ERR_CUDA",
          8: "SSD_ERR_ALIAS", 9: "SSD_ERR_TIMEOUT"}
EXPORTS = ["ssd_abi_version", "ssd_status_string", "ssd_fwd_workspace_bytes",
           "ssd_intermediate_bytes", "ssd_fwd", "ssd_chunk_cumsum", "ssd_fwd_pass_state",
           "ssd_fwd_pass_state_scratch_bytes", "ssd_compute_out", "ssd_fwd_noalloc",
           "ssd_take_device_errors", "ssd_debug_withhold_handoffs", "ssd_step",
           "ssd_causal_conv1d", "ssd_gdn_chunk_fwd_h", "ssd_gdn_chunk_fwd_o",
           "ssd_fwd_host_staging_bytes", "ssd_fwd_host"]


class SSDError(RuntimeError):
    """A non-OK status returned by the library."""

    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS.get(code, code)}: {message}")
        self.code = code


class ConvDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("dim", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("width", ctypes.c_int64), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class GdnDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("kdim", ctypes.c_int64), ("vdim", ctypes.c_int64), ("chunk", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("nheads", ctypes.c_int64), ("headdim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("chunk_size", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libssd.so (cached).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library not found at {path}; build it with "
                "`python -m state_space_sequence_chunk_gb300.build` (or __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        vp, dp = ctypes.c_void_p, ctypes.POINTER(Dims)
        sz = ctypes.c_size_t
        lib.ssd_abi_version.argtypes, lib.ssd_abi_version.restype = [], ctypes.c_int
        lib.ssd_status_string.argtypes, lib.ssd_status_string.restype = [ctypes.c_int], ctypes.c_char_p
        lib.ssd_fwd_workspace_bytes.argtypes, lib.ssd_fwd_workspace_bytes.restype = [dp], sz
        lib.ssd_intermediate_bytes.argtypes = [dp, ctypes.POINTER(sz), ctypes.POINTER(sz)]
        lib.ssd_intermediate_bytes.restype = ctypes.c_int
        lib.ssd_fwd.argtypes = [dp] + [vp] * 10 + [sz, vp]
        lib.ssd_fwd.restype = ctypes.c_int
        lib.ssd_chunk_cumsum.argtypes = [dp] + [vp] * 5
        lib.ssd_chunk_cumsum.restype = ctypes.c_int
        lib.ssd_fwd_pass_state.argtypes = [dp] + [vp] * 8 + [sz, vp]
        lib.ssd_fwd_pass_state_scratch_bytes.argtypes = [dp]
        lib.ssd_fwd_pass_state_scratch_bytes.restype = sz
        lib.ssd_fwd_pass_state.restype = ctypes.c_int
        lib.ssd_compute_out.argtypes = [dp] + [vp] * 9
        lib.ssd_compute_out.restype = ctypes.c_int
        lib.ssd_debug_withhold_handoffs.argtypes = [ctypes.c_int]
        lib.ssd_debug_withhold_handoffs.restype = ctypes.c_int
        lib.ssd_take_device_errors.argtypes = []
        lib.ssd_take_device_errors.restype = ctypes.c_uint
        lib.ssd_fwd_noalloc.argtypes = [dp] + [vp] * 10
        lib.ssd_fwd_noalloc.restype = ctypes.c_int
        lib.ssd_step.argtypes = [dp] + [vp] * 9
        lib.ssd_step.restype = ctypes.c_int
        lib.ssd_causal_conv1d.argtypes = [ctypes.POINTER(ConvDims)] + [vp] * 5
        lib.ssd_causal_conv1d.restype = ctypes.c_int
        lib.ssd_gdn_chunk_fwd_h.argtypes = [ctypes.POINTER(GdnDims)] + [vp] * 9
        lib.ssd_gdn_chunk_fwd_h.restype = ctypes.c_int
        lib.ssd_gdn_chunk_fwd_o.argtypes = [ctypes.POINTER(GdnDims)] + [vp] * 7
        lib.ssd_gdn_chunk_fwd_o.restype = ctypes.c_int
        lib.ssd_fwd_host_staging_bytes.argtypes = [dp, ctypes.c_int]
        lib.ssd_fwd_host_staging_bytes.restype = sz
        lib.ssd_fwd_host.argtypes = [dp] + [vp] * 10 + [sz, ctypes.c_int, ctypes.POINTER(vp)]
        lib.ssd_fwd_host.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(code: int):
    if code != 0:
        msg = load_library().ssd_status_string(code).decode()
        raise SSDError(code, msg)


def dims_for(x: torch.Tensor, B: torch.Tensor, chunk_size: int) -> Dims:
    """ssd_dims for x [b, L, H, P] and B [b, L, G, N]."""
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [b, L, H, P] and B [b, L, G, N]")
    if x.dtype == torch.bfloat16:
        dt_code = SSD_BF16
    elif x.dtype == torch.float32:
        dt_code = SSD_F32
    else:
        raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    return Dims(b, L, H, P, N, G, int(chunk_size), dt_code, 0)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def ssd_take_device_errors() -> int:
    """Read and clear the kernels' device-side error bits (0 = no bounded wait
    ever gave up).  Synchronises the device."""
    return int(load_library().ssd_take_device_errors())


def ssd_debug_withhold_handoffs(on: bool) -> None:
    """Test hook for failure detection: with ``on``, fwd_pass_state launches skip
    their range hand-offs, so the receiving CTAs' bounded waits give up and the
    launch ends early with error bit 0 set (see ``ssd_take_device_errors``)."""
    _check(load_library().ssd_debug_withhold_handoffs(1 if on else 0))


def ssd_fwd_workspace_bytes(dims: Dims) -> int:
    return int(load_library().ssd_fwd_workspace_bytes(ctypes.byref(dims)))


def ssd_intermediate_bytes(dims: Dims):
    g, h = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load_library().ssd_intermediate_bytes(ctypes.byref(dims), ctypes.byref(g), ctypes.byref(h)))
    return g.value, h.value


def ssd_fwd(x, dt, A, B, C, D=None, init_state=None, chunk_size: int = 256,
            return_final_state: bool = True, workspace=None, out=None, final_out=None):
    """The whole SSD forward pass on x's device and torch's current stream.

    x [b, L, H, P] and B, C [b, L, G, N] share one dtype (float32 or bfloat16);
    dt [b, L, H], A [H], D [H], init_state [b, H, P, N] are float32.
    Returns ``(y, final_state)`` (final_state None unless requested).
    ``workspace`` (uint8 CUDA tensor), ``out`` and ``final_out`` may be given
    to reuse buffers.
    """
    lib = load_library()
    dims = dims_for(x, B, chunk_size)
    y = out if out is not None else torch.empty_like(x)
    fin = None
    if return_final_state:
        fin = final_out if final_out is not None else torch.empty(
            (x.shape[0], x.shape[2], x.shape[3], B.shape[3]), dtype=torch.float32, device=x.device)
    nbytes = int(lib.ssd_fwd_workspace_bytes(ctypes.byref(dims)))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    _check(lib.ssd_fwd(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                       _ptr(init_state), _ptr(y), _ptr(fin), _ptr(workspace),
                       ctypes.c_size_t(workspace.numel()), _stream()))
    return y, fin


def _host_ptr(t):
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous host (CPU) tensors")
    return ctypes.c_void_p(t.data_ptr())


_copy_streams = {}


def ssd_fwd_host_staging_bytes(dims: Dims, nslices: int) -> int:
    return int(load_library().ssd_fwd_host_staging_bytes(ctypes.byref(dims), int(nslices)))


def ssd_fwd_host(x, dt, A, B, C, D=None, init_state=None, chunk_size: int = 256,
                 return_final_state: bool = True, nslices: int = None, staging=None, out=None,
                 final_out=None, device=None):
    """ssd_fwd on HOST tensors (pinned, for the copies to overlap): the batch is
    cut into ``nslices`` slices whose host-device copies overlap the other
    slices' computation.  The compute runs on torch's current stream of
    ``device`` (default: the current CUDA device); two copy streams are kept
    per device.  Returns host tensors ``(y, final_state)``; they are complete
    once that stream has reached the end of the call (synchronise it before
    reading them).  ``staging`` (uint8 CUDA tensor) may be given to reuse it.
    """
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    dims = dims_for(x, B, chunk_size)
    b = x.shape[0]
    if nslices is None:
        nslices = max(1, min(b, 4))
    y = out if out is not None else torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    fin = None
    if return_final_state:
        fin = final_out if final_out is not None else torch.empty(
            (b, x.shape[2], x.shape[3], B.shape[3]), dtype=torch.float32, pin_memory=True)
    if b == 0:
        return y, fin
    nbytes = ssd_fwd_host_staging_bytes(dims, nslices)
    if staging is None:
        staging = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        if dev.index not in _copy_streams:
            _copy_streams[dev.index] = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
        s_in, s_out = _copy_streams[dev.index]
        streams = (ctypes.c_void_p * 3)(torch.cuda.current_stream(dev).cuda_stream,
                                        s_in.cuda_stream, s_out.cuda_stream)
        _check(lib.ssd_fwd_host(ctypes.byref(dims), _host_ptr(x), _host_ptr(dt), _host_ptr(A),
                                _host_ptr(B), _host_ptr(C), _host_ptr(D), _host_ptr(init_state),
                                _host_ptr(y), _host_ptr(fin), _ptr(staging),
                                ctypes.c_size_t(staging.numel()), int(nslices), streams))
    return y, fin


def ssd_chunk_cumsum(dt, A, chunk_size: int, x_dtype=torch.bfloat16):
    """Step 1: returns ``(Gcs, dtT)``, both [b, H, Lp] float32."""
    lib = load_library()
    b, L, H = dt.shape
    dims = Dims(b, L, H, 16, 16, 1, int(chunk_size),
                SSD_BF16 if x_dtype == torch.bfloat16 else SSD_F32, 0)
    nc = (L + chunk_size - 1) // chunk_size
    Gcs = torch.empty((b, H, nc * chunk_size), dtype=torch.float32, device=dt.device)
    dtT = torch.empty_like(Gcs)
    _check(lib.ssd_chunk_cumsum(ctypes.byref(dims), _ptr(dt), _ptr(A), _ptr(Gcs), _ptr(dtT),
                                _stream()))
    return Gcs, dtT


def ssd_fwd_pass_state(x, B, Gcs, dtT, init_state=None, chunk_size: int = 256,
                       return_final_state: bool = True, scratch=None):
    """Step 2: returns ``(hiddens [b, H, nc, N, P] in x.dtype, final_state)``;
    hiddens[b, h, c] is the chunk-start state transposed.  ``scratch`` (uint8
    device tensor of at least ssd_fwd_pass_state_scratch_bytes) is allocated
    here when not given."""
    lib = load_library()
    dims = dims_for(x, B, chunk_size)
    b, L, H, P = x.shape
    N = B.shape[3]
    nc = (L + chunk_size - 1) // chunk_size
    hid = torch.empty((b, H, nc, N, P), dtype=x.dtype, device=x.device)
    fin = torch.empty((b, H, P, N), dtype=torch.float32, device=x.device) if return_final_state else None
    need = int(lib.ssd_fwd_pass_state_scratch_bytes(ctypes.byref(dims)))
    if scratch is None and need > 0:
        scratch = torch.empty(need, dtype=torch.uint8, device=x.device)
    nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
    _check(lib.ssd_fwd_pass_state(ctypes.byref(dims), _ptr(x), _ptr(B), _ptr(Gcs), _ptr(dtT),
                                  _ptr(init_state), _ptr(hid), _ptr(fin), _ptr(scratch), nbytes,
                                  _stream()))
    return hid, fin


def ssd_compute_out(x, B, C, Gcs, dtT, hiddens, D=None, chunk_size: int = 256):
    """Step 3: returns y [b, L, H, P] in x.dtype."""
    lib = load_library()
    dims = dims_for(x, B, chunk_size)
    y = torch.empty_like(x)
    _check(lib.ssd_compute_out(ctypes.byref(dims), _ptr(x), _ptr(B), _ptr(C), _ptr(Gcs), _ptr(dtT),
                               _ptr(hiddens), _ptr(D), _ptr(y), _stream()))
    return y


def _gdn_dims(k, vdim, chunk, *tensors):
    if k.dim() != 4:
        raise ValueError("k must be a [B, T, H, K] tensor")
    for t in (k,) + tensors:
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"the Gated DeltaNet kernels take float32 tensors, got {t.dtype}")
    B, T, H, K = k.shape
    return GdnDims(B, T, H, K, vdim, int(chunk), SSD_F32, 0)


def gdn_chunk_fwd_h(k, w, u, g, h0=None, chunk: int = 64, return_final_state: bool = True):
    """Gated DeltaNet state recurrence over chunks: returns ``(h [B, H, NT, K, V],
    v_new [B, T, H, V], final_state [B, H, K, V] or None)``; all fp32."""
    lib = load_library()
    d = _gdn_dims(k, u.shape[3], chunk, w, u, g, h0)
    B, T, H, K = k.shape
    V = u.shape[3]
    NT = -(-T // chunk)
    h = torch.empty((B, H, NT, K, V), dtype=torch.float32, device=k.device)
    v_new = torch.empty_like(u)
    fin = torch.empty((B, H, K, V), dtype=torch.float32, device=k.device) if return_final_state else None
    _check(lib.ssd_gdn_chunk_fwd_h(ctypes.byref(d), _ptr(k), _ptr(w), _ptr(u), _ptr(g), _ptr(h0),
                                   _ptr(h), _ptr(v_new), _ptr(fin), _stream()))
    return h, v_new, fin


def gdn_chunk_fwd_o(q, k, v_new, h, g, chunk: int = 64):
    """Gated DeltaNet chunk outputs: returns o [B, T, H, V] (fp32)."""
    lib = load_library()
    d = _gdn_dims(k, v_new.shape[3], chunk, q, v_new, h, g)
    o = torch.empty_like(v_new)
    _check(lib.ssd_gdn_chunk_fwd_o(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v_new), _ptr(h), _ptr(g),
                                   _ptr(o), _stream()))
    return o


def causal_conv1d(x, weight, bias=None):
    """Depthwise causal conv1d: x [b, dim, L] (bf16 or fp32), weight [dim, W] fp32,
    bias [dim] fp32 or None; returns out [b, dim, L] in x.dtype."""
    lib = load_library()
    if x.dim() != 3 or weight.dim() != 2:
        raise ValueError("x must be [b, dim, L] and weight [dim, W]")
    code = SSD_BF16 if x.dtype == torch.bfloat16 else SSD_F32
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")
    b, dim, L = x.shape
    d = ConvDims(b, dim, L, weight.shape[1], code, 0)
    out = torch.empty_like(x)
    _check(lib.ssd_causal_conv1d(ctypes.byref(d), _ptr(x), _ptr(weight), _ptr(bias), _ptr(out),
                                 _stream()))
    return out


def ssd_step(x, dt, A, B, C, D, state):
    """Token-by-token recurrence over x's L tokens (decode): updates ``state``
    [b, H, P, N] fp32 in place and returns y [b, L, H, P] in x.dtype."""
    lib = load_library()
    dims = dims_for(x, B, 64)
    y = torch.empty_like(x)
    _check(lib.ssd_step(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                        _ptr(state), _ptr(y), _stream()))
    return y


def ssd_fwd_noalloc(x, dt, A, B, C, D=None, init_state=None, chunk_size: int = 256,
                    out=None, final_out=None):
    """ssd_fwd without a workspace argument, for callers that cannot allocate
    device memory: the library uses its own fixed 32 MiB device scratch array.

    The caller passes every input and output buffer (``out`` for y and, if the
    final state is wanted, ``final_out``); nothing is allocated here when both
    are given.  Problems needing more scratch than the fixed array raise
    SSD_ERR_WORKSPACE.  Calls on one device share the array, so calls that
    overlap on the GPU must be serialised by the caller.
    """
    lib = load_library()
    dims = dims_for(x, B, chunk_size)
    y = out if out is not None else torch.empty_like(x)
    _check(lib.ssd_fwd_noalloc(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                               _ptr(D), _ptr(init_state), _ptr(y), _ptr(final_out), _stream()))
    return y, final_out
