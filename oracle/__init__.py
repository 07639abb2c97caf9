"""CPU oracle for the Mamba-2 SSD forward pass -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it: the two meet only through the seeded input generator
(``state_space_sequence_chunk_gb300.synth``), which holds none of the method's
arithmetic.

The arithmetic lives in ``ssd_oracle.c`` (plain single-threaded fp64 C); this
module compiles it with gcc and exposes it to numpy through ctypes.

Functions (all fp64, all pinned by ``tests/test_oracle_pins.py``):

* :func:`recurrence` -- the token-by-token recurrence of "Accelerating Mamba-2
  with High-Performance Forward Pass Kernels in NVIDIA CUDA Tile", section
  "The Mamba-2 Recurrence" (formulas in the zhiding.cn rendering, section
  "Mamba-2架构"); optionally records the chunk-start states.
* :func:`chunk_cumsum` -- the in-chunk cumulative decay sums of section
  "Kernel 1: chunk_cumsum", base-2 scaled.
* :func:`chunked` -- the chunked closed form of section "Step 3: Add Back the
  Decay, Safely, in Log-Space"; used only to pin :func:`recurrence`.
* :func:`causal_conv1d` -- the depthwise causal convolution of the Helion
  hackathon gallery's "Causal Conv1d" entries (the Mamba-2 block's neighbour).
* :func:`gdn_fwd_h`, :func:`gdn_fwd_o` -- the Gated DeltaNet chunk kernels of
  the same gallery's "GDN chunk_fwd_h" / "GDN chunk_fwd_o" entries, step by step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle C source into a shared library; returns its path.

    Plain ``gcc -O2`` without fast-math, so that fp64 rounding follows IEEE.
    """
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
           *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _declare(lib):
    i64, dp = ctypes.c_int64, ctypes.c_void_p
    lib.ssd_oracle_recurrence.argtypes = [i64] * 6 + [dp] * 9 + [i64, dp]
    lib.ssd_oracle_recurrence.restype = ctypes.c_int
    lib.ssd_oracle_chunk_cumsum.argtypes = [i64] * 4 + [dp] * 3
    lib.ssd_oracle_chunk_cumsum.restype = ctypes.c_int
    lib.ssd_oracle_chunked.argtypes = [i64] * 7 + [dp] * 9
    lib.ssd_oracle_chunked.restype = ctypes.c_int
    lib.ssd_oracle_causal_conv1d.argtypes = [i64] * 4 + [dp] * 4
    lib.ssd_oracle_causal_conv1d.restype = ctypes.c_int
    lib.ssd_oracle_gdn_fwd_h.argtypes = [i64] * 6 + [dp] * 8
    lib.ssd_oracle_gdn_fwd_h.restype = ctypes.c_int
    lib.ssd_oracle_gdn_fwd_o.argtypes = [i64] * 6 + [dp] * 6
    lib.ssd_oracle_gdn_fwd_o.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; cached per process."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH) or (
                    os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
        return _lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def recurrence(x, dt, A, B, C, D=None, init_state=None, ckpt_every: int = 0, lib=None):
    """Run the fp64 recurrence.

    Shapes: x [b, L, H, P], dt [b, L, H], A [H], B and C [b, L, G, N],
    D [H] or None, init_state [b, H, P, N] or None.
    Returns ``(y, final_state)`` or, with ``ckpt_every > 0``,
    ``(y, final_state, ckpt)`` where ``ckpt[b, h, c]`` is the state held
    before token ``c * ckpt_every``.
    """
    lib = lib or load()
    x, dt, A, B, C, D, init_state = map(_f64, (x, dt, A, B, C, D, init_state))
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert dt.shape == (b, L, H) and A.shape == (H,)
    assert B.shape == (b, L, G, N) and C.shape == (b, L, G, N)
    y = np.zeros((b, L, H, P), np.float64)
    fin = np.zeros((b, H, P, N), np.float64)
    nck = (L + ckpt_every - 1) // ckpt_every if ckpt_every > 0 else 0
    ck = np.zeros((b, H, nck, P, N), np.float64) if nck > 0 else None
    rc = lib.ssd_oracle_recurrence(b, L, H, P, N, G, _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                   _ptr(C), _ptr(D), _ptr(init_state), _ptr(y), _ptr(fin),
                                   ckpt_every if nck > 0 else 0, _ptr(ck))
    if rc != 0:
        raise ValueError(f"ssd_oracle_recurrence failed with code {rc}")
    return (y, fin, ck) if ckpt_every > 0 else (y, fin)


def chunk_cumsum(dt, A, chunk: int, lib=None):
    """G[b, h, t] = log2(e) * (inclusive in-chunk sum of A[h] * dt[b, k, h]); [b, H, L]."""
    lib = lib or load()
    dt, A = _f64(dt), _f64(A)
    b, L, H = dt.shape
    G = np.zeros((b, H, L), np.float64)
    rc = lib.ssd_oracle_chunk_cumsum(b, L, H, chunk, _ptr(dt), _ptr(A), _ptr(G))
    if rc != 0:
        raise ValueError(f"ssd_oracle_chunk_cumsum failed with code {rc}")
    return G


def chunked(x, dt, A, B, C, D=None, init_state=None, chunk: int = 64, lib=None):
    """The chunked closed form (fp64); returns ``(y, final_state)``."""
    lib = lib or load()
    x, dt, A, B, C, D, init_state = map(_f64, (x, dt, A, B, C, D, init_state))
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros((b, L, H, P), np.float64)
    fin = np.zeros((b, H, P, N), np.float64)
    rc = lib.ssd_oracle_chunked(b, L, H, P, N, G, chunk, _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                _ptr(C), _ptr(D), _ptr(init_state), _ptr(y), _ptr(fin))
    if rc != 0:
        raise ValueError(f"ssd_oracle_chunked failed with code {rc}")
    return y, fin


def causal_conv1d(x, weight, bias=None, lib=None):
    """Depthwise causal conv1d (fp64): x [b, d, L], weight [d, W], bias [d] or None;
    returns out [b, d, L] (Helion hackathon gallery, "Causal Conv1d")."""
    lib = lib or load()
    x, weight, bias = _f64(x), _f64(weight), _f64(bias)
    b, d, L = x.shape
    W = weight.shape[1]
    assert weight.shape == (d, W) and (bias is None or bias.shape == (d,))
    out = np.zeros((b, d, L), np.float64)
    rc = lib.ssd_oracle_causal_conv1d(b, d, L, W, _ptr(x), _ptr(weight), _ptr(bias), _ptr(out))
    if rc != 0:
        raise ValueError(f"ssd_oracle_causal_conv1d failed with code {rc}")
    return out


def gdn_fwd_h(k, w, u, g, h0=None, chunk: int = 64, lib=None):
    """Gated DeltaNet chunk_fwd_h (fp64): k, w [B, T, H, K], u [B, T, H, V], g [B, T, H]
    (in-chunk inclusive cumulative log gate), h0 [B, H, K, V] or None.  Returns
    ``(h [B, H, NT, K, V], v_new [B, T, H, V], final_state [B, H, K, V])``."""
    lib = lib or load()
    k, w, u, g, h0 = map(_f64, (k, w, u, g, h0))
    B, T, H, K = k.shape
    V = u.shape[3]
    NT = -(-T // chunk)
    h = np.zeros((B, H, NT, K, V)); v_new = np.zeros((B, T, H, V)); fin = np.zeros((B, H, K, V))
    rc = lib.ssd_oracle_gdn_fwd_h(B, T, H, K, V, chunk, _ptr(k), _ptr(w), _ptr(u), _ptr(g), _ptr(h0),
                                  _ptr(h), _ptr(v_new), _ptr(fin))
    if rc != 0:
        raise ValueError(f"ssd_oracle_gdn_fwd_h failed with code {rc}")
    return h, v_new, fin


def gdn_fwd_o(q, k, v_new, h, g, chunk: int = 64, lib=None):
    """Gated DeltaNet chunk_fwd_o (fp64): returns o [B, T, H, V]."""
    lib = lib or load()
    q, k, v_new, h, g = map(_f64, (q, k, v_new, h, g))
    B, T, H, K = q.shape
    V = v_new.shape[3]
    o = np.zeros((B, T, H, V))
    rc = lib.ssd_oracle_gdn_fwd_o(B, T, H, K, V, chunk, _ptr(q), _ptr(k), _ptr(v_new), _ptr(h), _ptr(g),
                                  _ptr(o))
    if rc != 0:
        raise ValueError(f"ssd_oracle_gdn_fwd_o failed with code {rc}")
    return o
