"""Seeded synthetic inputs for the SSD forward pass.

This module is the ONE piece shared by the CUDA path's tests/benchmark and the
CPU oracle's tests: it draws the inputs, and nothing else.  It holds none of the
method's arithmetic (no decay, no cumulative sum, no state update).

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based generator:
draw ``i`` of a stream with key ``k`` is ``mix64(k + (i + 1) * 0x9E3779B97F4A7C15)``.
Each tensor has its own stream key, derived from the workload seed and a fixed
stream number.  Normal deviates use the Box-Muller transform on the two 32-bit
halves of one draw.

Workloads are the five synthetic shapes used throughout (the pages' benchmark
is itself synthetic: inputs of a problem spec, no dataset):

==================  =====  ======  ===  ===  ===  ===  =====  =====
name                batch  seqlen    H    P    N    G  chunk  dtype
==================  =====  ======  ===  ===  ===  ===  =====  =====
tiny_fp32               1     256    2   32   16    1     64  f32
small_fp32              2    2048    8   64   64    1     64  f32
mamba2_layer_bf16       4    4096   80   64  128    1    256  bf16
long_context_bf16       1   65536   24   64  128    1    256  bf16
short_streams_bf16    128     512   32   64  128    8    128  bf16
==================  =====  ======  ===  ===  ===  ===  =====  =====

Distributions: x, B, C ~ N(0, 1) (rounded to bf16, round-to-nearest-even, for
the bf16 workloads); dt = softplus(z) with z ~ N(mu, sigma) ((-3, 0.5), or
(-4, 1) for the long-context workload); A[h] = -exp(u), u ~ U[0, ln 16), so
A lies in [-16, -1); D[h] ~ N(0, 1); init_state = 0 or ~ N(0, 0.1^2).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BLOCK = 1 << 22

# stream numbers: one per tensor
STREAMS = {"x": 1, "B": 2, "C": 3, "dt": 4, "A": 5, "D": 6, "init": 7}


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (wrapping uint64 arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    """Key of stream ``stream`` under workload seed ``seed``."""
    with np.errstate(over="ignore"):
        k = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * np.uint64(0x100000001B3) \
            + np.uint64(stream) * GOLDEN
    return mix64(np.array([k], dtype=np.uint64))[0]


def raw64(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the stream with key ``key``."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + i * GOLDEN)


def normal(key: np.uint64, count: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """``count`` N(mean, std^2) deviates (float64), Box-Muller on one draw each."""
    out = np.empty(count, dtype=np.float64)
    for s in range(0, count, _BLOCK):
        n = min(_BLOCK, count - s)
        r = raw64(key, s, n)
        u1 = ((r >> np.uint64(32)).astype(np.float64) + 1.0) * (1.0 / 4294967296.0)
        u2 = (r & np.uint64(0xFFFFFFFF)).astype(np.float64) * (1.0 / 4294967296.0)
        out[s:s + n] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return mean + std * out


def uniform(key: np.uint64, count: int) -> np.ndarray:
    """``count`` U[0, 1) deviates (float64, 53-bit)."""
    r = raw64(key, 0, count)
    return (r >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    rounded = ((bits + bias) >> np.uint32(16)) << np.uint32(16)
    return rounded.astype(np.uint32).view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-representable."""
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return (bits >> np.uint32(16)).astype(np.uint16)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    dtype: str            # "f32" or "bf16": the dtype of x, B, C and y
    dt_mu: float = -3.0
    dt_sigma: float = 0.5
    init_std: float = 0.0  # 0 -> no initial state (zeros)
    with_D: bool = True
    seed: int = 20261202

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_fp32", 1, 256, 2, 32, 16, 1, 64, "f32", seed=20261202 + 0),
        Workload("small_fp32", 2, 2048, 8, 64, 64, 1, 64, "f32", init_std=0.1, seed=20261202 + 1),
        Workload("mamba2_layer_bf16", 4, 4096, 80, 64, 128, 1, 256, "bf16", seed=20261202 + 2),
        Workload("long_context_bf16", 1, 65536, 24, 64, 128, 1, 256, "bf16", dt_mu=-4.0,
                 dt_sigma=1.0, init_std=0.1, seed=20261202 + 3),
        Workload("short_streams_bf16", 128, 512, 32, 64, 128, 8, 128, "bf16", init_std=0.1,
                 seed=20261202 + 4),
    ]
}


# Context shape beside the five: the pages' own example problem ("Accelerating
# Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA CUDA Tile",
# section "Mamba-2 Forward Pass Benchmarks: cuTile vs Triton on NVIDIA B300":
# batch 4, 16384 tokens, 1 group, 8 heads, state 128, head 64, chunk 128, bf16
# with an fp32 state).  The page does not print how its sample inputs are
# drawn; they follow the recipe above, with a zero initial state.
CONTEXT_WORKLOADS = {
    "pages_example_bf16": Workload("pages_example_bf16", 4, 16384, 8, 64, 128, 1, 128, "bf16",
                                   seed=20261202 + 5),
}
# The same page's chart sweeps the state size: the example problem at state
# sizes 64 and 256 beside the 128 above (512 is outside this library's sizes).
for _n in (64, 256):
    CONTEXT_WORKLOADS[f"pages_example_n{_n}_bf16"] = Workload(
        f"pages_example_n{_n}_bf16", 4, 16384, 8, 64, _n, 1, 128, "bf16", seed=20261202 + 5)


def workload(name: str) -> Workload:
    """A workload of either table by name."""
    return WORKLOADS[name] if name in WORKLOADS else CONTEXT_WORKLOADS[name]


def make_inputs(w: Workload) -> dict:
    """Draw every input of workload ``w``.

    Returns float32 numpy arrays ``x [b,L,H,P]``, ``dt [b,L,H]``, ``A [H]``,
    ``B, C [b,L,G,N]``, ``D [H]`` (or None), ``init_state [b,H,P,N]`` (or
    None).  For bf16 workloads x, B and C already hold bf16-representable
    values, so the device and the oracle see identical numbers.
    """
    b, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    key = lambda s: stream_key(w.seed, STREAMS[s])
    x = normal(key("x"), b * L * H * P).astype(np.float32).reshape(b, L, H, P)
    Bm = normal(key("B"), b * L * G * N).astype(np.float32).reshape(b, L, G, N)
    Cm = normal(key("C"), b * L * G * N).astype(np.float32).reshape(b, L, G, N)
    if w.dtype == "bf16":
        x, Bm, Cm = round_to_bf16(x), round_to_bf16(Bm), round_to_bf16(Cm)
    z = normal(key("dt"), b * L * H, w.dt_mu, w.dt_sigma)
    dt = np.log1p(np.exp(z)).astype(np.float32).reshape(b, L, H)   # softplus
    A = (-np.exp(uniform(key("A"), H) * math.log(16.0))).astype(np.float32)
    D = normal(key("D"), H).astype(np.float32) if w.with_D else None
    init = None
    if w.init_std > 0:
        init = normal(key("init"), b * H * P * N, 0.0, w.init_std).astype(np.float32)
        init = init.reshape(b, H, P, N)
    return {"x": x, "dt": dt, "A": A, "B": Bm, "C": Cm, "D": D, "init_state": init}
