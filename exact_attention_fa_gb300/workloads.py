"""Seeded synthetic workloads: the only module shared by the CUDA path's tests and the oracle.

It holds no attention arithmetic. It only draws inputs (i.i.d. standard normal Q, K, V, dO and a
Bernoulli block mask) and rounds them to bf16, so that both sides of a parity test see exactly the
same input values.

Generator: numpy's PCG64 seeded with ``SeedSequence([seed, stream])`` (one stream per tensor), its
standard-normal sampler in float32, then round-to-nearest-even to bf16 by integer arithmetic on
the fp32 bit pattern. The shapes and distributions follow the workloads of the FlashAttention pages
(multi-head attention, ``[B, H, N, d]`` tensors, N(0, 1) entries, 128x128 tile block mask).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# One independent random stream per tensor so that, e.g., the mask never depends on d.
STREAM_Q, STREAM_K, STREAM_V, STREAM_DO, STREAM_MASK = 1, 2, 3, 4, 5

TILE = 128  # block-mask granularity (query tiles x key tiles)


def normal_f32(shape, seed: int, stream: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))
    return rng.standard_normal(size=shape, dtype=np.float32)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); returns the uint16 bit patterns.

    Inputs here are finite normals, so the NaN/overflow corner of the rounding never arises.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    u = u + np.uint32(0x7FFF) + lsb
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


# OCP 8-bit float E4M3 ("e4m3fn"): sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0
# holds the subnormals m/8 * 2^-6; the all-ones pattern S.1111.111 is NaN and there is no
# infinity, so the largest finite value is 1.75 * 2^8 = 448.
def _e4m3_table() -> np.ndarray:
    codes = np.arange(256)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e = (codes >> 3) & 0xF
    m = codes & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    vals = sign * mag
    vals[(codes & 0x7F) == 0x7F] = np.nan
    return vals


E4M3_VALUES = _e4m3_table()
E4M3_MAX = 448.0


def e4m3_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to even (the even code has a 0 last mantissa bit),
    saturating at +-448; returns the uint8 codes. Inputs must be finite."""
    x = np.asarray(x, dtype=np.float64)
    pos = E4M3_VALUES[:0x7F]  # codes 0x00 .. 0x7E: 0, the subnormals, the normals, ascending
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(pos, a, side="left"), 1, 0x7E)
    lo = hi - 1
    d_lo, d_hi = a - pos[lo], pos[hi] - a
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a >= pos[hi], hi, code)  # exact hits of the upper candidate
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)  # -0 keeps its sign


def e4m3_bits_from_f32_fast(x: np.ndarray) -> np.ndarray:
    """e4m3_bits_from_f32 by integer arithmetic on the fp32 bit patterns, for large inputs (the
    table search above is the definition; tests compare the two). Normal range: the 23-bit
    mantissa is rounded to 3 bits, ties to even, by adding 0x7FFFF plus the kept bit's lowest bit
    (a carry moves into the exponent, as it should); the exponent is rebiased from 127 to 7.
    Below 2^-6: the value in units of the subnormal spacing 2^-9, rounded half to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    sign = ((u >> np.uint32(24)) & np.uint32(0x80)).astype(np.uint8)
    a = u & np.uint32(0x7FFFFFFF)
    lsb = (a >> np.uint32(20)) & np.uint32(1)
    normal = ((a + np.uint32(0x7FFFF) + lsb) >> np.uint32(20)).astype(np.int64) - (120 << 3)
    sub = np.rint(np.abs(x).astype(np.float64) * 2.0 ** 9).astype(np.int64)  # rint: half to even
    code = np.where(a < np.uint32(0x3C800000), sub, normal)  # 0x3C800000 = 2^-6
    code = np.minimum(code, 0x7E).astype(np.uint8)            # saturate at 448
    return code | sign


def e4m3_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return E4M3_VALUES[np.asarray(bits, dtype=np.uint8)]


def block_mask(n_tiles: int, seed: int, p: float = 0.25) -> np.ndarray:
    """Bernoulli(p) tile mask [n_tiles, n_tiles] (row = query tile, column = key tile), diagonal on."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, STREAM_MASK])))
    m = (rng.random((n_tiles, n_tiles)) < p).astype(np.uint8)
    np.fill_diagonal(m, 1)
    return m


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, dtype, masking mode and seed."""

    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str = "bf16"  # "bf16", "fp32" or "e4m3" (Q, K, V, dO; O is bf16 for e4m3 inputs)
    causal: bool = False
    block_sparse: bool = False
    backward: bool = False
    seed: int = 0
    scale: float | None = None  # None means 1/sqrt(d)
    nq: int = 0  # decoding: query rows per head (keys and values keep N rows); 0: N queries

    @property
    def decode(self) -> bool:
        return self.nq > 0

    @property
    def n_queries(self) -> int:
        return self.nq if self.nq > 0 else self.N

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d) if self.scale is None else float(self.scale)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the hot path is specified on (seed = position in this list, 1-based).
WORKLOADS = {
    "single_head_fp32": Workload("single_head_fp32", 1, 1, 256, 64, dtype="fp32", seed=1),
    "mha_N2048_d64": Workload("mha_N2048_d64", 4, 16, 2048, 64, seed=2),
    "causal_N8192_d128": Workload("causal_N8192_d128", 8, 32, 8192, 128, causal=True, seed=3),
    "blocksparse_N16384_d64": Workload("blocksparse_N16384_d64", 2, 16, 16384, 64,
                                       block_sparse=True, seed=4),
    "bwd_causal_N4096_d128": Workload("bwd_causal_N4096_d128", 4, 16, 4096, 128, causal=True,
                                      backward=True, seed=5),
    # decoding ("3 · FlashAttention", 3.6): one new query row per head against a 32k-key cache
    "decode_N32768_d128": Workload("decode_N32768_d128", 8, 32, 32768, 128, nq=1, seed=6),
    # the same per-head problem on 8 heads (134 MB of K, V: larger than L2, small enough for ncu)
    "decode_N32768_d128_h8": Workload("decode_N32768_d128_h8", 1, 8, 32768, 128, nq=1, seed=7),
    # the same at d = 64 (256-key blocks), and its profile case on 16 heads (134 MB of K, V)
    "decode_N32768_d64": Workload("decode_N32768_d64", 8, 32, 32768, 64, nq=1, seed=8),
    "decode_N32768_d64_h16": Workload("decode_N32768_d64_h16", 1, 16, 32768, 64, nq=1, seed=9),
    # the long-sequence causal forward's per-head problem on 8 heads, at N = 8192 and N = 4096
    # (a device footprint small enough for counter captures; DRAM bytes should grow with N)
    "causal_N8192_d128_h8": Workload("causal_N8192_d128_h8", 1, 8, 8192, 128, causal=True,
                                     seed=10),
    "causal_N4096_d128_h8": Workload("causal_N4096_d128_h8", 1, 8, 4096, 128, causal=True,
                                     seed=11),
}

# The long-sequence causal problem with e4m3 inputs (the FP8 forward; O bf16).
WORKLOADS["causal_N8192_d128_fp8"] = Workload("causal_N8192_d128_fp8", 8, 32, 8192, 128,
                                              dtype="e4m3", causal=True, seed=12)

# Decoding with 8 new query rows per head (the tensor-core decoding path), same cache sizes.
WORKLOADS["decode_N32768_d128_q8"] = Workload("decode_N32768_d128_q8", 8, 32, 32768, 128, nq=8,
                                              seed=15)
WORKLOADS["decode_N32768_d64_q8"] = Workload("decode_N32768_d64_q8", 8, 32, 32768, 64, nq=8,
                                             seed=16)

# The eight-row decoding problem on 2 x 32 heads (K, V 1.07 GB: larger than L2), measured on the
# default bench line.
WORKLOADS["decode_N32768_d128_q8_b2"] = Workload("decode_N32768_d128_q8_b2", 2, 32, 32768, 128,
                                                 nq=8, seed=17)

# Decoding with serving-sized caches: one new row per head against 4096 cached keys, for a
# batch of 8 (K, V 537 MB) and of 1 (67 MB: launch and ramp weigh most).
WORKLOADS["decode_N4096_d128"] = Workload("decode_N4096_d128", 8, 32, 4096, 128, nq=1, seed=18)
WORKLOADS["decode_N4096_d128_b1"] = Workload("decode_N4096_d128_b1", 1, 32, 4096, 128, nq=1,
                                             seed=19)

# Counter-capture cases of the e4m3 forward and of the backward on 8 heads (small device footprint).
WORKLOADS["causal_N4096_d128_fp8_h8"] = Workload("causal_N4096_d128_fp8_h8", 1, 8, 4096, 128,
                                                 dtype="e4m3", causal=True, seed=13)
WORKLOADS["bwd_causal_N4096_d128_h8"] = Workload("bwd_causal_N4096_d128_h8", 1, 8, 4096, 128,
                                                 causal=True, backward=True, seed=14)

# The five specified workloads in their order (the seed of each is its position).
SPECIFIED = ["single_head_fp32", "mha_N2048_d64", "causal_N8192_d128", "blocksparse_N16384_d64",
             "bwd_causal_N4096_d128"]


@dataclasses.dataclass
class Inputs:
    """Host-side inputs of one workload.

    ``*_bits`` are uint16 bf16 bit patterns (bf16 workloads) and ``*_f32`` the fp32 arrays
    (fp32 workloads); ``f64(name)`` returns the exact values as float64 for the oracle.
    """

    w: Workload
    arrays: dict

    def _decode(self, name: str, a: np.ndarray) -> np.ndarray:
        if a.dtype == np.uint16:
            return bf16_bits_to_f64(a)
        if a.dtype == np.uint8 and name != "mask":
            return e4m3_bits_to_f64(a)
        return a.astype(np.float64)

    def f64(self, name: str) -> np.ndarray:
        return self._decode(name, self.arrays[name])

    def f64_head(self, name: str, b: int, h: int) -> np.ndarray:
        """f64(name)[b, h] without converting the whole tensor."""
        return self._decode(name, self.arrays[name][b, h])

    def raw(self, name: str) -> np.ndarray:
        return self.arrays[name]


def make_inputs(w: Workload, with_do: bool | None = None) -> Inputs:
    shape = (w.B, w.H, w.N, w.d)
    qshape = (w.B, w.H, w.n_queries, w.d)
    names = [("q", STREAM_Q), ("k", STREAM_K), ("v", STREAM_V)]
    if with_do or (with_do is None and w.backward):
        names.append(("do", STREAM_DO))
    arrays = {}
    for nm, st in names:
        x = normal_f32(qshape if nm in ("q", "do") else shape, w.seed, st)
        if w.dtype == "bf16":
            arrays[nm] = bf16_bits_from_f32(x)
        elif w.dtype == "e4m3":
            arrays[nm] = e4m3_bits_from_f32_fast(x)
        else:
            arrays[nm] = x
        del x
    if w.block_sparse:
        arrays["mask"] = block_mask(-(-w.N // TILE), w.seed)
    return Inputs(w, arrays)


def flop_count(w: Workload, mask: np.ndarray | None = None, part: str = "fwd") -> float:
    """Algorithmic FLOPs: 4*B*H*N^2*d forward (causal: half; block-sparse: active tiles only,
    causal block-sparse: active tiles below the diagonal plus half of the active diagonal ones);
    the backward counts its five contractions, 2.5 times the forward. Block-sparse counts whole
    tiles, so they need N to be a multiple of 128. Decoding: 4*B*H*nq*N*d."""
    if w.decode:
        fwd = 4.0 * w.B * w.H * w.nq * w.N * w.d
    elif w.block_sparse:
        if w.N % TILE:
            raise ValueError("block-sparse FLOP counts need N to be a multiple of 128")
        if mask is None:
            mask = block_mask(w.N // TILE, w.seed)
        if w.causal:
            tiles = float(np.tril(mask, -1).sum()) + 0.5 * float(np.trace(mask))
        else:
            tiles = float(mask.sum())
        fwd = 4.0 * w.B * w.H * w.d * TILE * TILE * tiles
    else:
        fwd = 4.0 * w.B * w.H * w.N * w.N * w.d * (0.5 if w.causal else 1.0)
    if part == "fwd":
        return fwd
    if part == "bwd":
        return 2.5 * fwd
    if part == "fwd+bwd":
        return 3.5 * fwd
    raise ValueError(part)


def decode_bytes(w: Workload) -> float:
    """Algorithmic HBM bytes of one decoding pass: K and V read once, q read, O and lse written."""
    return float(w.B * w.H * (2 * w.N * w.d * 2 + 2 * w.nq * w.d * 2 + 4 * w.nq))
