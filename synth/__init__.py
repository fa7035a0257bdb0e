"""Seeded synthetic inputs for the CSA/HCA hybrid compressed attention path.

This module is the one piece both sides share: the fp64 oracle (``oracle/``)
and the GPU tests / bench draw their inputs from here.  It holds no step of the
method's arithmetic -- only counter-based random draws, bit-level encodings of
the drawn values, and the workload shapes.

Counter-based generator (one definition, two implementations: this numpy one
and ``synth/gen.cu`` for on-device fills of very large raw-row tensors):

* ``mix64`` is the output function of SplitMix64 (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014).
* ``key(seed, tid) = mix64(seed * 2**32 + tid)``; draw ``i`` of a tensor is the
  ``i``-th output of SplitMix64 seeded with that key:
  ``draw(seed, tid, i) = mix64(key + (i + 1) * GAMMA)`` (all mod 2**64).
* N(0,1)-like values: the four 16-bit lanes of one draw are summed
  (Irwin-Hall), centred, multiplied in fp32 by ``NORMAL_SCALE`` (the fp32
  nearest to 1/sqrt((2**32-1)/3), the reciprocal standard deviation of the sum)
  and rounded to bf16, round-to-nearest-even.
* FP4 e2m1 codes are uniform over the 15 distinct finite values (the negative
  zero code 0x8 is never drawn); 2**e block scales with e uniform in {-1,0,1}
  are stored as UE8M0 bytes (biased exponent, bias 127); indexer head weights
  are uniform in {0.5, 1, 2}.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
NORMAL_SCALE_BITS = 0x37DDB3D7            # fp32(1/sqrt((2**32-1)/3))
NORMAL_SCALE = np.uint32(NORMAL_SCALE_BITS).view(np.float32)
INV_SQRT128_BITS = 0x3DB504F3             # fp32(1/sqrt(128))

# e2m1 codes in draw order: +0, +0.5 .. +6, -0.5 .. -6  (0x8 = -0 excluded)
E2M1_DRAW_CODES = np.array([0, 1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15], dtype=np.uint8)

# tensor kinds (the high byte of a tensor id)
RAW, QUERY, IDX_Q, IDX_QS, IDX_K, IDX_KS, HEAD_W, COMP_W, COMP_B, LENGTHS, COMP_SCORES = range(1, 12)


def tensor_id(kind: int, layer: int = 0, seq: int = 0) -> int:
    """Tensor id: kind in bits 24..31, layer in 16..23, sequence in 0..15."""
    assert 0 <= kind < 256 and 0 <= layer < 256 and 0 <= seq < 65536
    return (kind << 24) | (layer << 16) | seq


def mix64(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tid: int) -> np.uint64:
    return mix64(np.uint64(((seed & 0xFFFFFFFF) << 32) | (tid & 0xFFFFFFFF)))


def draws(seed: int, tid: int, start: int, n: int) -> np.ndarray:
    """uint64 draws ``start .. start+n-1`` of tensor ``tid``."""
    key = stream_key(seed, tid)
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(key + i * GAMMA)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round-to-nearest-even (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_f32(seed: int, tid: int, start: int, n: int) -> np.ndarray:
    """The fp32 value before the final bf16 rounding (exact Irwin-Hall sum x scale)."""
    u = draws(seed, tid, start, n)
    m = np.uint64(0xFFFF)
    s = (u & m).astype(np.int64) + ((u >> np.uint64(16)) & m).astype(np.int64) \
        + ((u >> np.uint64(32)) & m).astype(np.int64) + (u >> np.uint64(48)).astype(np.int64) - 131070
    return s.astype(np.float32) * NORMAL_SCALE


def normal_bf16(seed: int, tid: int, start: int, n: int, scale_bits: int | None = None) -> np.ndarray:
    """bf16 bit patterns of N(0,1)-like draws; optional fp32 multiplier (given by its bits)."""
    v = normal_f32(seed, tid, start, n)
    if scale_bits is not None:
        v = v * np.uint32(scale_bits).view(np.float32)
    return f32_to_bf16_bits(v)


def e2m1_codes(seed: int, tid: int, start: int, n: int) -> np.ndarray:
    return E2M1_DRAW_CODES[(draws(seed, tid, start, n) % np.uint64(15)).astype(np.int64)]


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Pack codes two per byte along the last axis: even element in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    assert c.shape[-1] % 2 == 0
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def ue8m0_scales(seed: int, tid: int, start: int, n: int, lo: int = -1, hi: int = 1) -> np.ndarray:
    span = hi - lo + 1
    e = (draws(seed, tid, start, n) % np.uint64(span)).astype(np.int64) + lo
    return (e + 127).astype(np.uint8)


def head_weights(seed: int, tid: int, start: int, n: int) -> np.ndarray:
    table = np.array([0.5, 1.0, 2.0], dtype=np.float32)
    return table[(draws(seed, tid, start, n) % np.uint64(3)).astype(np.int64)]


def uniform01(seed: int, tid: int, start: int, n: int) -> np.ndarray:
    """Uniform [0,1) doubles from the top 53 bits of a draw."""
    return (draws(seed, tid, start, n) >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))


# --------------------------------------------------------------------------------------
# Workloads.  Shapes follow the five synthetic workloads of the hot path; every
# tensor is a pure function of (seed, tensor id, element index).
# --------------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    kind: str               # "csa" | "hca" | "mixed"
    num_seqs: int
    ctx_len: int            # raw tokens cached before the new ones (per sequence)
    new_tokens: int         # new tokens (= queries) per sequence in the step
    heads: int              # query heads H
    dim: int                # shared KV dim D
    row_format: str         # "bf16" | "fp8_split"
    m: int                  # compression ratio
    overlap: bool
    index_heads: int = 4    # Hi
    index_rank: int = 128   # r
    top_k: int = 512
    window: int = 128
    block_scaled: bool = True
    softmax_scale: float = 1.0 / math.sqrt(512.0)
    layers: int = 1


CONFIGS = {
    "csa_tiny": Workload("csa_tiny_4096tok_h8_d128", seed=0, kind="csa", num_seqs=1, ctx_len=0,
                         new_tokens=4096, heads=8, dim=128, row_format="bf16", m=4, overlap=True,
                         index_heads=1, index_rank=64, top_k=64, block_scaled=False, softmax_scale=1.0),
    "csa_decode": Workload("csa_decode_32x128k_h64_d512", seed=1, kind="csa", num_seqs=32, ctx_len=131072,
                           new_tokens=1, heads=64, dim=512, row_format="fp8_split", m=4, overlap=True,
                           index_heads=4, index_rank=128, top_k=512),
    # the decode batch at a 1M-token context with the larger top-k (k = 1024 for the Pro model)
    "csa_decode_1m": Workload("csa_decode_32x1m_h64_d512_k1024", seed=1, kind="csa", num_seqs=32,
                              ctx_len=1048576, new_tokens=1, heads=64, dim=512, row_format="fp8_split", m=4,
                              overlap=True, index_heads=4, index_rank=128, top_k=1024),
    "csa_prefill": Workload("csa_prefill_1m_plus_16k_h128_d512", seed=2, kind="csa", num_seqs=1,
                            ctx_len=1048576, new_tokens=16384, heads=128, dim=512, row_format="fp8_split",
                            m=4, overlap=True, index_heads=4, index_rank=128, top_k=1024),
    "hca_decode": Workload("hca_decode_64x1m_h64_d512", seed=3, kind="hca", num_seqs=64, ctx_len=1048576,
                           new_tokens=1, heads=64, dim=512, row_format="fp8_split", m=128, overlap=False),
    "mixed_decode": Workload("mixed_ragged_decode_16seq_8layers", seed=4, kind="mixed", num_seqs=16,
                             ctx_len=-1, new_tokens=1, heads=64, dim=512, row_format="fp8_split", m=4,
                             overlap=True, index_heads=4, index_rank=128, top_k=1024, layers=8),
}


def mixed_lengths(seed: int, num_seqs: int, lo: int = 4096, hi: int = 1048576) -> np.ndarray:
    """Log-uniform sequence lengths floor(lo * (hi/lo)**U) for the ragged multi-layer workload."""
    u = uniform01(seed, tensor_id(LENGTHS), 0, num_seqs)
    return np.floor(lo * np.power(hi / lo, u)).astype(np.int64)
