"""Seeded synthetic inputs and the packed-weight layout writer.

This module is the one piece shared by the CUDA path's callers (tests, bench)
and by the checks of the CPU oracle: it draws random tensors and writes them in
the packed layout.  It holds none of the product arithmetic (no unpacking, no
dequantization, no dot products).

Layout (affine group quantization, 2 to 8 bits, BaseRT pages: thakicloud.com
"BaseRT는 무엇인가"; group size 64 along K -- 32 and 128 also supported -- fp16
scale and bias, Q4 codes 8 per uint32; and plain fp16 weights as "bits = 16",
the top of the pages' Q2..FP16 range):

* ``W`` is ``[N, K]`` with K contiguous (``nn.Linear`` convention).  Groups are
  ``g`` consecutive elements along K; ``G = K / g`` groups per row.
* ``codes`` is ``uint32 [N, K*b/32]``.  Each group is a group-local LSB-first
  bitstream of ``g`` b-bit codes in exactly ``g*b/32`` words: code ``j`` of the
  group occupies stream bits ``[j*b, j*b + b)``, and stream bit ``t`` is bit
  ``t % 32`` of the group's word ``t // 32``.  For b = 4 this is "8 codes per
  uint32", code j in bits ``[4*(j%8), +4)`` of word ``j//8``.  For b = 3 and 6
  a code may straddle two words.
* ``scales`` and ``biases`` are fp16 ``[N, G]``; the dequantized weight is
  ``w = scale * q + bias`` with ``q`` unsigned in ``[0, 2^b - 1]``.
* All arrays are row-major.

Quantizer (min/max per group, both parameters rounded to fp16 *before* the codes
are chosen, so dequantization uses exactly the stored values):

    s16 = fp16((hi - lo) / Qmax)     b16 = fp16(lo)
    q   = clamp(rint((w - b16) / s16), 0, Qmax)      (q = 0 where s16 == 0)

computed in fp32.  Inputs are ``w ~ N(0, 0.02)`` fp32 and activations ``x ~
N(0, 1)`` rounded to fp16 or bf16.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np

SUPPORTED_BITS = (2, 3, 4, 5, 6, 8)
FP16_BITS = 16            # "bits = 16": plain fp16 weights, no codes, scales or biases
GROUP_SIZE = 64
GROUP_SIZES = (32, 64, 128)


def seed_for(*parts) -> int:
    """Stable 64-bit seed for a tuple of labels (config, layer, proj, kind)."""
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little")


def rng_for(*parts) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed_for(*parts)))


# ---------------------------------------------------------------- half formats
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    out = ((u + r) >> 16).astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def draw_activations(r: np.random.Generator, m: int, k: int, dtype: str) -> np.ndarray:
    """x ~ N(0, 1) as uint16 bit patterns of ``dtype`` ('f16' or 'bf16'), shape [m, k]."""
    x = r.standard_normal((m, k), dtype=np.float32)
    if dtype == "f16":
        return f32_to_f16_bits(x)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


def draw_weights(r: np.random.Generator, n: int, k: int, sigma: float = 0.02) -> np.ndarray:
    return r.standard_normal((n, k), dtype=np.float32) * np.float32(sigma)


# -------------------------------------------------------------------- quantizer
def quantize(w: np.ndarray, bits: int, group_size: int = GROUP_SIZE):
    """Min/max affine quantization per group along K.

    Returns ``(q uint8 [N, K], scales fp16-bits uint16 [N, G], biases uint16 [N, G])``.
    """
    if bits not in SUPPORTED_BITS:
        raise ValueError(f"bits must be one of {SUPPORTED_BITS}")
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    if k % group_size:
        raise ValueError("K must be a multiple of the group size")
    qmax = np.float32(2**bits - 1)
    wg = w.reshape(n, k // group_size, group_size)
    lo = wg.min(axis=2)
    hi = wg.max(axis=2)
    s16 = ((hi - lo) / qmax).astype(np.float16)
    b16 = lo.astype(np.float16)
    s32 = s16.astype(np.float32)[:, :, None]
    b32 = b16.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (wg - b32) / s32
    t = np.where(s32 == 0, np.float32(0), t)
    q = np.clip(np.rint(t), 0, qmax).astype(np.uint8).reshape(n, k)
    return q, s16.view(np.uint16), b16.view(np.uint16)


# ----------------------------------------------------------------------- packer
def pack_codes(q: np.ndarray, bits: int, group_size: int = GROUP_SIZE) -> np.ndarray:
    """Write codes ``q [N, K]`` as group-local LSB-first bitstreams, uint32 [N, K*b/32]."""
    q = np.asarray(q)
    n, k = q.shape
    if (group_size * bits) % 32:
        raise ValueError("group_size * bits must be a multiple of 32")
    if np.any(q.astype(np.int64) >> bits):
        raise ValueError("code out of range")
    words_per_row = k * bits // 32
    out = np.empty((n, words_per_row), dtype=np.uint32)
    step = max(1, (1 << 22) // max(k, 1))
    shifts = np.arange(bits, dtype=np.uint8)
    for r0 in range(0, n, step):
        blk = q[r0:r0 + step].astype(np.uint8)
        # [rows, K, b] bits of each code, least significant first; a group's stream
        # is its codes' bits in order, so a row's concatenated streams are exactly this.
        stream = ((blk[:, :, None] >> shifts) & 1).astype(np.uint8)
        stream = stream.reshape(blk.shape[0], k * bits)
        by = np.packbits(stream, axis=1, bitorder="little")
        out[r0:r0 + step] = by.view("<u4").reshape(blk.shape[0], words_per_row)
    return out


@dataclass
class QuantWeight:
    """One packed weight matrix (host numpy arrays)."""
    codes: np.ndarray     # uint32 [N, K*b/32]
    scales: np.ndarray    # uint16 (fp16 bits) [N, G]
    biases: np.ndarray    # uint16 (fp16 bits) [N, G]
    bits: int
    n: int
    k: int
    group_size: int = GROUP_SIZE


def make_qweight(r: np.random.Generator, n: int, k: int, bits: int,
                 group_size: int = GROUP_SIZE, sigma: float = 0.02) -> QuantWeight:
    """Seeded weights in the packed layout.  ``bits = 16`` gives fp16 weights:
    weight k of a row is the fp16 bit pattern in bits [16*(k%2), +16) of word
    k/2 (the same LSB-first stream with 16-bit "codes"); the scales and biases
    are zero arrays of the usual shape, never read."""
    w = draw_weights(r, n, k, sigma)
    if bits == FP16_BITS:
        if k % group_size:
            raise ValueError("K must be a multiple of the group size")
        codes = np.ascontiguousarray(f32_to_f16_bits(w)).view("<u4").reshape(n, k // 2).astype(np.uint32)
        zeros = np.zeros((n, k // group_size), dtype=np.uint16)
        return QuantWeight(codes, zeros, zeros.copy(), bits, n, k, group_size)
    q, s, b = quantize(w, bits, group_size)
    return QuantWeight(pack_codes(q, bits, group_size), s, b, bits, n, k, group_size)


def grid_exact_weights(r: np.random.Generator, n: int, k: int, bits: int,
                       group_size: int = GROUP_SIZE):
    """Weights that lie exactly on a dyadic quantization grid.

    Per group: ``s = i * 2^-8`` (``i`` a small integer), ``beta = -s * 2^(b-1)``,
    codes uniform in ``[0, Qmax]`` with both 0 and Qmax present, ``w = s*q + beta``.
    Returns ``(w fp32 [N, K], q, s fp32 [N, G], beta fp32 [N, G])``.
    """
    qmax = 2**bits - 1
    g = k // group_size
    i = r.integers(1, 16, size=(n, g))
    s = (i * 2.0**-8).astype(np.float32)
    beta = (-s * 2.0 ** (bits - 1)).astype(np.float32)
    q = r.integers(0, qmax + 1, size=(n, g, group_size))
    q[:, :, 0] = 0
    q[:, :, 1] = qmax
    perm = r.permuted(np.broadcast_to(np.arange(group_size), (n, g, group_size)), axis=2)
    q = np.take_along_axis(q, perm, axis=2)
    w = (s[:, :, None] * q + beta[:, :, None]).astype(np.float32).reshape(n, k)
    return w, q.reshape(n, k).astype(np.uint8), s, beta


# ------------------------------------------------------------------ MoE routing
def draw_routing(r: np.random.Generator, tokens: int, num_experts: int, top_k: int):
    """Seeded top-k routing: distinct uniform expert ids per token and softmax gates.

    Returns ``(ids int32 [T, top_k], gates float32 [T, top_k])``; the gate logits are
    N(0, 1) and the gates are their softmax over the token's ``top_k`` slots.
    """
    ids = np.empty((tokens, top_k), dtype=np.int32)
    for t in range(tokens):
        ids[t] = r.permutation(num_experts)[:top_k]
    logits = r.standard_normal((tokens, top_k)).astype(np.float64)
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    gates = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, gates
