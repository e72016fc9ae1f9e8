"""fp64 CPU oracle for affine group-quantized GEMV / GEMM / grouped-expert GEMM.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this module.  The library's
product path never calls it, and it shares no code with the CUDA path: it has
its own bit-level unpacker, its own half-float decoding and its own arithmetic.

What it computes is the plain definition, in fp64, of the products described on
the BaseRT pages:

* affine codes of 2 to 8 bits (thakicloud.com, "Apple Silicon 로컬 LLM 추론의
  새 기준 BaseRT", section "BaseRT는 무엇인가"): a weight is ``s*q + b`` with an
  unsigned code ``q`` and a per-group fp16 scale ``s`` and bias ``b``, groups of
  32, 64 or 128 along K; and plain fp16 weights (``bits = 16``), the top of the
  Q2..FP16 range (gist.science summary, "Metodologia");
* a GEMV for decode (M = 1) and a GEMM for prefill (M > 1), each expanding the
  codes in its inner loop (thetesserapress.com, "BaseRT claims fastest Apple
  Silicon inference", section "What BaseRT does differently"): both reduce to
  ``y[m, n] = sum_k x[m, k] * w_deq[n, k]``.  The oracle materializes ``w_deq``;
  the GPU path must not;
* grouped mixture-of-experts products (same page, section "Where the wins land,
  and where they don't"): the same product per expert over that expert's rows.

The exact result (up to rounding order) has a plain definition, so the oracle is
that definition written out: unpack, dequantize with exactly widened fp16
parameters, accumulate in fp64.  ``A = sum_k |x * w_deq|`` is the per-element
scale of the pass criterion ``|y - y_ref| <= rtol * A + atol``.

Pins (tests marked ``not gpu``): brute-force exact rational evaluation on tiny
inputs, codes in range, one-hot columns, grid-exact round trips, closed forms,
cross-check against numpy.matmul, and hand-written layout fixtures.
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------- half floats
def decode_f16(bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns (uint16) -> exact fp64 values."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values (bf16 is the top half of fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def decode_half(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return decode_f16(bits)
    if dtype == "bf16":
        return decode_bf16(bits)
    raise ValueError(dtype)


# ----------------------------------------------------------------- the layout
def unpack_codes(codes: np.ndarray, bits: int, k: int, group_size: int = 64) -> np.ndarray:
    """Read b-bit codes from group-local LSB-first bitstreams.

    ``codes`` is uint32 ``[N, K*b/32]``.  Each group of ``group_size`` codes is a
    stream of ``group_size*b`` bits held in consecutive words; stream bit ``t`` is
    bit ``t % 32`` of word ``t // 32``; code ``j`` is stream bits ``[j*b, (j+1)*b)``
    read least significant first.  Returns int64 ``[N, K]``.
    """
    codes = np.ascontiguousarray(codes, dtype=np.uint32)
    n = codes.shape[0]
    assert codes.shape[1] * 32 == k * bits, "codes row length does not match K and bits"
    assert (group_size * bits) % 32 == 0
    # Words are little-endian; split into bytes, then bytes into bits LSB first.
    as_bytes = codes.astype("<u4").view(np.uint8).reshape(n, -1)
    stream = np.unpackbits(as_bytes, axis=1, bitorder="little")      # [N, K*b]
    per_code = stream.reshape(n, k, bits).astype(np.int64)            # bit i of code at [.., i]
    weights = np.int64(1) << np.arange(bits, dtype=np.int64)
    return per_code @ weights


def dequantize(q: np.ndarray, scales: np.ndarray, biases: np.ndarray,
               group_size: int = 64) -> np.ndarray:
    """``w[n, k] = s[n, k//g] * q[n, k] + b[n, k//g]`` in fp64 from fp16 bit patterns."""
    s = decode_f16(scales)
    b = decode_f16(biases)
    n, k = q.shape
    s_full = np.repeat(s, group_size, axis=1)
    b_full = np.repeat(b, group_size, axis=1)
    assert s_full.shape == (n, k)
    return s_full * q.astype(np.float64) + b_full


def dequant_weight(codes, scales, biases, bits: int, k: int, group_size: int = 64,
                   rows=None) -> np.ndarray:
    """Dequantized fp64 ``[N, K]`` (or the selected ``rows``).

    ``bits = 16`` is the fp16-weight format (the "FP16" end of the pages'
    Q2..FP16 range, gist.science summary, "Metodologia"): the 16-bit "codes"
    are the weights' fp16 bit patterns and scales/biases are not used.
    """
    if rows is not None:
        rows = np.asarray(rows)
        codes = codes[rows]
        if bits != 16:
            scales, biases = scales[rows], biases[rows]
    if bits == 16:
        return decode_f16(unpack_codes(codes, 16, k, group_size).astype(np.uint16))
    return dequantize(unpack_codes(codes, bits, k, group_size), scales, biases, group_size)


# ------------------------------------------------------------------- products
def qgemm(codes, scales, biases, bits: int, x: np.ndarray, group_size: int = 64, rows=None):
    """``Y = X @ W_deq^T`` in fp64 and the tolerance scale ``A = |X| @ |W_deq|^T``.

    ``x`` is fp64 ``[M, K]``.  ``rows`` restricts the output columns (weight rows).
    """
    x = np.asarray(x, dtype=np.float64)
    k = x.shape[1]
    w = dequant_weight(codes, scales, biases, bits, k, group_size, rows)
    y = x @ w.T
    a = np.abs(x) @ np.abs(w).T
    return y, a


def qgemv(codes, scales, biases, bits: int, x: np.ndarray, group_size: int = 64, rows=None):
    """M = 1 case: ``y[n] = sum_k x[k] * w_deq[n, k]``; returns ``(y [N], A [N])``."""
    y, a = qgemm(codes, scales, biases, bits, np.asarray(x, dtype=np.float64)[None, :],
                 group_size, rows)
    return y[0], a[0]


def moe_qgemm(codes, scales, biases, bits: int, offsets, x: np.ndarray, group_size: int = 64):
    """Grouped expert product: rows ``[off[e], off[e+1])`` of ``x`` use expert ``e``.

    ``codes [E, N, K*b/32]``, ``scales/biases [E, N, G]``, ``offsets [E+1]``,
    ``x`` fp64 ``[R, K]``.  Returns ``(y [R, N], A [R, N])``.
    """
    x = np.asarray(x, dtype=np.float64)
    e_count = codes.shape[0]
    n = codes.shape[1]
    y = np.zeros((x.shape[0], n))
    a = np.zeros((x.shape[0], n))
    for e in range(e_count):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            y[lo:hi], a[lo:hi] = qgemm(codes[e], scales[e], biases[e], bits, x[lo:hi], group_size)
    return y, a


# ------------------------------------------------------------ MoE harness steps
def route_sort(ids: np.ndarray, num_experts: int):
    """Group (token, slot) pairs by expert, keeping (token, slot) order within an expert.

    Returns ``(offsets int64 [E+1], pair_index int64 [T*k])`` where ``pair_index[r]``
    is the flat index ``t*k + slot`` of the pair placed at grouped row ``r``.
    """
    flat = np.asarray(ids).reshape(-1).astype(np.int64)
    order = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=num_experts)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    return offsets, order


def silu(v: np.ndarray) -> np.ndarray:
    return v / (1.0 + np.exp(-v))


def swiglu(gate_up: np.ndarray):
    """``h = silu(gate) * up`` for ``gate_up = [gate | up]`` of shape ``[R, 2I]``.

    The step between an expert's gate/up and down products (thetesserapress.com,
    "Where the wins land, and where they don't": the MoE layers whose expert
    products these are).  The pages do not name the activation; SwiGLU is the
    reading taken, the plainest for the Qwen3 family the workloads are shaped
    after.  Returns ``(h [R, I], A = |h|)``: an elementwise step, so its
    tolerance scale is the magnitude of the exact result.
    """
    gu = np.asarray(gate_up, dtype=np.float64)
    inter = gu.shape[1] // 2
    h = silu(gu[:, :inter]) * gu[:, inter:]
    return h, np.abs(h)


def moe_combine(y_grouped: np.ndarray, gates: np.ndarray, pair_index: np.ndarray, top_k: int):
    """Gate-weighted combine: ``out[t] = sum_s g[t, s] * y_grouped[row of pair t*k + s]``.

    The last step of the expert layer (thetesserapress.com, "Where the wins
    land, and where they don't"): each token's expert outputs, weighted by its
    routing gates and summed.  ``pair_index[r]`` is the pair placed at grouped
    row ``r`` (from ``route_sort``).  Returns ``(out [T, H], A = sum_s |g[t, s]
    * y|)``, the per-element tolerance scale of a sum of products.
    """
    y = np.asarray(y_grouped, dtype=np.float64)
    g = np.asarray(gates, dtype=np.float64)
    t_count = g.shape[0]
    out = np.zeros((t_count, y.shape[1]))
    a = np.zeros((t_count, y.shape[1]))
    gflat = g.reshape(-1)
    for r, pair in enumerate(np.asarray(pair_index)):
        out[pair // top_k] += gflat[pair] * y[r]
        a[pair // top_k] += np.abs(gflat[pair] * y[r])
    return out, a


def moe_layer(x: np.ndarray, ids: np.ndarray, gates: np.ndarray, gate_w, up_w, down_w,
              bits: int, group_size: int = 64):
    """One expert layer in fp64: ``out[t] = sum_k g[t,k] * down_e(silu(gate_e x_t) * up_e x_t)``.

    ``gate_w``, ``up_w``, ``down_w`` are ``(codes [E, N, .], scales, biases)`` triples.
    Returns ``(out [T, H], h [T*k, I] in grouped row order, offsets, pair_index)``.
    """
    x = np.asarray(x, dtype=np.float64)
    top_k = ids.shape[1]
    e_count = gate_w[0].shape[0]
    offsets, pair_index = route_sort(ids, e_count)
    xg = x[pair_index // top_k]
    g_out, _ = moe_qgemm(*gate_w, bits, offsets, xg, group_size)
    u_out, _ = moe_qgemm(*up_w, bits, offsets, xg, group_size)
    h = silu(g_out) * u_out
    d_out, _ = moe_qgemm(*down_w, bits, offsets, h, group_size)
    out, _ = moe_combine(d_out, gates, pair_index, top_k)
    return out, h, offsets, pair_index


# ------------------------------------------------------------------ criterion
RTOL = {"f32": 1e-3, "bf16": 8e-3, "f16": 8e-3}
ATOL = 1e-5


def within_tolerance(y, y_ref, a, out_dtype: str):
    """Per-element ``|y - y_ref| <= rtol * A + 1e-5``; returns ``(ok, worst ratio)``."""
    y = np.asarray(y, dtype=np.float64)
    bound = RTOL[out_dtype] * np.asarray(a) + ATOL
    err = np.abs(y - y_ref)
    ratio = float(np.max(err / bound)) if err.size else 0.0
    return bool(np.all(err <= bound)), ratio
