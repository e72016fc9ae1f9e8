"""Python binding of libbt (ctypes; argument marshalling only).

Each function has the name of the C entry point it calls and takes torch CUDA
tensors; shapes are read from the tensors, outputs are allocated with torch
when not given, and every product runs in libbt's CUDA kernels.  There is no
fallback: importing this module raises when ``libbt.so`` is missing, and every
call raises :class:`BTError` when the library returns an error status.

Layout of a packed weight (see ``include/bt.h``): ``codes`` int32 (bit
patterns of uint32) ``[N, K*bits/32]``, ``scales`` and ``biases`` float16
``[N, K/64]``; grouped experts stack a leading ``[E]`` dimension.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbt.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libbt.so not found at {LIB_PATH}; build it with "
        "`python -m dequant_gemv_gemm_bt_b300.build` (nvcc, sm_103a)")

lib = ctypes.CDLL(LIB_PATH)

BT_OK, BT_ERR_INVALID_ARG, BT_ERR_UNSUPPORTED, BT_ERR_MISALIGNED, BT_ERR_CUDA, BT_ERR_TIMEOUT = range(6)
BT_F16, BT_BF16, BT_F32 = 0, 1, 2
(BT_OPT_PDL, BT_OPT_CONST_WEIGHTS, BT_OPT_WAIT_TIMEOUT_US, BT_OPT_TEST_DROP_STAGE,
 BT_OPT_GEMV_GENERIC, BT_OPT_GEMV_STAGES, BT_OPT_GEMM_PATH, BT_OPT_GEMM_SPLITS, BT_OPT_GEMV_MAX_CPL,
 BT_OPT_GEMV_STAGE_KB, BT_OPT_GEMV_RI, BT_OPT_GEMV_CUDA_CORE, BT_OPT_GEMV_MMA_STAGE_KB, BT_OPT_GEMV_MMA_SHAPE,
 BT_OPT_GEMV_MMA_GROUPS, BT_OPT_GEMV_TENSOR_PIPE, BT_OPT_GEMM_DEQ_WARPS, BT_OPT_GEMM_SMALL_WARPS) = range(18)

EXPORTS = ("bt_qgemv", "bt_qgemv_batched", "bt_qgemm", "bt_qgemm_batched", "bt_moe_qgemm", "bt_moe_qgemm_swiglu", "bt_moe_qgemv_pairs",
           "bt_moe_down_combine",
           "bt_moe_route", "bt_swiglu", "bt_moe_combine", "bt_status_string", "bt_last_device_error", "bt_set_option",
           "bt_plan_gemv", "bt_plan_gemv_batch", "bt_plan_gemm", "bt_pass_create", "bt_pass_run", "bt_pass_destroy")

_p = ctypes.c_void_p
_i = ctypes.c_int
_W = [_p, _p, _p, _i, _i]            # codes, scales, biases, bits, group_size
lib.bt_qgemv.argtypes = _W + [_i, _i, _p, _i, _p, _i, _p]
lib.bt_qgemm.argtypes = _W + [_i, _i, _i, _p, _i, _p, _i, _p]


class GemvProblem(ctypes.Structure):
    _fields_ = [("codes", _p), ("scales", _p), ("biases", _p), ("x", _p), ("y", _p), ("n", ctypes.c_int32),
                ("k", ctypes.c_int32)]


lib.bt_qgemv_batched.argtypes = [ctypes.POINTER(GemvProblem), _i, _i, _i, _i, _i, _i, _p]


class GemmProblem(ctypes.Structure):
    _fields_ = [("codes", _p), ("scales", _p), ("biases", _p), ("x", _p), ("y", _p), ("n", ctypes.c_int32),
                ("k", ctypes.c_int32)]


lib.bt_qgemm_batched.argtypes = [ctypes.POINTER(GemmProblem), _i, _i, _i, _i, _i, _i, _p]


class PassStage(ctypes.Structure):
    _fields_ = [("problems", ctypes.POINTER(GemmProblem)), ("count", _i)]


lib.bt_pass_create.argtypes = [ctypes.POINTER(PassStage), _i, _i, _i, _i, _i, _i, ctypes.POINTER(_p)]
lib.bt_pass_run.argtypes = [_p, _p]
lib.bt_pass_destroy.argtypes = [_p]
lib.bt_moe_qgemm.argtypes = _W + [_i, _i, _i, _p, _i, _p, _p, _i, _p, _i, _p]
lib.bt_moe_qgemm_swiglu.argtypes = _W + [_i, _i, _i, _p, _i, _p, _p, _i, _p, _i, _p]
lib.bt_moe_qgemv_pairs.argtypes = _W + [_i, _i, _i, _p, _i, _i, _p, _i, _p, _i, _i, _p]
lib.bt_moe_down_combine.argtypes = _W + [_i, _i, _i, _p, _p, _i, _i, _p, _i, _p, _i, _p]
lib.bt_moe_route.argtypes = [_p, _i, _i, _i, _p, _p, _p, _p, _p]
lib.bt_swiglu.argtypes = [_p, _i, _i, _i, _p, _i, _p]
lib.bt_moe_combine.argtypes = [_p, _i, _p, _p, _i, _i, _i, _p, _i, _p]
lib.bt_status_string.argtypes = [_i]
lib.bt_status_string.restype = ctypes.c_char_p
lib.bt_last_device_error.argtypes = [_p]
lib.bt_set_option.argtypes = [_i, ctypes.c_longlong]


class GemvPlan(ctypes.Structure):
    _fields_ = [("feasible", ctypes.c_int32), ("kw", ctypes.c_int32), ("cpl", ctypes.c_int32), ("ri", ctypes.c_int32),
                ("rows_per_unit", ctypes.c_int32), ("stage_bytes", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("grid", ctypes.c_int32), ("num_units", ctypes.c_int64),
                ("smem_bytes", ctypes.c_int64), ("tensor_pipe", ctypes.c_int32)]


lib.bt_plan_gemv.argtypes = [_i, _i, _i, _i, _i, _i, ctypes.POINTER(GemvPlan)]
lib.bt_plan_gemv_batch.argtypes = [_i, _i, _p, _p, _i, _i, ctypes.POINTER(GemvPlan), _p, _p]


class GemmPlan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("feasible", ctypes.c_int32), ("bn", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("stages", ctypes.c_int32), ("k_blocks", ctypes.c_int32),
                ("grid_x", ctypes.c_int32), ("grid_y", ctypes.c_int32), ("grid_z", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int64), ("rows_per_unit", ctypes.c_int32)]


lib.bt_plan_gemm.argtypes = [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(GemmPlan)]
GEMM_PATHS = {0: "none", 1: "gemv", 2: "simt", 3: "tc", 4: "mma"}
for _name in EXPORTS:
    if _name not in ("bt_status_string", "bt_pass_destroy"):
        getattr(lib, _name).restype = _i
lib.bt_pass_destroy.restype = None

_DT = {torch.float16: BT_F16, torch.bfloat16: BT_BF16, torch.float32: BT_F32}


class BTError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {bt_status_string(status)}")


def bt_status_string(status: int) -> str:
    return lib.bt_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != BT_OK:
        raise BTError(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _dt(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}") from None


def _weights(codes, scales, biases):
    """Device pointers of a packed weight (fp16 weights may pass None for scales and biases)."""
    return (_dev(codes, "codes"), None if scales is None else _dev(scales, "scales"),
            None if biases is None else _dev(biases, "biases"))


# The C entry points take plain pointers and sizes, so they cannot see a buffer
# that is smaller than the sizes say.  These checks compare every tensor with
# the sizes passed alongside it before any pointer reaches a kernel.
def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def check_weight(codes, scales, biases, bits: int, k: int, group_size: int = 64, experts: bool = False) -> int:
    """Packed weight [N, K*bits/32] words + [N, K/g] fp16 params ([E, ...] when ``experts``); returns N.

    ``bits = 16`` is the fp16-weight format: the words hold the weights' fp16 bit
    patterns, and scales/biases are not read (they may be None).
    """
    nd = 3 if experts else 2
    _need(isinstance(codes, torch.Tensor) and codes.dim() == nd, f"codes must be a {nd}-D tensor")
    _need(codes.element_size() == 4 and not codes.is_floating_point(), "codes must be int32/uint32 words")
    _need(codes.shape[-1] * 32 == k * bits,
          f"codes hold {codes.shape[-1] * 32 // max(bits, 1)} {bits}-bit codes per row, K is {k}")
    if bits == 16 and scales is None and biases is None:
        return codes.shape[-2]
    for t, nm in ((scales, "scales"), (biases, "biases")):
        _need(isinstance(t, torch.Tensor) and t.dim() == nd, f"{nm} must be a {nd}-D tensor")
    _need(scales.element_size() == 2 and biases.element_size() == 2, "scales and biases must be 16-bit (fp16)")
    g = k // group_size if group_size > 0 else -1
    want = tuple(codes.shape[:-1]) + (g,)
    _need(tuple(scales.shape) == want and tuple(biases.shape) == want,
          f"scales/biases must be {list(want)}, got {list(scales.shape)} and {list(biases.shape)}")
    return codes.shape[-2]


def _check_int32(t, nm: str, at_least: int) -> None:
    _need(isinstance(t, torch.Tensor) and t.dtype == torch.int32, f"{nm} must be an int32 tensor")
    _need(t.numel() >= at_least, f"{nm} holds {t.numel()} entries, needs {at_least}")


def _check_out(t, nm: str, at_least: int) -> None:
    _need(isinstance(t, torch.Tensor) and t.numel() >= at_least, f"{nm} holds too few elements (needs {at_least})")


def _same_device(*ts) -> None:
    devs = {t.device for t in ts if isinstance(t, torch.Tensor)}
    _need(len(devs) <= 1, f"tensors are on different devices: {sorted(map(str, devs))}")


def bt_set_option(option: int, value: int) -> None:
    _check(lib.bt_set_option(int(option), int(value)), "bt_set_option")


def bt_last_device_error(stream=None) -> int:
    """Synchronize the stream and return (and clear) the device error status."""
    return lib.bt_last_device_error(_stream(stream))


def bt_qgemv(codes, scales, biases, bits: int, x, y=None, *, group_size: int = 64,
             out_dtype=torch.float32, stream=None):
    """``y[n] = sum_k x[k] * w_deq[n, k]``; ``x`` [K] fp16/bf16, ``y`` [N]."""
    k = x.shape[-1]
    n = check_weight(codes, scales, biases, bits, k, group_size)
    _need(x.numel() == k, f"x must hold one row of K = {k}, got shape {list(x.shape)}")
    if y is None:
        y = torch.empty(n, dtype=out_dtype, device=x.device)
    _check_out(y, "y", n)
    _same_device(codes, scales, biases, x, y)
    c, s, b = _weights(codes, scales, biases)
    _check(lib.bt_qgemv(c, s, b, bits, group_size, n, k, _dev(x, "x"), _dt(x), _dev(y, "y"), _dt(y),
                        _stream(stream)), "bt_qgemv")
    return y


def bt_qgemv_batched(problems, bits: int, *, group_size: int = 64, stream=None):
    """Independent GEMVs in one launch.

    ``problems`` is a list of ``(codes, scales, biases, x, y)`` tensors with
    common dtypes; each problem's K is ``x.shape[-1]`` and its ``y`` gets
    ``codes.shape[0]`` rows.  Problems of different K go out as one mixed-K batch.
    """
    ks = set()
    x0, y0 = problems[0][3], problems[0][4]
    for i, (c, s, b, x, y) in enumerate(problems):   # every entry is checked before any is marshalled
        k = x.shape[-1]
        if c.shape[-1] * 32 != k * bits:
            raise ValueError(f"problem {i}: codes hold {c.shape[-1] * 32 // bits} codes per row, x has {k}")
        try:
            check_weight(c, s, b, bits, k, group_size)
            _need(x.numel() == k, f"x must hold one row of K = {k}")
            _check_out(y, "y", c.shape[0])
            _need(x.dtype == x0.dtype and y.dtype == y0.dtype, "every problem must share x and y dtypes")
            _same_device(c, s, b, x, y, x0)
        except ValueError as err:
            raise ValueError(f"problem {i}: {err}") from None
        ks.add(k)
    arr = (GemvProblem * len(problems))()
    for i, (c, s, b, x, y) in enumerate(problems):
        cw, sw, bw = _weights(c, s, b)
        arr[i] = GemvProblem(cw, sw, bw, _dev(x, "x"), _dev(y, "y"), c.shape[0], x.shape[-1])
    k_all = ks.pop() if len(ks) == 1 else 0
    _check(lib.bt_qgemv_batched(arr, len(problems), bits, group_size, k_all, _dt(problems[0][3]),
                                _dt(problems[0][4]), _stream(stream)), "bt_qgemv_batched")
    return [pr[4] for pr in problems]


def bt_qgemm(codes, scales, biases, bits: int, x, y=None, *, group_size: int = 64,
             out_dtype=torch.bfloat16, stream=None):
    """``Y = X @ W_deq^T``; ``x`` [M, K] bf16/fp16, ``Y`` [M, N]."""
    _need(x.dim() == 2, f"x must be [M, K], got shape {list(x.shape)}")
    m, k = x.shape
    n = check_weight(codes, scales, biases, bits, k, group_size)
    if y is None:
        y = torch.empty((m, n), dtype=out_dtype, device=x.device)
    _check_out(y, "y", m * n)
    _same_device(codes, scales, biases, x, y)
    c, s, b = _weights(codes, scales, biases)
    _check(lib.bt_qgemm(c, s, b, bits, group_size, m, n, k, _dev(x, "x"), _dt(x), _dev(y, "y"), _dt(y),
                        _stream(stream)), "bt_qgemm")
    return y


def bt_qgemm_batched(problems, bits: int, *, group_size: int = 64, stream=None):
    """Independent products of the same M in one launch where the shapes allow.

    ``problems`` is a list of ``(codes, scales, biases, x [M, K], y [M, N])`` tensors
    with common dtypes and a common M; each problem has its own K and N.
    """
    m = problems[0][3].shape[0]
    x0, y0 = problems[0][3], problems[0][4]
    arr = _gemm_table(problems, bits, group_size, m, x0, y0, "")
    _check(lib.bt_qgemm_batched(arr, len(problems), bits, group_size, m, _dt(x0), _dt(y0), _stream(stream)),
           "bt_qgemm_batched")
    return [pr[4] for pr in problems]


def _gemm_table(problems, bits, group_size, m, x0, y0, where):
    """Checks one list of ``(codes, scales, biases, x, y)`` products and marshals it."""
    for i, (c, s, b, x, y) in enumerate(problems):   # every entry is checked before any is marshalled
        try:
            _need(x.dim() == 2 and x.shape[0] == m, f"x must be [M={m}, K], got shape {list(x.shape)}")
            n = check_weight(c, s, b, bits, x.shape[1], group_size)
            _check_out(y, "y", m * n)
            _need(x.dtype == x0.dtype and y.dtype == y0.dtype, "every problem must share x and y dtypes")
            _same_device(c, s, b, x, y, x0)
        except ValueError as err:
            raise ValueError(f"{where}problem {i}: {err}") from None
    arr = (GemmProblem * len(problems))()
    for i, (c, s, b, x, y) in enumerate(problems):
        cw, sw, bw = _weights(c, s, b)
        arr[i] = GemmProblem(cw, sw, bw, _dev(x, "x"), _dev(y, "y"), c.shape[0], x.shape[1])
    return arr


class DecodePass:
    """A planned decode pass (``bt_pass_create``); holds the tensors it reads and writes."""

    def __init__(self, handle, tensors):
        self._handle = handle
        self._tensors = tensors   # the pass reads and writes these buffers for its whole life
        self._ran = False

    def run(self, stream=None):
        bt_pass_run(self, stream=stream)

    def close(self):
        bt_pass_destroy(self)

    def __del__(self):
        try:
            bt_pass_destroy(self)
        except Exception:   # interpreter shutdown: the library may already be unloaded
            pass


def bt_pass_create(stages, bits: int, *, group_size: int = 64):
    """Plans an ordered list of stages once; ``stages`` is a list of lists of
    ``(codes, scales, biases, x [M, K], y [M, N])`` products with one common M and
    common dtypes.  A stage may read what an earlier stage writes; runs write
    the same y buffers and read the x buffers as they are at the time."""
    _need(len(stages) > 0 and all(len(st) > 0 for st in stages), "every stage needs at least one product")
    first = stages[0][0]
    m, x0, y0 = first[3].shape[0], first[3], first[4]
    tables = [_gemm_table(st, bits, group_size, m, x0, y0, f"stage {si}: ") for si, st in enumerate(stages)]
    arr = (PassStage * len(stages))()
    for si, t in enumerate(tables):
        arr[si] = PassStage(ctypes.cast(t, ctypes.POINTER(GemmProblem)), len(t))
    handle = _p()
    _check(lib.bt_pass_create(arr, len(stages), bits, group_size, m, _dt(x0), _dt(y0), ctypes.byref(handle)),
           "bt_pass_create")
    return DecodePass(handle, [t for st in stages for pr in st for t in pr])


def bt_pass_run(dpass: DecodePass, stream=None):
    """Launches the pass on ``stream`` (the first run also records it as a CUDA graph)."""
    _need(dpass._handle is not None, "the pass was destroyed")
    _check(lib.bt_pass_run(dpass._handle, _stream(stream)), "bt_pass_run")
    dpass._ran = True


def bt_pass_destroy(dpass: DecodePass):
    """Frees the pass (its graph and stream) once its runs have finished; the
    tensors stay the caller's."""
    if dpass._handle is not None:
        if dpass._ran and torch.cuda.is_available():
            torch.cuda.synchronize()   # no run of the pass may still be in flight
        lib.bt_pass_destroy(dpass._handle)
        dpass._handle = None


def bt_moe_qgemm(codes, scales, biases, bits: int, expert_offsets, x, y=None, *, total_rows=None,
                 x_row_index=None, group_size: int = 64, out_dtype=torch.bfloat16, stream=None):
    """Grouped expert product; ``codes`` [E, N, .], ``expert_offsets`` int32 [E+1] on the device.

    ``total_rows`` defaults to ``len(x_row_index)`` when a gather index is given, else ``x.shape[0]``.
    """
    k = x.shape[-1]
    n = check_weight(codes, scales, biases, bits, k, group_size, experts=True)
    e = codes.shape[0]
    if total_rows is None:
        total_rows = x_row_index.shape[0] if x_row_index is not None else x.shape[0]
    _check_int32(expert_offsets, "expert_offsets", e + 1)
    if x_row_index is not None:
        _check_int32(x_row_index, "x_row_index", total_rows)
    else:
        _need(x.numel() >= total_rows * k, f"x holds {x.numel() // max(k, 1)} rows, total_rows is {total_rows}")
    if y is None:
        y = torch.empty((total_rows, n), dtype=out_dtype, device=x.device)
    _check_out(y, "y", total_rows * n)
    _same_device(codes, scales, biases, x, y, expert_offsets, x_row_index)
    c, s, b = _weights(codes, scales, biases)
    ri = _dev(x_row_index, "x_row_index") if x_row_index is not None else None
    _check(lib.bt_moe_qgemm(c, s, b, bits, group_size, e, n, k, _dev(expert_offsets, "expert_offsets"),
                            total_rows, ri, _dev(x, "x"), _dt(x), _dev(y, "y"), _dt(y), _stream(stream)),
           "bt_moe_qgemm")
    return y


def bt_moe_qgemm_swiglu(codes, scales, biases, bits: int, expert_offsets, x, h=None, *, total_rows=None,
                        x_row_index=None, group_size: int = 64, out_dtype=torch.bfloat16, stream=None):
    """Grouped gate|up product with the SwiGLU epilogue: ``codes`` [E, 2I, .] with gate/up rows
    interleaved (row 2i gate i, row 2i+1 up i); returns ``h`` [total_rows, I]."""
    k = x.shape[-1]
    n = check_weight(codes, scales, biases, bits, k, group_size, experts=True)
    _need(n % 2 == 0, f"gate|up rows must be even (interleaved pairs), got {n}")
    e = codes.shape[0]
    if total_rows is None:
        total_rows = x_row_index.shape[0] if x_row_index is not None else x.shape[0]
    _check_int32(expert_offsets, "expert_offsets", e + 1)
    if x_row_index is not None:
        _check_int32(x_row_index, "x_row_index", total_rows)
    else:
        _need(x.numel() >= total_rows * k, f"x holds {x.numel() // max(k, 1)} rows, total_rows is {total_rows}")
    if h is None:
        h = torch.empty((total_rows, n // 2), dtype=out_dtype, device=x.device)
    _check_out(h, "h", total_rows * (n // 2))
    _same_device(codes, scales, biases, x, h, expert_offsets, x_row_index)
    c, s, b = _weights(codes, scales, biases)
    ri = _dev(x_row_index, "x_row_index") if x_row_index is not None else None
    _check(lib.bt_moe_qgemm_swiglu(c, s, b, bits, group_size, e, n, k, _dev(expert_offsets, "expert_offsets"),
                                   total_rows, ri, _dev(x, "x"), _dt(x), _dev(h, "h"), _dt(h), _stream(stream)),
           "bt_moe_qgemm_swiglu")
    return h


def bt_moe_qgemv_pairs(codes, scales, biases, bits: int, topk_ids, x, y=None, *, swiglu: bool = False,
                       group_size: int = 64, out_dtype=torch.float16, stream=None):
    """Routed pairs without a sort: pair r = t*top_k + s uses expert ``topk_ids[t, s]`` and x row t;
    returns ``y`` [T*top_k, N] (``N/2`` with the SwiGLU epilogue, gate/up rows interleaved)."""
    _need(x.dim() == 2, f"x must be [T, K], got shape {list(x.shape)}")
    t, k = x.shape
    n = check_weight(codes, scales, biases, bits, k, group_size, experts=True)
    _check_int32(topk_ids, "topk_ids", 0)
    _need(topk_ids.dim() == 2 and topk_ids.shape[0] == t, f"topk_ids must be [T={t}, top_k]")
    top_k = topk_ids.shape[1]
    cols = n // 2 if swiglu else n
    _need(not swiglu or n % 2 == 0, "gate|up rows must be even (interleaved pairs)")
    if y is None:
        y = torch.empty((t * top_k, cols), dtype=out_dtype, device=x.device)
    _check_out(y, "y", t * top_k * cols)
    _same_device(codes, scales, biases, x, y, topk_ids)
    c, s, b = _weights(codes, scales, biases)
    _check(lib.bt_moe_qgemv_pairs(c, s, b, bits, group_size, codes.shape[0], n, k, _dev(topk_ids, "topk_ids"), t,
                                  top_k, _dev(x, "x"), _dt(x), _dev(y, "y"), _dt(y), 1 if swiglu else 0,
                                  _stream(stream)), "bt_moe_qgemv_pairs")
    return y


def bt_moe_down_combine(codes, scales, biases, bits: int, topk_ids, gates, h, out=None, *, group_size: int = 64,
                        out_dtype=torch.float32, stream=None):
    """Down products of each token's routed experts, gate-weighted and summed in the kernel:
    ``out[t] = sum_s gates[t, s] * W_down[ids[t, s]] @ h[t*top_k + s]``; ``h`` [T*top_k, K]."""
    _check_int32(topk_ids, "topk_ids", 0)
    _need(topk_ids.dim() == 2, "topk_ids must be [T, top_k]")
    t, top_k = topk_ids.shape
    k = h.shape[-1]
    n = check_weight(codes, scales, biases, bits, k, group_size, experts=True)
    _need(h.dim() == 2 and h.shape[0] == t * top_k, f"h must be [T*top_k = {t * top_k}, K]")
    _need(isinstance(gates, torch.Tensor) and gates.dtype == torch.float32 and gates.numel() >= t * top_k,
          "gates must be a float32 tensor of [T, top_k]")
    if out is None:
        out = torch.empty((t, n), dtype=out_dtype, device=h.device)
    _check_out(out, "out", t * n)
    _same_device(codes, scales, biases, h, out, topk_ids, gates)
    c, s, b = _weights(codes, scales, biases)
    _check(lib.bt_moe_down_combine(c, s, b, bits, group_size, codes.shape[0], n, k, _dev(topk_ids, "topk_ids"),
                                   _dev(gates, "gates"), t, top_k, _dev(h, "h"), _dt(h), _dev(out, "out"),
                                   _dt(out), _stream(stream)), "bt_moe_down_combine")
    return out


def bt_moe_route(topk_ids, num_experts: int, offsets=None, pair_index=None, pair_row=None, pair_token=None,
                 stream=None, with_token=False):
    """Stable grouping of (token, slot) pairs by expert.

    Returns ``(offsets, pair_index, pair_row)``, plus ``pair_token`` (the token of each
    grouped row, for ``x_row_index``) when ``with_token`` or a ``pair_token`` buffer is given.
    """
    _need(topk_ids.dim() == 2, "topk_ids must be [T, top_k]")
    t, top_k = topk_ids.shape
    _check_int32(topk_ids, "topk_ids", t * top_k)
    dev = topk_ids.device
    if offsets is None:
        offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    if pair_index is None:
        pair_index = torch.empty(t * top_k, dtype=torch.int32, device=dev)
    if pair_row is None:
        pair_row = torch.empty(t * top_k, dtype=torch.int32, device=dev)
    want_token = with_token or pair_token is not None
    if want_token and pair_token is None:
        pair_token = torch.empty(t * top_k, dtype=torch.int32, device=dev)
    _check_int32(offsets, "offsets", num_experts + 1)
    for buf, nm in ((pair_index, "pair_index"), (pair_row, "pair_row")) + (((pair_token, "pair_token"),) if want_token else ()):
        _check_int32(buf, nm, t * top_k)
    _same_device(topk_ids, offsets, pair_index, pair_row, pair_token)
    _check(lib.bt_moe_route(_dev(topk_ids, "topk_ids"), t, top_k, num_experts, _dev(offsets, "offsets"),
                            _dev(pair_index, "pair_index"), _dev(pair_row, "pair_row"),
                            _dev(pair_token, "pair_token") if want_token else None, _stream(stream)),
           "bt_moe_route")
    if want_token:
        return offsets, pair_index, pair_row, pair_token
    return offsets, pair_index, pair_row


def bt_swiglu(gate_up, h=None, *, out_dtype=None, stream=None):
    """``h = silu(gate_up[:, :I]) * gate_up[:, I:]``."""
    _need(gate_up.dim() == 2 and gate_up.shape[1] % 2 == 0, "gate_up must be [rows, 2*I]")
    rows, two_i = gate_up.shape
    inter = two_i // 2
    if h is None:
        h = torch.empty((rows, inter), dtype=out_dtype or gate_up.dtype, device=gate_up.device)
    _check_out(h, "h", rows * inter)
    _same_device(gate_up, h)
    _check(lib.bt_swiglu(_dev(gate_up, "gate_up"), _dt(gate_up), rows, inter, _dev(h, "h"), _dt(h),
                         _stream(stream)), "bt_swiglu")
    return h


def bt_moe_combine(y_grouped, gates, pair_row, top_k: int, out=None, *, out_dtype=None, stream=None):
    """``out[t] = sum_s gates[t, s] * y_grouped[pair_row[t*top_k + s]]``."""
    _need(y_grouped.dim() == 2, "y_grouped must be [T*top_k, H]")
    _need(gates.dim() == 2 and gates.shape[1] == top_k and gates.dtype == torch.float32,
          "gates must be float32 [T, top_k]")
    hidden = y_grouped.shape[1]
    tokens = gates.shape[0]
    _need(y_grouped.shape[0] >= tokens * top_k, f"y_grouped holds {y_grouped.shape[0]} rows, needs {tokens * top_k}")
    _check_int32(pair_row, "pair_row", tokens * top_k)
    if out is None:
        out = torch.empty((tokens, hidden), dtype=out_dtype or y_grouped.dtype, device=y_grouped.device)
    _check_out(out, "out", tokens * hidden)
    _same_device(y_grouped, gates, pair_row, out)
    _check(lib.bt_moe_combine(_dev(y_grouped, "y_grouped"), _dt(y_grouped), _dev(gates, "gates"),
                              _dev(pair_row, "pair_row"), tokens, top_k, hidden, _dev(out, "out"), _dt(out),
                              _stream(stream)), "bt_moe_combine")
    return out


def _plan_dict(pl) -> dict:
    return {name: getattr(pl, name) for name, _ in type(pl)._fields_}


def bt_plan_gemv(bits: int, n: int, k: int, *, problems: int = 1, x_dtype=torch.float16, sms: int = 148) -> dict:
    """The GEMV launch plan for ``problems`` GEMVs of [n, k] on ``sms`` SMs (host only, no GPU needed)."""
    pl = GemvPlan()
    _check(lib.bt_plan_gemv(bits, _DT[x_dtype], n, k, problems, sms, ctypes.byref(pl)), "bt_plan_gemv")
    return _plan_dict(pl)


def bt_plan_gemv_batch(bits: int, shapes, *, x_dtype=torch.float16, sms: int = 148):
    """Plan of one mixed-K batched launch over ``shapes`` = [(n, k), ...] (host only).

    Returns ``(plan dict, [(kw, rows_per_unit) per problem])``.
    """
    cnt = len(shapes)
    n = (ctypes.c_int32 * cnt)(*[int(a) for a, _ in shapes])
    k = (ctypes.c_int32 * cnt)(*[int(b) for _, b in shapes])
    kw = (ctypes.c_int32 * cnt)()
    rb = (ctypes.c_int32 * cnt)()
    pl = GemvPlan()
    _check(lib.bt_plan_gemv_batch(bits, _DT[x_dtype], n, k, cnt, sms, ctypes.byref(pl), kw, rb),
           "bt_plan_gemv_batch")
    return _plan_dict(pl), list(zip(kw, rb))


def bt_plan_gemm(bits: int, m: int, n: int, k: int, *, num_experts: int = 0, x_dtype=torch.bfloat16,
                 sms: int = 148) -> dict:
    """Launch plan of a dense (num_experts=0) or grouped product of m rows (host only, no GPU needed).

    ``path`` is one of "none", "gemv", "simt" (CUDA-core tile), "tc" (tensor cores) or "mma"
    (the small-token tensor-pipe kernel).
    """
    pl = GemmPlan()
    _check(lib.bt_plan_gemm(bits, _DT[x_dtype], m, n, k, num_experts, sms, ctypes.byref(pl)), "bt_plan_gemm")
    d = _plan_dict(pl)
    d["path"] = GEMM_PATHS[d["path"]]
    return d
