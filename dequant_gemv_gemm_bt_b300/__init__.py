"""Affine group-quantized GEMV / GEMM / grouped-expert GEMM for B300 (sm_103a).

``synth`` (layout writer and seeded inputs) imports without the native library.
The products live in ``dequant_gemv_gemm_bt_b300.bt``, which loads ``libbt.so``
on import and raises if it is missing.
"""
import importlib

__all__ = ["synth", "bt"]


def __getattr__(name):
    if name in ("synth", "bt"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
