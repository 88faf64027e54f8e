"""moe_int4_affine_gb300: int4 affine group-quantised dequant-GEMV / MoE-gather decode path for
NVIDIA GB300 (sm_103a).

The compute lives in the CUDA shared library ``libqg.so`` (built from ``csrc/``) behind the C ABI
declared in ``include/qg.h``.  ``moe_int4_affine_gb300.qg`` is the thin ctypes binding with the
same entry-point names; it raises ImportError when the library is missing, so no call can fall
back to anything else.  ``inputs`` holds the seeded synthetic data generators.
"""
from importlib import import_module

_API = ("qgemv_int4", "qgemv_int4_multi", "moe_router_topk", "moe_gather_qgemv_int4", "moe_gather_qgemv_int4_noalloc", "moe_layer_int4",
        "scalar_fma_chain8_residual", "qgemm_int4", "qg_workspace_bytes", "qg_device_status",
        "qg_strerror", "qg_set_pdl", "qg_version", "Int4Weight", "QGError", "to_device", "to_numpy")


def __getattr__(name):
    if name in _API:
        return getattr(import_module(".qg", __name__), name)
    raise AttributeError(name)
