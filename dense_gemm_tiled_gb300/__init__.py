"""GB300-native dense GEMM: C = alpha * op(A) @ op(B) + beta * C, row-major.

The compute path is the C-ABI library built from csrc/ (hand-written sm_103a
kernels: an FP32 FFMA SGEMM and an fp16 -> fp32-accumulate tcgen05 GEMM).
`binding` loads it with ctypes; importing the binding raises if the library is
missing -- there is no fallback.  The `inputs` module (seeded synthetic data)
does not load the library, so it can be imported on a machine without a GPU.
"""
__all__ = ["gemm", "gemm_raw", "gemm_host", "check_device_status", "status_string", "binding",
           "inputs"]


def __getattr__(name):
    if name in ("gemm", "gemm_raw", "gemm_host", "check_device_status", "status_string"):
        from . import binding
        return getattr(binding, name)
    if name in ("binding", "inputs"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
