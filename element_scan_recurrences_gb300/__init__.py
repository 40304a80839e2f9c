"""GB300-native `element-scan`: nonlinear per-lane recurrences on sm_103a.

The compute path is the C-ABI library ``libes.so`` (hand-written CUDA kernels
for sm_103a, declared in ``include/es.h``); ``scan`` and friends are a thin
ctypes binding over it that only marshals arguments.  The binding loads the
library on first use and raises if it is missing: there is no CPU fallback.
"""
from . import workloads  # noqa: F401  (pure Python: seeded inputs only)

_BINDING_NAMES = {
    "scan", "scan_into", "scan_host", "lib", "LibraryMissing", "EsError", "PATHS",
    "TANH_DECAY", "NORMCAP", "MAXPLUS", "device_status", "plan", "status_string",
    "launch_count", "set_path_override", "set_wait_limit_ns", "set_drop_tile", "scan_backward", "plan_backward",
    "Body", "body_compile_count", "matrix_scan", "plan_matrix_scan", "linear_scan", "plan_linear_scan",
    "table_scan", "plan_table_scan", "matrix_scan_workspace", "matrix_scan_ws", "plan_matrix_scan_ws",
    "matrix_scan_static", "matrix_scan_backward", "plan_matrix_scan_backward", "linear_scan_backward",
    "plan_linear_scan_backward", "matrix_scan_backward_ws", "plan_matrix_scan_backward_ws",
}


def __getattr__(name):
    if name == "element_scan":
        from .autograd import element_scan
        return element_scan
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
