"""ctypes binding of ``libmlora.so`` (the C ABI declared in ``include/mlora.h``).

The functions here carry the C names and only marshal arguments: every step of the layer runs
in the library's CUDA kernels.  PyTorch is used for device memory and streams only.  If the
library has not been built, :func:`lib` raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmlora.so")

MLORA_OK, MLORA_ERR_INVALID, MLORA_ERR_UNSUPPORTED, MLORA_ERR_CUDA, MLORA_ERR_TIMEOUT, MLORA_ERR_OOM = range(6)
MLORA_F32, MLORA_BF16, MLORA_BF16_W4 = 0, 1, 2
MLORA_PLAN_HOST_ONLY = 1
MLORA_DEBUG_SHORT_TIMEOUT = 2
MLORA_GEMM_SINGLE_CTA = 4
MLORA_NO_OVERLAP = 8
MLORA_OVERLAP = 1024
MLORA_REUSE_STAGING = 32
MLORA_W4_FUSED = 64
MLORA_WINDOW_PAIRS = 128
MLORA_WINDOW_SINGLE = 256
MLORA_DEBUG_DROP_COPY = 16
MLORA_DEBUG_DROP_COPY_PAIRS = 512
(MLORA_Q_SUMMARY, MLORA_Q_MTILES, MLORA_Q_COLUMNS, MLORA_Q_WGRAD_A, MLORA_Q_WGRAD_B, MLORA_Q_WINDOW,
 MLORA_Q_ADAPTERS, MLORA_Q_WINDOW_PAIRS, MLORA_Q_GEMM_FWD, MLORA_Q_GEMM_BWD) = range(10)

# every symbol include/mlora.h declares
EXPORTS = ["mlora_plan", "mlora_plan_destroy", "mlora_forward", "mlora_backward", "mlora_adamw",
           "mlora_sync_status", "mlora_h_elems", "mlora_plan_describe", "mlora_status_string",
           "mlora_last_error", "mlora_version", "mlora_profile_enable", "mlora_profile_read",
           "mlora_kernel_name", "mlora_launch_count", "mlora_forward_static_ws", "mlora_memory_estimate",
           "mlora_shard_jobs", "mlora_shard_jobs_multi", "mlora_forward_w4", "mlora_backward_w4",
           "mlora_plan_grouped", "mlora_adamw_ws", "mlora_cost_estimate"]


class mlora_segment(C.Structure):
    _fields_ = [("tok_offset", C.c_int64), ("n_tokens", C.c_int32), ("rank", C.c_int32), ("scale", C.c_float),
                ("At", C.c_void_p), ("Bt", C.c_void_p), ("dAt", C.c_void_p), ("dBt", C.c_void_p),
                ("mA", C.c_void_p), ("vA", C.c_void_p), ("mB", C.c_void_p), ("vB", C.c_void_p)]


class mlora_problem(C.Structure):
    _fields_ = [("n_tokens", C.c_int64), ("d_in", C.c_int32), ("d_out", C.c_int32), ("dtype", C.c_int32),
                ("flags", C.c_uint32), ("mem_budget_bytes", C.c_int64)]


class mlora_cost_point(C.Structure):
    _fields_ = [("d_in", C.c_int32), ("d_out", C.c_int32), ("n_tokens", C.c_int64), ("lora_work", C.c_double),
                ("step_ms", C.c_double)]


class mlora_group(C.Structure):
    _fields_ = [("col_offset", C.c_int32), ("d_out", C.c_int32)]


class mlora_memory(C.Structure):
    _fields_ = [(k, C.c_int64) for k in ("base_weight", "activations", "lora_params", "lora_grad_state", "lora_act",
                                          "workspace", "plan_tables", "total")]


class MloraError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {detail} (status {status})")


_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it was not built (run ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_float
        L.mlora_plan.argtypes = [C.POINTER(mlora_problem), C.POINTER(mlora_segment), i32, C.POINTER(C.c_size_t),
                                 C.POINTER(vp)]
        L.mlora_plan.restype = i32
        L.mlora_plan_grouped.argtypes = [C.POINTER(mlora_problem), C.POINTER(mlora_group), i32,
                                         C.POINTER(mlora_segment), i32, C.POINTER(C.c_size_t), C.POINTER(vp)]
        L.mlora_plan_grouped.restype = i32
        L.mlora_plan_destroy.argtypes = [vp]
        L.mlora_plan_destroy.restype = None
        L.mlora_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        L.mlora_forward.restype = i32
        L.mlora_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.mlora_backward.restype = i32
        L.mlora_adamw.argtypes = [vp, f32, f32, f32, f32, f32, i32, vp]
        L.mlora_adamw.restype = i32
        L.mlora_adamw_ws.argtypes = [vp, f32, f32, f32, f32, f32, i32, vp, vp]
        L.mlora_adamw_ws.restype = i32
        L.mlora_sync_status.argtypes = [vp, vp]
        L.mlora_sync_status.restype = i32
        L.mlora_h_elems.argtypes = [vp]
        L.mlora_h_elems.restype = i64
        L.mlora_plan_describe.argtypes = [vp, i32, C.POINTER(i64), i64, C.POINTER(i64)]
        L.mlora_plan_describe.restype = i32
        L.mlora_status_string.argtypes = [i32]
        L.mlora_status_string.restype = C.c_char_p
        L.mlora_last_error.argtypes = []
        L.mlora_last_error.restype = C.c_char_p
        L.mlora_version.argtypes = []
        L.mlora_version.restype = i32
        L.mlora_profile_enable.argtypes = [vp, i32]
        L.mlora_profile_enable.restype = i32
        L.mlora_profile_read.argtypes = [vp, C.POINTER(C.c_double), C.POINTER(i64), i32, C.POINTER(i32)]
        L.mlora_profile_read.restype = i32
        L.mlora_kernel_name.argtypes = [i32]
        L.mlora_kernel_name.restype = C.c_char_p
        L.mlora_launch_count.argtypes = []
        L.mlora_launch_count.restype = i64
        L.mlora_forward_static_ws.argtypes = [vp, vp, vp, vp, vp, vp]
        L.mlora_forward_static_ws.restype = i32
        L.mlora_forward_w4.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
        L.mlora_forward_w4.restype = i32
        L.mlora_backward_w4.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.mlora_backward_w4.restype = i32
        L.mlora_memory_estimate.argtypes = [vp, C.POINTER(mlora_memory)]
        L.mlora_memory_estimate.restype = i32
        L.mlora_shard_jobs.argtypes = [C.POINTER(mlora_problem), C.POINTER(mlora_segment), i32, i32,
                                       C.POINTER(i32), C.POINTER(C.c_double)]
        L.mlora_shard_jobs.restype = i32
        L.mlora_shard_jobs_multi.argtypes = [C.POINTER(mlora_problem), i32, C.POINTER(mlora_segment), i32, i32,
                                             C.POINTER(i32), C.POINTER(C.c_double)]
        L.mlora_shard_jobs_multi.restype = i32
        L.mlora_cost_estimate.argtypes = [vp, C.POINTER(mlora_cost_point), i32, C.POINTER(C.c_double),
                                          C.POINTER(i32)]
        L.mlora_cost_estimate.restype = i32
        _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != MLORA_OK:
        L = lib()
        raise MloraError(status, where, (L.mlora_last_error() or b"").decode() or
                         L.mlora_status_string(status).decode())


# ------------------------------------------------------------------ thin wrappers, C names

def mlora_plan(problem: mlora_problem, segs) -> tuple[int, int]:
    """Returns (plan handle, workspace bytes)."""
    arr = (mlora_segment * len(segs))(*segs)
    ws = C.c_size_t(0)
    h = C.c_void_p(0)
    _check(lib().mlora_plan(C.byref(problem), arr, len(segs), C.byref(ws), C.byref(h)), "mlora_plan")
    return h.value, ws.value


def mlora_plan_grouped(problem: mlora_problem, groups, segs) -> tuple[int, int]:
    """groups: [(col_offset, d_out), ...]; segs: n_jobs x n_groups entries, job-major.
    Returns (plan handle, workspace bytes)."""
    garr = (mlora_group * len(groups))(*[mlora_group(int(o), int(w)) for o, w in groups])
    arr = (mlora_segment * len(segs))(*segs)
    ws = C.c_size_t(0)
    h = C.c_void_p(0)
    _check(lib().mlora_plan_grouped(C.byref(problem), garr, len(groups), arr, len(segs), C.byref(ws), C.byref(h)),
           "mlora_plan_grouped")
    return h.value, ws.value


def mlora_plan_destroy(plan: int) -> None:
    lib().mlora_plan_destroy(plan)


def mlora_forward(plan, X, Wt, Y, H, workspace, stream) -> None:
    _check(lib().mlora_forward(plan, X, Wt, Y, H, workspace, stream), "mlora_forward")


def mlora_forward_w4(plan, X, Wq, Wscale, Y, H, workspace, stream) -> None:
    _check(lib().mlora_forward_w4(plan, X, Wq, Wscale, Y, H, workspace, stream), "mlora_forward_w4")


def mlora_backward_w4(plan, X, Wq, Wscale, dY, H, dX, dH, workspace, stream) -> None:
    _check(lib().mlora_backward_w4(plan, X, Wq, Wscale, dY, H, dX, dH, workspace, stream), "mlora_backward_w4")


def mlora_backward(plan, X, Wt, dY, H, dX, dH, workspace, stream) -> None:
    _check(lib().mlora_backward(plan, X, Wt, dY, H, dX, dH, workspace, stream), "mlora_backward")


def mlora_adamw(plan, lr, beta1, beta2, eps, weight_decay, step, stream) -> None:
    _check(lib().mlora_adamw(plan, lr, beta1, beta2, eps, weight_decay, step, stream), "mlora_adamw")


def mlora_adamw_ws(plan, lr, beta1, beta2, eps, weight_decay, step, workspace, stream) -> None:
    _check(lib().mlora_adamw_ws(plan, lr, beta1, beta2, eps, weight_decay, step, workspace, stream),
           "mlora_adamw_ws")


def mlora_sync_status(plan, stream) -> int:
    """Returns the status code (does not raise on MLORA_ERR_TIMEOUT)."""
    st = lib().mlora_sync_status(plan, stream)
    if st not in (MLORA_OK, MLORA_ERR_TIMEOUT):
        _check(st, "mlora_sync_status")
    return st


def mlora_h_elems(plan) -> int:
    return int(lib().mlora_h_elems(plan))


def mlora_plan_describe(plan, what: int) -> list[int]:
    L = lib()
    n = C.c_int64(0)
    _check(L.mlora_plan_describe(plan, what, None, 0, C.byref(n)), "mlora_plan_describe")
    buf = (C.c_int64 * max(1, n.value))()
    _check(L.mlora_plan_describe(plan, what, buf, n.value, C.byref(n)), "mlora_plan_describe")
    return list(buf[:n.value])


def mlora_status_string(status: int) -> str:
    return lib().mlora_status_string(status).decode()


def mlora_version() -> int:
    return int(lib().mlora_version())


def mlora_profile_enable(plan, enable: bool) -> None:
    _check(lib().mlora_profile_enable(plan, 1 if enable else 0), "mlora_profile_enable")


def mlora_profile_read(plan) -> dict:
    """{kernel name: (summed ms, timed launches)} since the last read."""
    L = lib()
    n = C.c_int32(0)
    ms = (C.c_double * 64)()
    cnt = (C.c_int64 * 64)()
    _check(L.mlora_profile_read(plan, ms, cnt, 64, C.byref(n)), "mlora_profile_read")
    return {L.mlora_kernel_name(i).decode(): (ms[i], int(cnt[i])) for i in range(n.value)}


def mlora_launch_count() -> int:
    return int(lib().mlora_launch_count())


def mlora_forward_static_ws(plan, X, Wt, Y, H, stream) -> None:
    """Forward pass using the library's static device scratch instead of a caller workspace."""
    _check(lib().mlora_forward_static_ws(plan, X, Wt, Y, H, stream), "mlora_forward_static_ws")


def mlora_memory_estimate(plan) -> dict:
    m = mlora_memory()
    _check(lib().mlora_memory_estimate(plan, C.byref(m)), "mlora_memory_estimate")
    return {k: int(getattr(m, k)) for k, _ in mlora_memory._fields_}


def mlora_shard_jobs(problem: mlora_problem, segs, n_ranks: int):
    """Returns (rank of each job, load per rank)."""
    arr = (mlora_segment * len(segs))(*segs)
    ranks = (C.c_int32 * len(segs))()
    load = (C.c_double * n_ranks)()
    _check(lib().mlora_shard_jobs(C.byref(problem), arr, len(segs), n_ranks, ranks, load), "mlora_shard_jobs")
    return list(ranks), list(load)


def mlora_shard_jobs_multi(problems, segs, n_ranks: int):
    """Jobs shared by several projections (one problem each). Returns (rank of each job, load per rank)."""
    parr = (mlora_problem * len(problems))(*problems)
    arr = (mlora_segment * len(segs))(*segs)
    ranks = (C.c_int32 * len(segs))()
    load = (C.c_double * n_ranks)()
    _check(lib().mlora_shard_jobs_multi(parr, len(problems), arr, len(segs), n_ranks, ranks, load),
           "mlora_shard_jobs_multi")
    return list(ranks), list(load)


def mlora_cost_estimate(plan, points) -> tuple[float, int]:
    """points: [(d_in, d_out, n_tokens, lora_work, step_ms), ...].  Returns (step ms, basis)."""
    arr = (mlora_cost_point * len(points))(*[mlora_cost_point(int(a), int(b), int(n), float(w), float(t))
                                             for a, b, n, w, t in points])
    ms = C.c_double(0.0)
    basis = C.c_int32(0)
    _check(lib().mlora_cost_estimate(plan, arr, len(points), C.byref(ms), C.byref(basis)), "mlora_cost_estimate")
    return ms.value, basis.value
