"""ctypes declarations of the C ABI in include/topk.h (libtopk_gb300.so, built in-tree)."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtopk_gb300.so")

TOPK_F32, TOPK_BF16 = 0, 1
TOPK_OK, TOPK_EINVAL, TOPK_ENOMEM, TOPK_ECUDA, TOPK_EUNSUPPORTED, TOPK_ETIMEOUT = 0, -1, -2, -3, -4, -5
TOPK_RULE_EXACT, TOPK_RULE_ALG1 = 0, 1
TOPK_PATH_AUTO, TOPK_PATH_DIRECT, TOPK_PATH_PROFK, TOPK_PATH_EXACT = 0, 1, 2, 3
PATH_NAMES = {TOPK_PATH_DIRECT: "direct", TOPK_PATH_PROFK: "profk", TOPK_PATH_EXACT: "exact"}

# Every symbol include/topk.h declares.
EXPORTS = ("topk_options_init", "topk_select", "topk_select_global", "topk_select_ex", "topk_plan",
           "topk_status_str", "topk_version", "topk_index_bits", "topk_prof_sample", "topk_prof_filter",
           "topk_select_noalloc", "topk_last_status", "topk_autotune", "topk_tuning")


class TopkOptions(ctypes.Structure):
    _fields_ = [("s_min", ctypes.c_int64), ("s_max", ctypes.c_int64), ("cost_ratio", ctypes.c_double),
                ("rule", ctypes.c_int), ("path", ctypes.c_int), ("seed", ctypes.c_uint64),
                ("counter", ctypes.c_int64), ("force_miss", ctypes.c_int), ("m_override", ctypes.c_int64),
                ("t_override", ctypes.c_int64), ("events", ctypes.c_void_p * 6), ("unsorted", ctypes.c_int),
                ("wait_limit_ns", ctypes.c_int64), ("inject_wait_timeout", ctypes.c_int), ("recall", ctypes.c_double)]


class TopkStats(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("index_bits", ctypes.c_int), ("S", ctypes.c_int64),
                ("t", ctypes.c_int64), ("M", ctypes.c_int64), ("R", ctypes.c_int64),
                ("misses", ctypes.c_int64), ("tau", ctypes.c_uint64), ("tau_index", ctypes.c_int64),
                ("seed", ctypes.c_uint64), ("counter", ctypes.c_int64), ("cluster", ctypes.c_int),
                ("launches", ctypes.c_int), ("shortfalls", ctypes.c_int64)]


class TopkTuning(ctypes.Structure):
    _fields_ = [("tau_a_ns", ctypes.c_double), ("tau_b_ns", ctypes.c_double), ("cost_ratio", ctypes.c_double),
                ("crossover_n", ctypes.c_int64), ("crossover_k", ctypes.c_int64)]


class TopkPlan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("S", ctypes.c_int64), ("t", ctypes.c_int64), ("M", ctypes.c_int64),
                ("p_recall_fail", ctypes.c_double), ("p_overflow", ctypes.c_double)]


_lib = None


def get():
    """The loaded library; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libtopk_gb300.so is not built; run `python -m top_selection_prof_gb300.build` "
                               "(the engine has no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, u64, c_int, c_double = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int,
                                         ctypes.c_double)
        lib.topk_options_init.argtypes = [ctypes.POINTER(TopkOptions)]
        lib.topk_options_init.restype = None
        sel = [vp, c_int, i64, i64, i64, c_int, c_double, vp, vp, vp]
        lib.topk_select.argtypes = sel
        lib.topk_select.restype = c_int
        lib.topk_select_global.argtypes = sel
        lib.topk_select_global.restype = c_int
        lib.topk_select_ex.argtypes = sel + [c_int, ctypes.POINTER(TopkOptions), ctypes.POINTER(TopkStats)]
        lib.topk_select_ex.restype = c_int
        lib.topk_plan.argtypes = [i64, i64, c_double, ctypes.POINTER(TopkOptions), ctypes.POINTER(TopkPlan)]
        lib.topk_plan.restype = c_int
        lib.topk_autotune.argtypes = [i64, vp, ctypes.POINTER(TopkTuning)]
        lib.topk_autotune.restype = c_int
        lib.topk_tuning.argtypes = [ctypes.POINTER(TopkTuning)]
        lib.topk_tuning.restype = c_int
        lib.topk_last_status.argtypes = [vp]
        lib.topk_last_status.restype = c_int
        lib.topk_status_str.argtypes = [c_int]
        lib.topk_status_str.restype = ctypes.c_char_p
        lib.topk_version.argtypes = []
        lib.topk_version.restype = c_int
        lib.topk_index_bits.argtypes = [i64]
        lib.topk_index_bits.restype = c_int
        lib.topk_prof_sample.argtypes = [vp, c_int, i64, i64, c_int, c_int, i64, u64, i64, vp, vp]
        lib.topk_prof_sample.restype = c_int
        lib.topk_prof_filter.argtypes = [vp, c_int, i64, i64, c_int, c_int, vp, i64, vp, vp, vp]
        lib.topk_prof_filter.restype = c_int
        _lib = lib
    return _lib


class TopkError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = get().topk_status_str(status).decode()
        super().__init__("%s failed: %s (status %d)" % (what, msg, status))


def check(status: int, what: str) -> None:
    if status != TOPK_OK:
        raise TopkError(status, what)
