"""ctypes binding of the library's host-side controller and metrics
(spec_ctrl_* and spec_step_stats in include/spec_verify.h).

Argument marshalling only: every rule and statistic is computed by the
native library.  Inputs are host numpy arrays (copies of the verify step's
outputs)."""
from __future__ import annotations

import ctypes

import numpy as np

from ._native import SpecError, lib

MAX_WINDOW = 64
HIST_BINS = 10
MAX_POS = 129  # SPEC_STEP_MAX_POS


class CtrlConfig(ctypes.Structure):
    _fields_ = [("window", ctypes.c_int32), ("high_acceptance", ctypes.c_float),
                ("low_acceptance", ctypes.c_float), ("gamma_high", ctypes.c_int32),
                ("gamma_mid", ctypes.c_int32), ("gamma_low", ctypes.c_int32),
                ("hot_temperature", ctypes.c_float), ("gamma_hot", ctypes.c_int32),
                ("draft_cost", ctypes.c_float), ("min_efficiency", ctypes.c_float),
                ("max_gamma", ctypes.c_int32)]


class CtrlRequest(ctypes.Structure):
    _fields_ = [("drafted", ctypes.c_int16 * MAX_WINDOW),
                ("accepted", ctypes.c_int16 * MAX_WINDOW),
                ("head", ctypes.c_int32), ("steps", ctypes.c_int32),
                ("gamma", ctypes.c_int32), ("fallback", ctypes.c_int32),
                ("failed_steps", ctypes.c_int32)]


class CtrlMetrics(ctypes.Structure):
    _fields_ = [("requests", ctypes.c_int32), ("acceptance_hist", ctypes.c_int32 * HIST_BINS),
                ("acceptance_mean", ctypes.c_float), ("acceptance_p50", ctypes.c_float),
                ("acceptance_p95", ctypes.c_float), ("acceptance_p99", ctypes.c_float),
                ("emitted_per_step", ctypes.c_float),
                ("speculative_efficiency", ctypes.c_float), ("fallback_rate", ctypes.c_float)]


class StepStats(ctypes.Structure):
    _fields_ = [("requests", ctypes.c_int32), ("failed", ctypes.c_int32),
                ("accepted", ctypes.c_int64), ("emitted", ctypes.c_int64),
                ("rejection_pos", ctypes.c_int32 * MAX_POS),
                ("tree_width_effective", ctypes.c_float)]


def _setup():
    L = lib()
    if getattr(L, "_ctrl_ready", False):
        return L
    P = ctypes.POINTER
    L.spec_ctrl_default_config.argtypes = [P(CtrlConfig)]
    L.spec_ctrl_default_config.restype = None
    L.spec_ctrl_init.argtypes = [P(CtrlRequest), ctypes.c_int32, ctypes.c_int32]
    L.spec_ctrl_init.restype = ctypes.c_int32
    L.spec_ctrl_update.argtypes = [P(CtrlConfig), P(CtrlRequest), ctypes.c_int32,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    L.spec_ctrl_update.restype = ctypes.c_int32
    L.spec_ctrl_metrics.argtypes = [P(CtrlConfig), P(CtrlRequest), ctypes.c_int32,
                                    P(CtrlMetrics)]
    L.spec_ctrl_metrics.restype = ctypes.c_int32
    L.spec_step_stats.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_int32, ctypes.c_int32, P(StepStats)]
    L.spec_step_stats.restype = ctypes.c_int32
    L._ctrl_ready = True
    return L


def _i32(x):
    a = np.ascontiguousarray(x, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _check(fn, code):
    if code != 0:
        raise SpecError(fn, code)


def default_config(**overrides) -> CtrlConfig:
    cfg = CtrlConfig()
    _setup().spec_ctrl_default_config(ctypes.byref(cfg))
    for k, v in overrides.items():
        setattr(cfg, k, v)
    return cfg


class Controller:
    """Dynamic draft length per request plus the observability metrics."""

    def __init__(self, n_requests: int, gamma0: int, cfg: CtrlConfig | None = None):
        self.L = _setup()
        self.cfg = cfg or default_config()
        self.n = int(n_requests)
        self.reqs = (CtrlRequest * self.n)()
        _check("spec_ctrl_init", self.L.spec_ctrl_init(self.reqs, self.n, int(gamma0)))

    def update(self, accepted_len, temperature=None) -> np.ndarray:
        a, ap = _i32(accepted_len)
        assert a.shape == (self.n,)
        tp = None
        if temperature is not None:
            t = np.ascontiguousarray(temperature, dtype=np.float32)
            tp = t.ctypes.data_as(ctypes.c_void_p)
        out = np.empty(self.n, dtype=np.int32)
        _check("spec_ctrl_update",
               self.L.spec_ctrl_update(ctypes.byref(self.cfg), self.reqs, self.n, ap, tp,
                                       out.ctypes.data_as(ctypes.c_void_p)))
        return out

    def metrics(self) -> dict:
        m = CtrlMetrics()
        _check("spec_ctrl_metrics",
               self.L.spec_ctrl_metrics(ctypes.byref(self.cfg), self.reqs, self.n,
                                        ctypes.byref(m)))
        return {f: (list(getattr(m, f)) if f == "acceptance_hist" else getattr(m, f))
                for f, _ in CtrlMetrics._fields_}


def step_stats(accepted_len, path=None, parent=None, M=None) -> dict:
    """spec_step_stats over host copies of one step's outputs; M (the rows
    per request) comes from path or parent when given."""
    L = _setup()
    a, ap = _i32(accepted_len)
    B = a.shape[0]
    pp = qp = None
    if path is not None:
        p, pp = _i32(path)
        M = p.shape[1]
    if parent is not None:
        q, qp = _i32(parent)
        M = q.shape[1]
    if M is None:
        M = int(a.max()) + 1 if B else 1
    s = StepStats()
    _check("spec_step_stats", L.spec_step_stats(ap, pp, qp, B, M, ctypes.byref(s)))
    return {"requests": s.requests, "failed": s.failed, "accepted": s.accepted,
            "emitted": s.emitted, "rejection_pos": list(s.rejection_pos)[:M + 1],
            "tree_width_effective": s.tree_width_effective}
