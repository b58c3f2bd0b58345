"""Thin ctypes binding of the QEvict C ABI (include/qevict.h).

Argument marshalling only: every step of the decode path runs in the CUDA library.  PyTorch
provides the device memory (the arena and the tensors) and the stream.  If the library is
missing this module raises; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
# QEVICT_LIB=check loads the checked build (device bounds checks that report to the status word)
LIB_PATH = os.path.join(HERE, "libqevict_check.so" if os.environ.get("QEVICT_LIB") == "check" else "libqevict.so")

OK, EINVAL, EBUDGET, ENOMEM, ESCHEDULE, ECUDA, EDEVICE = range(7)
COUNTER_NAMES = ("promotions", "demotions", "first_quant", "reactivations", "evictions", "aged_full", "aged_quant")


class QEvictError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("batch", "n_layers", "h_q", "h_kv", "d_head", "n_sink", "n_recent",
                                             "window", "bits", "omega", "q_num", "q_den", "budget_num",
                                             "budget_den")] + \
               [("b_total", ctypes.c_int64), ("prompt_len", ctypes.c_int32), ("max_len", ctypes.c_int32),
                ("ranker", ctypes.c_int32), ("no_promotion", ctypes.c_int32), ("decay", ctypes.c_float),
                ("pnorm", ctypes.c_float), ("rope", ctypes.c_int32), ("reserved0", ctypes.c_int32)]


class BudgetInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("full_bytes", "b_total", "b_sink", "b_local", "b_hist", "payload",
                                             "m_f", "m_q")] + \
               [(n, ctypes.c_int32) for n in ("k_f", "k_q", "n_windows", "ring_windows")]


_LAYOUT_REGIONS = ("sink", "ring", "fpool", "ledger", "score", "state", "fslot", "lslot", "ftab", "qtab", "meta")


class Layout(ctypes.Structure):
    _fields_ = [(f"{k}_{r}", ctypes.c_int64) for r in _LAYOUT_REGIONS for k in ("off", "stride")] + \
               [("qblock", ctypes.c_int64), ("arena_bytes", ctypes.c_int64), ("n_split", ctypes.c_int32),
                ("pad_", ctypes.c_int32), ("off_agg", ctypes.c_int64), ("stride_agg", ctypes.c_int64),
                ("off_rope", ctypes.c_int64)]


class Tuple(ctypes.Structure):
    """Device views of one (layer, sequence) cache tuple (qevict_tuple)."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("sink", "ring", "fpool", "ledger", "score", "state", "f_slot",
                                               "l_slot", "f_table", "q_table", "meta")]


class DiagConfig(ctypes.Structure):
    _fields_ = [("horizon", ctypes.c_int32), ("lir_m", ctypes.c_int32)]


class DiagReport(ctypes.Structure):
    _fields_ = [("events", ctypes.c_int64), ("fmm", ctypes.c_double), ("fmm_terms", ctypes.c_int64),
                ("churn", ctypes.c_double), ("churn_terms", ctypes.c_int64), ("qsa", ctypes.c_double),
                ("r_q", ctypes.c_double), ("qsa_terms", ctypes.c_int64), ("tier_mass", ctypes.c_double * 4),
                ("lir_eligible", ctypes.c_int64), ("lir_rescued", ctypes.c_int64),
                ("lir_fullkv_eligible", ctypes.c_int64), ("lir_fullkv_rescued", ctypes.c_int64),
                ("lag", ctypes.c_int64 * 32)]


_lib = None


def load() -> ctypes.CDLL:
    """Loads libqevict.so from the package directory; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with recoverable_quantized_kv_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "qevict_budget": [ctypes.POINTER(Config), ctypes.POINTER(BudgetInfo)],
        "qevict_cache_bytes": [ctypes.POINTER(Config), ctypes.POINTER(ctypes.c_size_t)],
        "qevict_init_cache": [ctypes.POINTER(Config), P, ctypes.c_size_t, P, ctypes.POINTER(P)],
        "qevict_get_layout": [P, ctypes.POINTER(Layout)],
        "qevict_prefill_scores": [P, P, P, P, P],
        "qevict_prefill_route": [P, I32, P, P, P, P, P],
        "qevict_decode_step": [P, I32, P, P, P, P, P],
        "qevict_route": [P, P],
        "qevict_flush_scores": [P, P],
        "qevict_set_rope_table": [P, P, I64, P],
        "qevict_diag_bytes": [P, ctypes.POINTER(DiagConfig), ctypes.POINTER(ctypes.c_size_t)],
        "qevict_diag_init": [P, P, ctypes.POINTER(DiagConfig), P, ctypes.c_size_t, P, ctypes.POINTER(P)],
        "qevict_diag_route": [P, P],
        "qevict_diag_read": [P, ctypes.POINTER(DiagReport), P],
        "qevict_diag_destroy": [P],
        "qevict_get_tuple": [P, I32, I32, ctypes.POINTER(Tuple)],
        "qevict_export_bytes": [P, ctypes.POINTER(ctypes.c_size_t)],
        "qevict_export_state": [P, P, ctypes.c_size_t, P],
        "qevict_import_state": [P, P, ctypes.c_size_t, P],
        "qevict_read_counters": [P, ctypes.POINTER(I64), P],
        "qevict_check": [P, P],
        "qevict_selftest_wait": [P, P],
        "qevict_destroy": [P],
        "qevict_prefill_scores_noalloc": [I32, I32, I32, I32, I32, I32, P, P, P, P],
        "qevict_prefill_scores_noalloc_status": [P],
        "qevict_debug_cap_free_slots": [P, I32],
        "qevict_read_status": [P, ctypes.POINTER(I32), P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.qevict_status_string.argtypes = [ctypes.c_int]
    lib.qevict_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def exported_symbols():
    """Names of the C ABI entry points declared in include/qevict.h."""
    return ["qevict_budget", "qevict_cache_bytes", "qevict_init_cache", "qevict_get_layout",
            "qevict_prefill_scores", "qevict_prefill_route", "qevict_decode_step", "qevict_route",
            "qevict_read_counters", "qevict_check", "qevict_destroy", "qevict_status_string",
            "qevict_prefill_scores_noalloc", "qevict_flush_scores", "qevict_get_tuple", "qevict_export_bytes",
            "qevict_export_state", "qevict_import_state", "qevict_set_rope_table", "qevict_diag_bytes",
            "qevict_diag_init", "qevict_diag_route", "qevict_diag_read", "qevict_diag_destroy",
            "qevict_selftest_wait", "qevict_prefill_scores_noalloc_status", "qevict_debug_cap_free_slots",
            "qevict_read_status"]


def _check(status: int, where: str):
    if status != OK:
        raise QEvictError(status, where, load().qevict_status_string(status).decode())


def make_config(wl, **over) -> Config:
    """C config from any object with the workload's field names (e.g. synth.Workload)."""
    c = Config()
    for name, _ in Config._fields_:
        if name == "b_total":
            c.b_total = int(over.get("b_total", getattr(wl, "b_total", 0) or 0))
        elif name == "max_len":
            c.max_len = int(over.get("max_len", wl.prompt_len + wl.steps))
        elif name in ("decay", "pnorm"):
            setattr(c, name, float(over.get(name, getattr(wl, name, 0.0))))
        elif name in ("ranker", "no_promotion"):
            setattr(c, name, int(over.get(name, getattr(wl, name, 0))))
        elif name == "rope":   # keys carry RoPE and are quantised before it when the workload has a base
            c.rope = int(over.get("rope", 1 if float(getattr(wl, "rope_base", 0.0) or 0.0) > 0 else 0))
        elif name == "reserved0":
            c.reserved0 = 0
        else:
            setattr(c, name, int(over.get(name, getattr(wl, name))))
    return c


def budget(cfg: Config) -> BudgetInfo:
    b = BudgetInfo()
    _check(load().qevict_budget(ctypes.byref(cfg), ctypes.byref(b)), "qevict_budget")
    return b


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def prefill_scores_noalloc(batch, prompt_len, h_q, h_kv, n_sink, window, q_prompt, k_prompt, s0_out, stream=None):
    """Prefill scores through the allocation-free entry point (scratch inside the library image)."""
    _check(load().qevict_prefill_scores_noalloc(batch, prompt_len, h_q, h_kv, n_sink, window, _ptr(q_prompt),
                                                _ptr(k_prompt), _ptr(s0_out), _stream(stream)),
           "qevict_prefill_scores_noalloc")


def prefill_scores_noalloc_status(stream=None):
    """Reads and clears the allocation-free entry point's device status word (raises EDEVICE if set)."""
    _check(load().qevict_prefill_scores_noalloc_status(_stream(stream)), "qevict_prefill_scores_noalloc_status")


class Cache:
    """A QEvict cache over a torch-allocated arena (uint8 CUDA tensor)."""

    def __init__(self, cfg: Config, device="cuda", stream=None, arena=None):
        import torch
        lib = load()
        self.cfg = cfg
        self.bud = budget(cfg)
        nbytes = ctypes.c_size_t()
        _check(lib.qevict_cache_bytes(ctypes.byref(cfg), ctypes.byref(nbytes)), "qevict_cache_bytes")
        self.arena = arena if arena is not None else torch.empty(nbytes.value, dtype=torch.uint8, device=device)
        if self.arena.data_ptr() % 256:
            raise QEvictError(EINVAL, "Cache", "arena must be 256-byte aligned")
        h = ctypes.c_void_p()
        _check(lib.qevict_init_cache(ctypes.byref(cfg), self.arena.data_ptr(), self.arena.numel(), _stream(stream),
                                     ctypes.byref(h)), "qevict_init_cache")
        self.handle = h
        self.layout = Layout()
        _check(lib.qevict_get_layout(h, ctypes.byref(self.layout)), "qevict_get_layout")

    def close(self):
        if self.handle:
            load().qevict_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- the C ABI calls
    def prefill_scores(self, q_prompt, k_prompt, s0_out, stream=None):
        _check(load().qevict_prefill_scores(self.handle, _ptr(q_prompt), _ptr(k_prompt), _ptr(s0_out),
                                            _stream(stream)), "qevict_prefill_scores")

    def set_rope_table(self, table, stream=None):
        """table: fp32 CUDA tensor [rows][64][2] of (cos, sin) per position and channel pair."""
        import torch
        if table.dtype != torch.float32 or not table.is_cuda or not table.is_contiguous():
            raise QEvictError(EINVAL, "set_rope_table", "table must be a contiguous float32 CUDA tensor")
        _check(load().qevict_set_rope_table(self.handle, _ptr(table), int(table.shape[0]), _stream(stream)),
               "qevict_set_rope_table")

    def prefill_route(self, layer: int, k_prompt, v_prompt, s0=None, q_prompt=None, stream=None):
        _check(load().qevict_prefill_route(self.handle, layer, _ptr(k_prompt), _ptr(v_prompt), _ptr(s0),
                                           _ptr(q_prompt), _stream(stream)), "qevict_prefill_route")

    def decode_step(self, layer: int, q, k_new, v_new, out, stream=None):
        _check(load().qevict_decode_step(self.handle, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                         _stream(stream)), "qevict_decode_step")

    def route(self, stream=None):
        _check(load().qevict_route(self.handle, _stream(stream)), "qevict_route")

    def flush_scores(self, stream=None):
        _check(load().qevict_flush_scores(self.handle, _stream(stream)), "qevict_flush_scores")

    def tuple(self, layer: int, seq: int) -> Tuple:
        t = Tuple()
        _check(load().qevict_get_tuple(self.handle, layer, seq, ctypes.byref(t)), "qevict_get_tuple")
        return t

    def export_state(self, stream=None):
        """Checkpoint of the whole cache as a host uint8 numpy array (synchronises the stream)."""
        import numpy as np
        n = ctypes.c_size_t()
        _check(load().qevict_export_bytes(self.handle, ctypes.byref(n)), "qevict_export_bytes")
        buf = np.empty(n.value, dtype=np.uint8)
        _check(load().qevict_export_state(self.handle, buf.ctypes.data, buf.nbytes, _stream(stream)),
               "qevict_export_state")
        return buf

    def import_state(self, buf, stream=None):
        """Loads a checkpoint made by export_state of a cache with the same configuration."""
        import numpy as np
        buf = np.ascontiguousarray(buf, dtype=np.uint8)
        _check(load().qevict_import_state(self.handle, buf.ctypes.data, buf.nbytes, _stream(stream)),
               "qevict_import_state")

    def counters(self, stream=None) -> dict:
        buf = (ctypes.c_int64 * 7)()
        _check(load().qevict_read_counters(self.handle, buf, _stream(stream)), "qevict_read_counters")
        return dict(zip(COUNTER_NAMES, list(buf)))

    def check(self, stream=None):
        _check(load().qevict_check(self.handle, _stream(stream)), "qevict_check")

    def selftest_wait(self, stream=None):
        """Enqueue the bounded-wait self-test: a wait that runs out and records a timeout."""
        _check(load().qevict_selftest_wait(self.handle, _stream(stream)), "qevict_selftest_wait")

    def status_word(self, stream=None) -> int:
        """The device status word (bit 1 timeout, 2 slot exhaustion, 4 inconsistent state, 8 bounds)."""
        w = ctypes.c_int32()
        _check(load().qevict_read_status(self.handle, ctypes.byref(w), _stream(stream)), "qevict_read_status")
        return w.value

    def debug_cap_free_slots(self, cap: int):
        """Routing events see at most `cap` free F / ledger slots (-1: no cap); a test hook."""
        _check(load().qevict_debug_cap_free_slots(self.handle, cap), "qevict_debug_cap_free_slots")

    # ---- tensor views of the cache tuple inside the arena (read-only use in tests)
    def region(self, name: str, unit: int, nbytes: int):
        off = getattr(self.layout, f"off_{name}") + unit * getattr(self.layout, f"stride_{name}")
        return self.arena[off:off + nbytes]

    def unit(self, layer: int, seq: int) -> int:
        return layer * self.cfg.batch + seq


class Diagnostics:
    """Routing diagnostics of a policy cache against a FullKV cache fed the same inputs (QEvict App. I).
    Create after both caches are prefilled; call route() in place of both caches' route()."""

    def __init__(self, policy: "Cache", fullkv: "Cache", horizon: int = 0, lir_m: int = 0, stream=None):
        import torch
        lib = load()
        self.policy, self.fullkv = policy, fullkv
        self.dc = DiagConfig(horizon, lir_m)
        n = ctypes.c_size_t()
        _check(lib.qevict_diag_bytes(policy.handle, ctypes.byref(self.dc), ctypes.byref(n)), "qevict_diag_bytes")
        self.buf = torch.empty(n.value, dtype=torch.uint8, device=policy.arena.device)
        h = ctypes.c_void_p()
        _check(lib.qevict_diag_init(policy.handle, fullkv.handle, ctypes.byref(self.dc), self.buf.data_ptr(),
                                    self.buf.numel(), _stream(stream), ctypes.byref(h)), "qevict_diag_init")
        self.handle = h

    def route(self, stream=None):
        _check(load().qevict_diag_route(self.handle, _stream(stream)), "qevict_diag_route")

    def report(self, stream=None) -> dict:
        r = DiagReport()
        _check(load().qevict_diag_read(self.handle, ctypes.byref(r), _stream(stream)), "qevict_diag_read")
        import numpy as np
        return {"events": r.events, "fmm": r.fmm, "fmm_terms": r.fmm_terms, "churn": r.churn,
                "churn_terms": r.churn_terms, "qsa": r.qsa, "r_q": r.r_q, "qsa_terms": r.qsa_terms,
                "tier_mass": np.array(list(r.tier_mass)), "lir_eligible": r.lir_eligible,
                "lir_rescued": r.lir_rescued, "lir_fullkv_eligible": r.lir_fullkv_eligible,
                "lir_fullkv_rescued": r.lir_fullkv_rescued, "lag": np.array(list(r.lag)).reshape(8, 2, 2)}

    def close(self):
        if self.handle:
            load().qevict_diag_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
