"""Python binding of librx.so (the C ABI in include/rx.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  Import
fails loudly when the library has not been built -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librx.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        "librx.so is not built (expected at %s); run `python -c \"import __graft_entry__ as g; "
        "g.build()\"` or `python -m partitioned_kv_cache_gb300.build`" % _LIB_PATH)
_lib = ctypes.CDLL(_LIB_PATH)

RX_OK = 0
STATUS_NAMES = {0: "RX_OK", -1: "RX_ERR_ARG", -2: "RX_ERR_LAYER", -3: "RX_ERR_CAPACITY",
                -4: "RX_ERR_CUDA", -5: "RX_ERR_TIMEOUT", -6: "RX_ERR_UNSUPPORTED",
                -7: "RX_ERR_STATE"}

#: Every symbol include/rx.h declares.
EXPORTS = ("rx_cache_create", "rx_cache_destroy", "rx_pin_prefix", "rx_push_frame",
           "rx_attend_suffix", "rx_attend_batch", "rx_ada_gamma", "rx_adarmsnorm",
           "rx_get_state", "rx_debug_window", "rx_export_window", "rx_check_device_error",
           "rx_set_attn_splits", "rx_launch_count", "rx_status_str", "rx_last_error",
           "rx_attend_regions_static", "rx_attend_suffix_block_causal", "rx_tail_append",
           "rx_snapshot_bytes", "rx_snapshot", "rx_restore", "rx_push_frame_async",
           "rx_set_attn_dparts", "rx_debug_inject_timeout", "rx_debug_choose_partition",
           "rx_attend_suffix_norms", "rx_attend_batch_norms")


class RxConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("L", "Hq", "Hkv", "D", "P_cap", "N", "F", "S_cap", "tail_cap", "max_req",
                 "spare_slot")]


class RxStreamBatch(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_tail", ctypes.c_void_p), ("v_tail", ctypes.c_void_p),
                ("tail_len", ctypes.c_void_p), ("out", ctypes.c_void_p), ("B", ctypes.c_int),
                ("T", ctypes.c_int)]


class RxNormRows(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("rows", ctypes.c_int), ("d", ctypes.c_int), ("eps", ctypes.c_float)]


MAX_NORM_JOBS = 2

_vp, _i, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
_sigs = {
    "rx_cache_create": (_i, [ctypes.POINTER(RxConfig), ctypes.POINTER(_vp)]),
    "rx_cache_destroy": (_i, [_vp]),
    "rx_pin_prefix": (_i, [_vp, _vp, _vp, _i, _vp]),
    "rx_push_frame": (_i, [_vp, _vp, _vp, ctypes.POINTER(_i), _vp]),
    "rx_attend_suffix": (_i, [_vp, _i, _vp, _vp, _vp, _i, _vp, _vp]),
    "rx_attend_batch": (_i, [_vp, _i, _vp, _vp, _vp, _i, _vp, ctypes.POINTER(RxStreamBatch), _vp]),
    "rx_ada_gamma": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _i, _vp, _vp, _i, _i, _vp, _vp]),
    "rx_adarmsnorm": (_i, [_vp, _vp, _i, _i, _f, _vp, _vp]),
    "rx_get_state": (_i, [_vp, ctypes.POINTER(_i), ctypes.POINTER(_i),
                          ctypes.POINTER(ctypes.c_longlong), _vp]),
    "rx_debug_window": (_i, [_vp, ctypes.POINTER(_i), ctypes.POINTER(_i), _vp]),
    "rx_export_window": (_i, [_vp, _i, _vp, _vp, _vp]),
    "rx_check_device_error": (_i, [_vp, ctypes.POINTER(_i), _vp]),
    "rx_set_attn_splits": (_i, [_vp, _i]),
    "rx_set_attn_dparts": (_i, [_vp, _i]),
    "rx_debug_inject_timeout": (_i, [_vp, _i]),
    "rx_debug_choose_partition": (_i, [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_i),
                                       ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    "rx_launch_count": (ctypes.c_longlong, []),
    "rx_status_str": (ctypes.c_char_p, [_i]),
    "rx_last_error": (ctypes.c_char_p, []),
    "rx_attend_regions_static": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _i, _vp, _vp, _i,
                                      _vp, _vp, _i, _vp, _vp]),
    "rx_attend_suffix_block_causal": (_i, [_vp, _i, _vp, _vp, _vp, _i, _i, _vp, _vp]),
    "rx_tail_append": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "rx_snapshot_bytes": (_i, [_vp, ctypes.POINTER(ctypes.c_longlong)]),
    "rx_snapshot": (_i, [_vp, _vp, _vp]),
    "rx_restore": (_i, [_vp, _vp, _vp]),
    "rx_push_frame_async": (_i, [_vp, _vp, _vp, ctypes.POINTER(_i), _vp, _vp]),
    "rx_attend_suffix_norms": (_i, [_vp, _i, _vp, _vp, _vp, _i, _vp, ctypes.POINTER(RxNormRows), _i, _vp]),
    "rx_attend_batch_norms": (_i, [_vp, _i, _vp, _vp, _vp, _i, _vp, ctypes.POINTER(RxStreamBatch),
                                   ctypes.POINTER(RxNormRows), _i, _vp]),
}
for _name, (_res, _args) in _sigs.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class RxError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.rx_last_error().decode(errors="replace")
        super().__init__("%s failed: %s: %s" % (where, STATUS_NAMES.get(status, status), msg))


def _check(status: int, where: str) -> None:
    if status != RX_OK:
        raise RxError(status, where)


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor], dtype=torch.bfloat16, name: str = "tensor",
         device: bool = True) -> Optional[int]:
    if t is None:
        return None
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if device and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    return t.data_ptr()


def _shape(t: Optional[torch.Tensor], shape, name: str) -> None:
    """Refuse a tensor whose shape differs from the one the library will
    assume from the sizes it is given (it would read or write past the
    caller's buffer)."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _norm_jobs(norms) -> Tuple[Optional[ctypes.Array], int]:
    """norms: a sequence of (x [rows][d] bf16, gamma [d] fp32, eps, y [rows][d]
    bf16) -> the C array of rx_norm_rows (or None) and its length."""
    if not norms:
        return None, 0
    if len(norms) > MAX_NORM_JOBS:
        raise ValueError("at most %d norm jobs per launch" % MAX_NORM_JOBS)
    arr = (RxNormRows * len(norms))()
    for i, (x, gamma, eps, y) in enumerate(norms):
        rows, d = x.shape
        _shape(gamma, (d,), "gamma")
        _shape(y, x.shape, "y")
        arr[i] = RxNormRows(_ptr(x, name="x"), _ptr(gamma, torch.float32, "gamma"), _ptr(y, name="y"),
                            rows, d, float(eps))
    return arr, len(norms)


def launch_count() -> int:
    return int(_lib.rx_launch_count())


def choose_partition(t_max: int, units: int, D: int, num_sms: int, max_splits: int,
                     cluster_capacity, splits: int = 0, dparts: int = 0):
    """Test aid: (splits, dparts, fused) of an attention launch, computed on
    the host from the given device figures (rx_debug_choose_partition).
    cluster_capacity: 17 ints, entry c = clusters of c CTAs the device holds."""
    cap = (_i * 17)(*[int(c) for c in cluster_capacity])
    sp, dp, fu = _i(0), _i(0), _i(0)
    _check(_lib.rx_debug_choose_partition(t_max, units, D, num_sms, max_splits, splits, dparts, cap,
                                          ctypes.byref(sp), ctypes.byref(dp), ctypes.byref(fu)),
           "rx_debug_choose_partition")
    return sp.value, dp.value, bool(fu.value)


def library_path() -> str:
    return _LIB_PATH


class Cache:
    """The partitioned KV store of one stream (rx_cache_t)."""

    def __init__(self, L: int, Hq: int, Hkv: int, D: int, P_cap: int, N: int, F: int,
                 S_cap: int, tail_cap: int = 0, max_req: int = 0, spare_slot: int = 0):
        self.cfg = RxConfig(L, Hq, Hkv, D, P_cap, N, F, S_cap, tail_cap, max_req, spare_slot)
        h = _vp()
        _check(_lib.rx_cache_create(ctypes.byref(self.cfg), ctypes.byref(h)), "rx_cache_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self) -> None:
        if getattr(self, "_h", None):
            _check(_lib.rx_cache_destroy(self._h), "rx_cache_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def pin_prefix(self, k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
        c = self.cfg
        P = k.shape[1]
        _shape(k, (c.L, P, c.Hkv, c.D), "k")
        _shape(v, k.shape, "v")
        _check(_lib.rx_pin_prefix(self._h, _ptr(k, name="k", device=False),
                                  _ptr(v, name="v", device=False), P, _stream(stream)),
               "rx_pin_prefix")

    def _frame_shape(self, k: torch.Tensor, v: torch.Tensor) -> None:
        c = self.cfg
        _shape(k, (c.L, c.F, c.Hkv, c.D), "k")
        _shape(v, k.shape, "v")

    def push_frame(self, k: torch.Tensor, v: torch.Tensor, stream=None) -> int:
        self._frame_shape(k, v)
        ev = _i(0)
        _check(_lib.rx_push_frame(self._h, _ptr(k, name="k"), _ptr(v, name="v"),
                                  ctypes.byref(ev), _stream(stream)), "rx_push_frame")
        return ev.value

    def push_frame_async(self, k: torch.Tensor, v: torch.Tensor, producer_stream,
                         consumer_stream) -> int:
        """Push on producer_stream, concurrent with attention on consumer_stream
        (needs spare_slot=1)."""
        self._frame_shape(k, v)
        ev = _i(0)
        _check(_lib.rx_push_frame_async(self._h, _ptr(k, name="k"), _ptr(v, name="v"), ctypes.byref(ev),
                                        producer_stream.cuda_stream, consumer_stream.cuda_stream),
               "rx_push_frame_async")
        return ev.value

    def attend_suffix(self, layer: int, q: torch.Tensor, k_dyn: torch.Tensor, v_dyn: torch.Tensor,
                      out: Optional[torch.Tensor] = None, stream=None,
                      n_state: Optional[int] = None, norms=None) -> torch.Tensor:
        """Eq. 1 for one layer; with n_state, the block-causal variant (the
        first n_state suffix tokens see only their own dynamic keys); with
        norms, a list of up to two (x, gamma, eps, y) AdaRMSNorm jobs run in
        the same launch (rx_attend_suffix_norms)."""
        c = self.cfg
        S = q.shape[0]
        _shape(q, (S, c.Hq, c.D), "q")
        _shape(k_dyn, (S, c.Hkv, c.D), "k_dyn")
        _shape(v_dyn, (S, c.Hkv, c.D), "v_dyn")
        _shape(out, q.shape, "out")
        if out is None:
            out = torch.empty_like(q)
        if norms:
            if n_state is not None:
                raise ValueError("norm jobs run with the plain Eq. 1 call only")
            arr, n = _norm_jobs(norms)
            _check(_lib.rx_attend_suffix_norms(self._h, layer, _ptr(q, name="q"), _ptr(k_dyn, name="k_dyn"),
                                               _ptr(v_dyn, name="v_dyn"), S, _ptr(out, name="out"), arr, n,
                                               _stream(stream)), "rx_attend_suffix_norms")
        elif n_state is None:
            _check(_lib.rx_attend_suffix(self._h, layer, _ptr(q, name="q"), _ptr(k_dyn, name="k_dyn"),
                                         _ptr(v_dyn, name="v_dyn"), S, _ptr(out, name="out"),
                                         _stream(stream)), "rx_attend_suffix")
        else:
            _check(_lib.rx_attend_suffix_block_causal(
                self._h, layer, _ptr(q, name="q"), _ptr(k_dyn, name="k_dyn"), _ptr(v_dyn, name="v_dyn"),
                S, int(n_state), _ptr(out, name="out"), _stream(stream)), "rx_attend_suffix_block_causal")
        return out

    def snapshot_bytes(self) -> int:
        n = ctypes.c_longlong(0)
        _check(_lib.rx_snapshot_bytes(self._h, ctypes.byref(n)), "rx_snapshot_bytes")
        return n.value

    def snapshot(self, dst: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """Copy the cache's state into a uint8 CUDA tensor (allocated if not given)."""
        if dst is None:
            dst = torch.empty(self.snapshot_bytes(), dtype=torch.uint8, device="cuda")
        _check(_lib.rx_snapshot(self._h, _ptr(dst, torch.uint8, "dst"), _stream(stream)), "rx_snapshot")
        return dst

    def restore(self, src: torch.Tensor, stream=None) -> None:
        _check(_lib.rx_restore(self._h, _ptr(src, torch.uint8, "src"), _stream(stream)), "rx_restore")

    def attend_batch(self, layer: int, action=None, lang=None, out_act: Optional[torch.Tensor] = None,
                     out_lang: Optional[torch.Tensor] = None, stream=None, norms=None):
        """One launch for an action suffix and a batch of language streams.

        action: (q [S][Hq][D], k_dyn [S][Hkv][D], v_dyn) or None.
        lang: (q [B][T][Hq][D], k_tail [B][tail_cap][Hkv][D], v_tail,
               tail_len int32 CUDA tensor [B]) or None.
        norms: up to two (x, gamma, eps, y) AdaRMSNorm jobs run in the same
               launch (rx_attend_batch_norms).
        Returns (out_act or None, out_lang or None).
        """
        c = self.cfg
        S, qa, kd, vd = 0, None, None, None
        if action is not None:
            qa, kd, vd = action
            S = qa.shape[0]
            _shape(qa, (S, c.Hq, c.D), "q")
            _shape(kd, (S, c.Hkv, c.D), "k_dyn")
            _shape(vd, (S, c.Hkv, c.D), "v_dyn")
            _shape(out_act, qa.shape, "out_act")
            if out_act is None:
                out_act = torch.empty_like(qa)
        batch = None
        if lang is not None:
            ql, kt, vt, tl = lang
            B = ql.shape[0]
            _shape(ql, (B, ql.shape[1] if ql.dim() > 1 else 0, c.Hq, c.D), "q_lang")
            _shape(kt, (B, c.tail_cap, c.Hkv, c.D), "k_tail")
            _shape(vt, kt.shape, "v_tail")
            _shape(tl, (B,), "tail_len")
            _shape(out_lang, ql.shape, "out_lang")
            if out_lang is None:
                out_lang = torch.empty_like(ql)
            batch = RxStreamBatch(_ptr(ql, name="q_lang"), _ptr(kt, name="k_tail"),
                                  _ptr(vt, name="v_tail"), _ptr(tl, torch.int32, "tail_len"),
                                  _ptr(out_lang, name="out_lang"), ql.shape[0], ql.shape[1])
        if norms:
            arr, n = _norm_jobs(norms)
            _check(_lib.rx_attend_batch_norms(self._h, layer, _ptr(qa, name="q"), _ptr(kd, name="k_dyn"),
                                              _ptr(vd, name="v_dyn"), S, _ptr(out_act, name="out_act"),
                                              ctypes.byref(batch) if batch is not None else None,
                                              arr, n, _stream(stream)), "rx_attend_batch_norms")
        else:
            _check(_lib.rx_attend_batch(self._h, layer, _ptr(qa, name="q"), _ptr(kd, name="k_dyn"),
                                        _ptr(vd, name="v_dyn"), S, _ptr(out_act, name="out_act"),
                                        ctypes.byref(batch) if batch is not None else None,
                                        _stream(stream)), "rx_attend_batch")
        return (out_act if action is not None else None), (out_lang if lang is not None else None)

    def get_state(self, stream=None) -> Tuple[int, int, int]:
        h, v, p = _i(0), _i(0), ctypes.c_longlong(0)
        _check(_lib.rx_get_state(self._h, ctypes.byref(h), ctypes.byref(v), ctypes.byref(p),
                                 _stream(stream)), "rx_get_state")
        return h.value, v.value, p.value

    def debug_window(self, stream=None) -> List[int]:
        slots = (_i * self.cfg.N)()
        valid = _i(0)
        _check(_lib.rx_debug_window(self._h, slots, ctypes.byref(valid), _stream(stream)),
               "rx_debug_window")
        return [slots[i] for i in range(valid.value)]

    def export_window(self, layer: int, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        valid = len(self.debug_window(stream))
        c = self.cfg
        k = torch.empty((valid * c.F, c.Hkv, c.D), dtype=torch.bfloat16, device="cuda")
        v = torch.empty_like(k)
        if valid:
            _check(_lib.rx_export_window(self._h, layer, _ptr(k), _ptr(v), _stream(stream)),
                   "rx_export_window")
        return k, v

    def check_device_error(self, stream=None) -> int:
        code = _i(0)
        _check(_lib.rx_check_device_error(self._h, ctypes.byref(code), _stream(stream)),
               "rx_check_device_error")
        return code.value

    def set_attn_splits(self, splits: int) -> None:
        _check(_lib.rx_set_attn_splits(self._h, splits), "rx_set_attn_splits")

    def set_attn_dparts(self, dparts: int) -> None:
        _check(_lib.rx_set_attn_dparts(self._h, dparts), "rx_set_attn_dparts")

    def debug_inject_timeout(self, nbytes: int) -> None:
        """Test aid: the next attention launch's first CTA waits for nbytes
        that never arrive, so its bounded waits run out (see rx.h)."""
        _check(_lib.rx_debug_inject_timeout(self._h, nbytes), "rx_debug_inject_timeout")


def ada_gamma(t: torch.Tensor, state: torch.Tensor, W1: torch.Tensor, b1: torch.Tensor,
              W2: torch.Tensor, b2: torch.Tensor, emb_dim: int,
              out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """gamma [n_sets][n_cond][d] for weights W1 [n_sets][hidden][cond], W2 [n_sets][d][hidden]."""
    n_cond = t.shape[0]
    state_dim = state.shape[1] if state.dim() == 2 else 0
    n_sets, hidden, cond = W1.shape
    d = W2.shape[1]
    if cond != emb_dim + state_dim:
        raise ValueError("W1 input width %d != emb_dim + state_dim = %d" % (cond, emb_dim + state_dim))
    _shape(t, (n_cond,), "t")
    _shape(state, (n_cond, state_dim), "state")
    _shape(b1, (n_sets, hidden), "b1")
    _shape(W2, (n_sets, d, hidden), "W2")
    _shape(b2, (n_sets, d), "b2")
    _shape(out, (n_sets, n_cond, d), "gamma")
    if out is None:
        out = torch.empty((n_sets, n_cond, d), dtype=torch.float32, device=t.device)
    _check(_lib.rx_ada_gamma(_ptr(t, torch.float32, "t"), _ptr(state, torch.float32, "state"),
                             n_cond, emb_dim, state_dim, _ptr(W1, name="W1"), _ptr(b1, name="b1"),
                             hidden, _ptr(W2, name="W2"), _ptr(b2, name="b2"), d, n_sets,
                             _ptr(out, torch.float32, "gamma"), _stream(stream)), "rx_ada_gamma")
    return out


def adarmsnorm(x: torch.Tensor, gamma: torch.Tensor, eps: float,
               out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    rows, d = x.shape
    _shape(gamma, (d,), "gamma")
    _shape(out, x.shape, "y")
    if out is None:
        out = torch.empty_like(x)
    _check(_lib.rx_adarmsnorm(_ptr(x, name="x"), _ptr(gamma, torch.float32, "gamma"), rows, d,
                              float(eps), _ptr(out, name="y"), _stream(stream)), "rx_adarmsnorm")
    return out


def attend_regions_static(q: torch.Tensor, k_pin: Optional[torch.Tensor], v_pin: Optional[torch.Tensor],
                          k_win: Optional[torch.Tensor], v_win: Optional[torch.Tensor],
                          k_dyn: Optional[torch.Tensor], v_dyn: Optional[torch.Tensor],
                          out: torch.Tensor, stream=None) -> torch.Tensor:
    """Attention over caller-held regions through rx_attend_regions_static.

    For callers that cannot allocate device memory: the library allocates
    nothing on this path (its scratch is a fixed array inside librx.so), so
    `out` must be supplied.  Regions are [tokens][Hkv][D] bf16 or None.
    """
    S, Hq, D = q.shape
    regions = [(k_pin, v_pin), (k_win, v_win), (k_dyn, v_dyn)]
    for k, v in regions:
        if (k is None) != (v is None):
            raise ValueError("a region needs both its keys and its values (or neither)")
    Hkv = next((k.shape[1] for k, _ in regions if k is not None and k.dim() == 3), 1)
    for (k, v), name in zip(regions, ("pin", "win", "dyn")):
        if k is not None:
            _shape(k, (k.shape[0], Hkv, D), "k_" + name)
            _shape(v, k.shape, "v_" + name)
    _shape(out, q.shape, "out")
    counts = [0 if k is None else k.shape[0] for k, _ in regions]
    ptrs = [(_ptr(k, name="k") if n else None, _ptr(v, name="v") if n else None)
            for (k, v), n in zip(regions, counts)]
    _check(_lib.rx_attend_regions_static(_ptr(q, name="q"), S, Hq, Hkv, D,
                                         ptrs[0][0], ptrs[0][1], counts[0],
                                         ptrs[1][0], ptrs[1][1], counts[1],
                                         ptrs[2][0], ptrs[2][1], counts[2],
                                         _ptr(out, name="out"), _stream(stream)),
           "rx_attend_regions_static")
    return out


def tail_append(k_tail: torch.Tensor, v_tail: torch.Tensor, tail_len: torch.Tensor,
                k_new: torch.Tensor, v_new: torch.Tensor, active: Optional[torch.Tensor] = None,
                overflow: Optional[torch.Tensor] = None, stream=None) -> None:
    """Append one token per (active) stream: tails [B][tail_cap][Hkv][D],
    tail_len int32 [B] (advanced on the device), new tokens [B][Hkv][D]."""
    B, tail_cap, Hkv, D = k_tail.shape
    _shape(v_tail, k_tail.shape, "v_tail")
    _shape(tail_len, (B,), "tail_len")
    _shape(k_new, (B, Hkv, D), "k_new")
    _shape(v_new, (B, Hkv, D), "v_new")
    _shape(active, (B,), "active")
    if overflow is not None and overflow.numel() < 1:
        raise ValueError("overflow must hold one int32")
    _check(_lib.rx_tail_append(_ptr(k_tail, name="k_tail"), _ptr(v_tail, name="v_tail"),
                               _ptr(tail_len, torch.int32, "tail_len"), _ptr(k_new, name="k_new"),
                               _ptr(v_new, name="v_new"), _ptr(active, torch.int32, "active"), B,
                               tail_cap, Hkv, D, _ptr(overflow, torch.int32, "overflow"),
                               _stream(stream)), "rx_tail_append")
