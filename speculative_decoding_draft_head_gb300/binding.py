"""Thin ctypes binding of libdspark (argument marshalling only).

Every function checks shapes, dtypes, devices and contiguity of torch tensors,
allocates missing outputs and workspaces with torch, and calls the C entry
point of the same name on the current CUDA stream.  No step of the method runs
in Python.  If the library cannot be loaded the functions raise: there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

DSPARK_OK = 0
DSPARK_BF16 = 0
DSPARK_F32 = 1
WS_DRAFT, WS_SCHEDULE, WS_VERIFY, WS_DRAFT_RNN = 0, 1, 2, 3

FLAG_BAD_TOKEN = 1
FLAG_BAD_TEMPERATURE = 2
FLAG_BAD_VERIFY_LEN = 4
FLAG_BAD_POS_TEMP = 8
FLAG_TIMEOUT = 16
FLAG_BAD_TARGET_ROW = 32

EXPORTS = ("dspark_version", "dspark_last_error", "dspark_workspace_bytes", "dspark_draft_sample",
           "dspark_schedule_prefix", "dspark_schedule_policy", "dspark_verify", "dspark_read_device_flags",
           "dspark_verify_noalloc", "dspark_draft_sample_rnn", "dspark_verify_packed", "dspark_pack_target",
           "dspark_selftest_bounded_wait", "dspark_read_noalloc_flags", "dspark_selftest_philox_rate")

_lib = None
_lock = threading.Lock()


class DSparkError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("dspark status %d: %s" % (status, message))
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libdspark.so (building it first when missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build_library()
        if not os.path.exists(path):
            raise RuntimeError("libdspark.so not built: run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        vp, i32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
        L.dspark_version.restype = ctypes.c_int
        L.dspark_version.argtypes = []
        L.dspark_last_error.restype = ctypes.c_char_p
        L.dspark_last_error.argtypes = []
        L.dspark_workspace_bytes.restype = sz
        L.dspark_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        L.dspark_draft_sample.restype = ctypes.c_int
        L.dspark_draft_sample.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, u64,
                                          vp, vp, vp, vp, vp, sz, vp]
        L.dspark_draft_sample_rnn.restype = ctypes.c_int
        L.dspark_draft_sample_rnn.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, u64,
                                              vp, vp, vp, vp, vp, vp, sz, vp]
        L.dspark_schedule_prefix.restype = ctypes.c_int
        L.dspark_schedule_prefix.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                             vp, sz, vp]
        L.dspark_schedule_policy.restype = ctypes.c_int
        L.dspark_schedule_policy.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, ctypes.c_float,
                                             vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.dspark_verify.restype = ctypes.c_int
        L.dspark_verify.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                    i32, i32, i32, i32, i32, u64, vp, vp, vp, vp, vp, vp, sz, vp]
        L.dspark_verify_packed.restype = ctypes.c_int
        L.dspark_verify_packed.argtypes = [vp, vp, ctypes.c_int64] + L.dspark_verify.argtypes[1:]
        L.dspark_selftest_bounded_wait.restype = ctypes.c_int
        L.dspark_selftest_bounded_wait.argtypes = [ctypes.c_uint, ctypes.POINTER(ctypes.c_uint32), vp]
        L.dspark_pack_target.restype = ctypes.c_int
        L.dspark_pack_target.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
        L.dspark_verify_noalloc.restype = ctypes.c_int
        L.dspark_verify_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            i32, i32, i32, i32, i32, u64, vp, vp, vp, vp, vp, vp]
        L.dspark_read_device_flags.restype = ctypes.c_int
        L.dspark_read_device_flags.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        L.dspark_selftest_philox_rate.restype = ctypes.c_int
        L.dspark_selftest_philox_rate.argtypes = [vp, sz, i32, ctypes.POINTER(ctypes.c_double), vp]
        L.dspark_read_noalloc_flags.restype = ctypes.c_int
        L.dspark_read_noalloc_flags.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        _lib = L
        return L


def _check(status):
    if status != DSPARK_OK:
        raise DSparkError(status, load().dspark_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return DSPARK_BF16
    if t.dtype == torch.float32:
        return DSPARK_F32
    raise TypeError("logits must be bfloat16 or float32, got %s" % t.dtype)


def _need(t, name, dtype=None, shape=None, device=None):
    if t is None:
        raise ValueError("%s is required" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _rid(request_id, B, device):
    if request_id is None:
        return None
    rid = request_id
    if rid.dtype not in (torch.int32,):
        raise TypeError("request_id must be int32 storage of uint32 ids")
    return _need(rid, "request_id", shape=(B,), device=device)


def version() -> int:
    return int(load().dspark_version())


def workspace_bytes(which: int, B: int, G: int, V: int, r: int) -> int:
    return int(load().dspark_workspace_bytes(which, B, G, V, r))


class WorkspaceCache:
    """Device scratch buffers reused across calls of the same shape."""

    def __init__(self):
        self._bufs = {}

    def get(self, which, B, G, V, r, device):
        n = workspace_bytes(which, B, G, V, r)
        if n == 0:
            raise ValueError("invalid sizes for a workspace")
        key = (which, device)
        buf = self._bufs.get(key)
        if buf is None or buf.numel() < n:
            buf = torch.empty(n + 256, dtype=torch.uint8, device=device)
            self._bufs[key] = buf
        off = (-buf.data_ptr()) % 256
        return buf[off:off + n]


_default_ws = WorkspaceCache()


def draft_sample(base, e_in, w_out, anchor, temperature, request_id=None, seed=0, *,
                 out=None, store_logits=False, workspace=None, stream=None):
    """Draft one block per request.  Returns dict(tokens, lse, logq[, logits])."""
    lib = load()
    B, G, V = base.shape
    r = e_in.shape[1]
    dev = base.device
    _need(base, "base", shape=(B, G, V), device=dev)
    _need(e_in, "e_in", dtype=base.dtype, shape=(V, r), device=dev)
    _need(w_out, "w_out", dtype=base.dtype, shape=(V, r), device=dev)
    _need(anchor, "anchor", dtype=torch.int32, shape=(B,), device=dev)
    _need(temperature, "temperature", dtype=torch.float32, shape=(B,), device=dev)
    rid = _rid(request_id, B, dev)
    if out is None:
        out = dict(tokens=torch.empty((B, G), dtype=torch.int32, device=dev),
                   lse=torch.empty((B, G), dtype=torch.float32, device=dev),
                   logq=torch.empty((B, G), dtype=torch.float32, device=dev))
        if store_logits:
            out["logits"] = torch.empty((B, G, V), dtype=torch.float32, device=dev)
    ws = workspace if workspace is not None else _default_ws.get(WS_DRAFT, B, G, V, r, dev)
    _check(lib.dspark_draft_sample(
        _ptr(base), _ptr(e_in), _ptr(w_out), _ptr(anchor), _ptr(temperature), _ptr(rid),
        B, G, V, r, _dtype_code(base), int(seed) & 0xFFFFFFFFFFFFFFFF,
        _ptr(out["tokens"]), _ptr(out["lse"]), _ptr(out["logq"]), _ptr(out.get("logits")),
        _ptr(ws), ws.numel(), _stream(stream)))
    return out


def draft_sample_rnn(base, e_in, w_h, w_out, anchor, temperature, request_id=None, seed=0, *,
                     out=None, store_logits=False, store_states=False, workspace=None, stream=None):
    """Draft one block per request with the recurrent head (bf16 weights).

    Returns dict(tokens, lse, logq[, logits][, h]); ``h`` [B,G,r] bf16 are the
    states h_j.  Verify the block with :func:`verify` and ``draft_logits``."""
    lib = load()
    B, G, V = base.shape
    r = e_in.shape[1]
    dev = base.device
    _need(base, "base", dtype=torch.bfloat16, shape=(B, G, V), device=dev)
    _need(e_in, "e_in", dtype=torch.bfloat16, shape=(V, r), device=dev)
    _need(w_h, "w_h", dtype=torch.bfloat16, shape=(r, r), device=dev)
    _need(w_out, "w_out", dtype=torch.bfloat16, shape=(V, r), device=dev)
    _need(anchor, "anchor", dtype=torch.int32, shape=(B,), device=dev)
    _need(temperature, "temperature", dtype=torch.float32, shape=(B,), device=dev)
    rid = _rid(request_id, B, dev)
    if out is None:
        out = dict(tokens=torch.empty((B, G), dtype=torch.int32, device=dev),
                   lse=torch.empty((B, G), dtype=torch.float32, device=dev),
                   logq=torch.empty((B, G), dtype=torch.float32, device=dev))
        if store_logits:
            out["logits"] = torch.empty((B, G, V), dtype=torch.float32, device=dev)
        if store_states:
            out["h"] = torch.empty((B, G, r), dtype=torch.bfloat16, device=dev)
    ws = workspace if workspace is not None else _default_ws.get(WS_DRAFT_RNN, B, G, V, r, dev)
    _check(lib.dspark_draft_sample_rnn(
        _ptr(base), _ptr(e_in), _ptr(w_h), _ptr(w_out), _ptr(anchor), _ptr(temperature), _ptr(rid),
        B, G, V, r, DSPARK_BF16, int(seed) & 0xFFFFFFFFFFFFFFFF,
        _ptr(out["tokens"]), _ptr(out["lse"]), _ptr(out["logq"]), _ptr(out.get("logits")),
        _ptr(out.get("h")), _ptr(ws), ws.numel(), _stream(stream)))
    return out


# verify-length policies of dspark_schedule_policy
SCHED_EARLY_STOP, SCHED_BEST_PREFIX, SCHED_THRESHOLD_CUM, SCHED_THRESHOLD_CONF = 0, 1, 2, 3


def schedule_prefix(conf_logits, pos_temp, sps, L_min, L_max, *, policy=SCHED_EARLY_STOP, threshold=0.0,
                    out=None, workspace=None, stream=None):
    """Calibrate confidences and choose verify lengths (early stop by default;
    ``policy`` selects another rule of dspark_schedule_policy).

    Returns dict(conf, cum_conf, verify_len, theta)."""
    lib = load()
    B, G = conf_logits.shape
    dev = conf_logits.device
    _need(conf_logits, "conf_logits", dtype=torch.float32, device=dev)
    _need(pos_temp, "pos_temp", dtype=torch.float32, shape=(G,), device=dev)
    _need(sps, "sps", dtype=torch.float32, device=dev)
    if out is None:
        out = dict(conf=torch.empty((B, G), dtype=torch.float32, device=dev),
                   cum_conf=torch.empty((B, G), dtype=torch.float32, device=dev),
                   verify_len=torch.empty((B,), dtype=torch.int32, device=dev),
                   theta=torch.empty((1,), dtype=torch.float64, device=dev))
    ws = workspace if workspace is not None else _default_ws.get(WS_SCHEDULE, B, G, 8, 1, dev)
    _check(lib.dspark_schedule_policy(
        _ptr(conf_logits), _ptr(pos_temp), _ptr(sps), sps.numel(), B, G, int(L_min), int(L_max),
        int(policy), float(threshold),
        _ptr(out["conf"]), _ptr(out["cum_conf"]), _ptr(out["verify_len"]), _ptr(out.get("theta")),
        _ptr(ws), ws.numel(), _stream(stream)))
    return out


class LaggedScheduler:
    """The deployed scheduling mode: round t's verify lengths come from the
    calibrated confidences of round t - ``lag`` ("DSpark, la bozza che sa quando
    fermarsi", section "Che cosa resta da verificare": the production scheduler
    works from confidences two rounds old and has no early stop), so the
    schedule need not wait for the current round's confidence head.

    Keeps a device ring of the last ``lag`` rounds' confidence logits [B, G];
    until it has filled, a round is scheduled from its own logits.  Each
    :meth:`step` runs one dspark_schedule_policy launch (policy ``policy``,
    best prefix by default) and returns its outputs."""

    def __init__(self, pos_temp, sps, L_min, L_max, *, lag=2, policy=SCHED_BEST_PREFIX, threshold=0.0):
        if lag < 0:
            raise ValueError("lag must be >= 0")
        self.pos_temp, self.sps = pos_temp, sps
        self.L_min, self.L_max = int(L_min), int(L_max)
        self.lag, self.policy, self.threshold = int(lag), int(policy), float(threshold)
        self._ring = []

    def step(self, conf_logits, *, out=None, stream=None):
        """Schedule this round; ``conf_logits`` [B, G] are this round's logits."""
        src = self._ring[0] if len(self._ring) == self.lag and self.lag > 0 else conf_logits
        res = schedule_prefix(src, self.pos_temp, self.sps, self.L_min, self.L_max, policy=self.policy,
                              threshold=self.threshold, out=out, stream=stream)
        if self.lag > 0:
            self._ring.append(conf_logits.clone())
            if len(self._ring) > self.lag:
                self._ring.pop(0)
        return res


def verify(target, base, e_in, w_out, anchor, draft, verify_len, temperature, request_id=None,
           seed=0, *, draft_logits=None, target_row0=None, out=None, workspace=None, stream=None):
    """Verify one drafted block per request.

    ``draft`` is the dict returned by :func:`draft_sample`.  ``target`` is
    [B, G+1, V], or with ``target_row0`` ([B] int64) the packed rows [n, V]
    (request b's row j at row target_row0[b] + j, see dspark_verify_packed).
    Returns dict(accept_len, out_tokens, num_out, target_lse, logp)."""
    lib = load()
    B, G = draft["tokens"].shape
    V = target.shape[-1]
    dev = target.device
    if target_row0 is None:
        _need(target, "target", shape=(B, G + 1, V), device=dev)
    else:
        _need(target, "target", device=dev)
        if target.dim() != 2:
            raise ValueError("a packed target is [rows, V]")
        _need(target_row0, "target_row0", dtype=torch.int64, shape=(B,), device=dev)
    if draft_logits is None:
        _need(base, "base", dtype=target.dtype, shape=(B, G, V), device=dev)
        _need(e_in, "e_in", dtype=target.dtype, device=dev)
        _need(w_out, "w_out", dtype=target.dtype, device=dev)
        r = e_in.shape[1]
    else:
        _need(draft_logits, "draft_logits", dtype=torch.float32, shape=(B, G, V), device=dev)
        r = e_in.shape[1] if e_in is not None else 16
    _need(anchor, "anchor", dtype=torch.int32, shape=(B,), device=dev)
    for k in ("tokens", "lse", "logq"):
        _need(draft[k], "draft." + k, shape=(B, G), device=dev)
    if verify_len is not None:
        _need(verify_len, "verify_len", dtype=torch.int32, shape=(B,), device=dev)
    _need(temperature, "temperature", dtype=torch.float32, shape=(B,), device=dev)
    rid = _rid(request_id, B, dev)
    if out is None:
        out = dict(accept_len=torch.empty((B,), dtype=torch.int32, device=dev),
                   out_tokens=torch.empty((B, G + 1), dtype=torch.int32, device=dev),
                   num_out=torch.empty((B,), dtype=torch.int32, device=dev),
                   target_lse=torch.empty((B, G + 1), dtype=torch.float32, device=dev),
                   logp=torch.empty((B, G), dtype=torch.float32, device=dev))
    ws = workspace if workspace is not None else _default_ws.get(WS_VERIFY, B, G, V, r, dev)
    args = (_ptr(base), _ptr(e_in), _ptr(w_out), _ptr(draft_logits), _ptr(anchor),
            _ptr(draft["tokens"]), _ptr(draft["lse"]), _ptr(draft["logq"]), _ptr(verify_len),
            _ptr(temperature), _ptr(rid), B, G, V, r, _dtype_code(target),
            int(seed) & 0xFFFFFFFFFFFFFFFF,
            _ptr(out["accept_len"]), _ptr(out["out_tokens"]), _ptr(out["num_out"]),
            _ptr(out.get("target_lse")), _ptr(out.get("logp")), _ptr(ws), ws.numel(),
            _stream(stream))
    if target_row0 is None:
        _check(lib.dspark_verify(_ptr(target), *args))
    else:
        _check(lib.dspark_verify_packed(_ptr(target), _ptr(target_row0), target.shape[0], *args))
    return out


def pack_target(target, verify_len, *, out=None, stream=None):
    """Rows 0 .. L_b of every request of ``target`` [B, G+1, V] (device, or
    pinned host memory, which the device reads directly) packed for
    :func:`verify` with ``target_row0`` (dspark_pack_target).

    Returns dict(target [B*(G+1), V] with the packed rows first, row0 [B]
    int64, n_rows [1] int64), all on the device of ``verify_len``."""
    lib = load()
    B, G1, V = target.shape
    dev = verify_len.device if verify_len is not None else torch.device("cuda", torch.cuda.current_device())
    if not target.is_contiguous():
        raise ValueError("target must be contiguous")
    if target.device.type == "cpu" and not target.is_pinned():
        raise ValueError("a host target must be in pinned memory")
    if verify_len is not None:
        _need(verify_len, "verify_len", dtype=torch.int32, shape=(B,), device=dev)
    if out is None:
        out = dict(target=torch.empty((B * G1, V), dtype=target.dtype, device=dev),
                   row0=torch.empty((B,), dtype=torch.int64, device=dev),
                   n_rows=torch.empty((1,), dtype=torch.int64, device=dev))
    _check(lib.dspark_pack_target(_ptr(target), _ptr(verify_len), B, G1 - 1, V, _dtype_code(target),
                                  _ptr(out["target"]), _ptr(out["row0"]), _ptr(out.get("n_rows")),
                                  _stream(stream)))
    return out


NOALLOC_SCRATCH_BYTES = 4 << 20


def verify_noalloc(target, base, e_in, w_out, anchor, draft, verify_len, temperature,
                   request_id=None, seed=0, *, draft_logits=None, out=None, stream=None):
    """:func:`verify` through ``dspark_verify_noalloc``: no workspace is passed
    or allocated; the library uses its fixed device scratch array."""
    lib = load()
    B, G1, V = target.shape
    G = G1 - 1
    dev = target.device
    _need(target, "target", device=dev)
    r = e_in.shape[1] if e_in is not None else 16
    if out is None:
        out = dict(accept_len=torch.empty((B,), dtype=torch.int32, device=dev),
                   out_tokens=torch.empty((B, G + 1), dtype=torch.int32, device=dev),
                   num_out=torch.empty((B,), dtype=torch.int32, device=dev),
                   target_lse=torch.empty((B, G + 1), dtype=torch.float32, device=dev),
                   logp=torch.empty((B, G), dtype=torch.float32, device=dev))
    rid = _rid(request_id, B, dev)
    _check(lib.dspark_verify_noalloc(
        _ptr(target), _ptr(base), _ptr(e_in), _ptr(w_out), _ptr(draft_logits), _ptr(anchor),
        _ptr(draft["tokens"]), _ptr(draft["lse"]), _ptr(draft["logq"]), _ptr(verify_len),
        _ptr(temperature), _ptr(rid), B, G, V, r, _dtype_code(target),
        int(seed) & 0xFFFFFFFFFFFFFFFF,
        _ptr(out["accept_len"]), _ptr(out["out_tokens"]), _ptr(out["num_out"]),
        _ptr(out.get("target_lse")), _ptr(out.get("logp")), _stream(stream)))
    return out


def selftest_bounded_wait(limit_us=1000, stream=None) -> int:
    """Run dspark_selftest_bounded_wait: 3 when both probe waits report their
    timeout."""
    val = ctypes.c_uint32(0)
    _check(load().dspark_selftest_bounded_wait(int(limit_us), ctypes.byref(val), _stream(stream)))
    return int(val.value)


def selftest_philox_rate(iters=2048, stream=None) -> float:
    """Philox4x32-10 blocks per second of the draft's word code on this
    device (dspark_selftest_philox_rate)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    sink = torch.empty(1 << 16, dtype=torch.uint8, device=dev)
    val = ctypes.c_double(0.0)
    _check(load().dspark_selftest_philox_rate(_ptr(sink), sink.numel(), int(iters), ctypes.byref(val),
                                              _stream(stream)))
    return float(val.value)


def read_device_flags(workspace, stream=None) -> int:
    val = ctypes.c_uint32(0)
    _check(load().dspark_read_device_flags(_ptr(workspace), _stream(stream), ctypes.byref(val)))
    return int(val.value)


def read_noalloc_flags(stream=None) -> int:
    """The flag word of the last :func:`verify_noalloc` call."""
    val = ctypes.c_uint32(0)
    _check(load().dspark_read_noalloc_flags(_stream(stream), ctypes.byref(val)))
    return int(val.value)


def default_workspace(which, B, G, V, r, device):
    return _default_ws.get(which, B, G, V, r, device)
