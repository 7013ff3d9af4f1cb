"""Plain CPU oracle for the DSpark draft-sample / schedule / verify path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's ``cpu_baseline`` / reference leg may import this package.  The
product library never links, loads or calls it, and the oracle shares no code
with the CUDA kernels: the arithmetic lives in ``dspark_oracle.c`` (double
precision, written in the order the method states it) and this module only
marshals numpy arrays into it.

Parity status per function (what pins each one is listed in the test suite):
  philox4x32_10 / uniform / gumbel : pinned (cuRAND host generator, uniformity,
                                     range bounds)
  draft_sample                     : pinned (per-token Gumbel-max: argmax of the
                                     uniforms on constant rows, chi-square vs
                                     softmax over 10^6 draws, textbook matmul,
                                     Markov toy)
  schedule                         : pinned (brute force over length vectors,
                                     closed-form threshold, sigmoid identities)
  verify                           : pinned (1 - TV acceptance, expected tokens
                                     per pass, the exact output law by brute-force
                                     enumeration against 10^6 oracle rounds,
                                     residual and bonus laws, greedy limit)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _nullable(ptr_type):
    def from_param(obj):
        if obj is None:
            return None
        return ptr_type.from_param(obj)
    return type("Nullable", (), {"from_param": staticmethod(from_param)})


def lib():
    global _lib
    with _lock:
        if _lib is None:
            so = build()
            L = ctypes.CDLL(so)
            L.or_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
            L.or_philox4x32_10.restype = None
            L.or_random_word.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                         ctypes.c_uint32, ctypes.c_uint32]
            L.or_random_word.restype = ctypes.c_uint32
            L.or_uniform.argtypes = L.or_random_word.argtypes
            L.or_uniform.restype = ctypes.c_double
            L.or_gumbel.argtypes = L.or_random_word.argtypes
            L.or_gumbel.restype = ctypes.c_double
            L.or_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                      ctypes.c_uint32, ctypes.c_int, ctypes.c_uint32, _f64p]
            L.or_uniforms.restype = None
            nf = _nullable(_f64p)
            nu = _nullable(_u32p)
            ni = _nullable(_i32p)
            L.or_draft_sample.argtypes = [
                _f64p, _f64p, _f64p, _i32p, _f64p, nu,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
                _i32p, _f64p, _f64p, _f64p, _f64p, nf]
            L.or_draft_sample.restype = ctypes.c_int
            L.or_schedule.argtypes = [
                _f64p, _f64p, _f64p, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _f64p, _f64p, _i32p, _f64p, _i32p, _f64p, _f64p]
            L.or_schedule.restype = ctypes.c_int
            L.or_draft_sample_rnn.argtypes = [
                _f64p, _f64p, _f64p, _f64p, _i32p, _f64p, nu,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
                _i32p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, nf]
            L.or_draft_sample_rnn.restype = ctypes.c_int
            L.or_schedule_policy.argtypes = [
                _f64p, _f64p, _f64p, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                _f64p, _f64p, _i32p, _f64p, _i32p, _f64p, _f64p]
            L.or_schedule_policy.restype = ctypes.c_int
            L.or_verify.argtypes = [
                _f64p, _f64p, _f64p, _f64p, _i32p, _i32p, ni, _f64p, nu,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
                _i32p, _i32p, _i32p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _i32p]
            L.or_verify.restype = ctypes.c_int
            _lib = L
    return _lib


def _f64(x):
    """Exact widening of fp32 / bf16 / fp64 data (numpy or torch) to float64."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _u32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x).astype(np.uint32))


# ---------------------------------------------------------------------------
# random streams
# ---------------------------------------------------------------------------

def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().or_philox4x32_10(c, k, out)
    return out


def random_word(seed, request_id, j, v, stream):
    return int(lib().or_random_word(seed, request_id, j, v, stream))


def uniform(seed, request_id, j, v, stream):
    return float(lib().or_uniform(seed, request_id, j, v, stream))


def uniforms(seed, request_id, j, v0, n, stream):
    out = np.zeros(n)
    lib().or_uniforms(seed, request_id, j, v0, n, stream, out)
    return out


def gumbel(seed, request_id, j, v, stream):
    return float(lib().or_gumbel(seed, request_id, j, v, stream))


# ---------------------------------------------------------------------------
# the three steps
# ---------------------------------------------------------------------------

def draft_sample(U, E_in, W_out, anchor, temp, rid=None, seed=0, want_z=False):
    """Draft a block for every request (see ``or_draft_sample``).

    U [B,G,V], E_in [V,r], W_out [V,r] (row v scores token v), anchor [B], temp [B],
    rid [B] or None.
    Returns a dict of numpy arrays: tokens, lse, logq, gap, top (all [B,G]),
    and z [B,G,V] when ``want_z``.
    """
    U = _f64(U)
    E_in = _f64(E_in)
    W_out = _f64(W_out)
    B, G, V = U.shape
    r = E_in.shape[1]
    assert E_in.shape == (V, r) and W_out.shape == (V, r)
    anchor = _i32(anchor)
    temp = _f64(temp)
    rid = _u32(rid)
    out = dict(tokens=np.zeros((B, G), np.int32), lse=np.zeros((B, G)),
               logq=np.zeros((B, G)), gap=np.zeros((B, G)), top=np.zeros((B, G)))
    z = np.zeros((B, G, V)) if want_z else None
    rc = lib().or_draft_sample(U, E_in, W_out, anchor, temp, rid, B, G, V, r, seed,
                               out["tokens"], out["lse"], out["logq"], out["gap"], out["top"], z)
    if rc != 0:
        raise ValueError("or_draft_sample failed: %d" % rc)
    if want_z:
        out["z"] = z
    return out


def draft_sample_rnn(U, E_in, W_h, W_out, anchor, temp, rid=None, seed=0, want_z=False):
    """Draft a block with the recurrent head (see ``or_draft_sample_rnn``).

    W_h [r,r] (row n: weights of state unit n).  Returns the keys of
    ``draft_sample`` plus h [B,G,r] (the bf16 states) and h_margin [B,G]."""
    U = _f64(U)
    E_in = _f64(E_in)
    W_h = _f64(W_h)
    W_out = _f64(W_out)
    B, G, V = U.shape
    r = E_in.shape[1]
    assert E_in.shape == (V, r) and W_out.shape == (V, r) and W_h.shape == (r, r)
    anchor = _i32(anchor)
    temp = _f64(temp)
    rid = _u32(rid)
    out = dict(tokens=np.zeros((B, G), np.int32), lse=np.zeros((B, G)),
               logq=np.zeros((B, G)), gap=np.zeros((B, G)), top=np.zeros((B, G)),
               h=np.zeros((B, G, r)), h_margin=np.zeros((B, G)))
    z = np.zeros((B, G, V)) if want_z else None
    rc = lib().or_draft_sample_rnn(U, E_in, W_h, W_out, anchor, temp, rid, B, G, V, r, seed,
                                   out["tokens"], out["lse"], out["logq"], out["gap"], out["top"],
                                   out["h"], out["h_margin"], z)
    if rc != 0:
        raise ValueError("or_draft_sample_rnn failed: %d" % rc)
    if want_z:
        out["z"] = z
    return out


def schedule(conf_logits, pos_temp, sps, L_min, L_max):
    """Calibrate confidences and choose verify lengths (see ``or_schedule``)."""
    cl = _f64(conf_logits)
    B, G = cl.shape
    pt = _f64(pos_temp)
    sp = _f64(sps)
    out = dict(conf=np.zeros((B, G)), cum_conf=np.zeros((B, G)),
               verify_len=np.zeros(B, np.int32))
    theta = np.zeros(1)
    nadm = np.zeros(1, np.int32)
    mm = np.zeros(1)
    mt = np.zeros(1)
    rc = lib().or_schedule(cl, pt, sp, len(sp), B, G, int(L_min), int(L_max),
                           out["conf"], out["cum_conf"], out["verify_len"], theta, nadm, mm, mt)
    if rc != 0:
        raise ValueError("or_schedule failed: %d" % rc)
    out.update(theta=float(theta[0]), n_admitted=int(nadm[0]), min_margin=float(mm[0]),
               min_tie=float(mt[0]))
    return out


def schedule_policy(conf_logits, pos_temp, sps, L_min, L_max, policy, threshold=0.0):
    """Verify lengths under one of the policies of ``or_schedule_policy``
    (0 early stop, 1 best prefix without early stop, 2 threshold on a,
    3 threshold on c)."""
    cl = _f64(conf_logits)
    B, G = cl.shape
    pt = _f64(pos_temp)
    sp = _f64(sps)
    out = dict(conf=np.zeros((B, G)), cum_conf=np.zeros((B, G)),
               verify_len=np.zeros(B, np.int32))
    theta = np.zeros(1)
    nadm = np.zeros(1, np.int32)
    mm = np.zeros(1)
    mt = np.zeros(1)
    rc = lib().or_schedule_policy(cl, pt, sp, len(sp), B, G, int(L_min), int(L_max), int(policy),
                                  float(threshold), out["conf"], out["cum_conf"], out["verify_len"], theta,
                                  nadm, mm, mt)
    if rc != 0:
        raise ValueError("or_schedule_policy failed: %d" % rc)
    out.update(theta=float(theta[0]), n_admitted=int(nadm[0]), min_margin=float(mm[0]),
               min_tie=float(mt[0]))
    return out


def verify(target, U, E_in, W_out, anchor, draft_tokens, verify_len, temp, rid=None, seed=0):
    """Rejection-sampling verification of one block per request (see ``or_verify``)."""
    target = _f64(target)
    U = _f64(U)
    E_in = _f64(E_in)
    W_out = _f64(W_out)
    B, G, V = U.shape
    r = E_in.shape[1]
    assert target.shape == (B, G + 1, V)
    anchor = _i32(anchor)
    dt = _i32(draft_tokens)
    vl = None if verify_len is None else _i32(verify_len)
    temp = _f64(temp)
    rid = _u32(rid)
    out = dict(accept_len=np.zeros(B, np.int32), out_tokens=np.zeros((B, G + 1), np.int32),
               num_out=np.zeros(B, np.int32), target_lse=np.zeros((B, G + 1)),
               logp=np.zeros((B, G)), logq=np.zeros((B, G)), accept_margin=np.zeros((B, G)),
               final_gap=np.zeros(B), final_top=np.zeros(B), final_kind=np.zeros(B, np.int32))
    rc = lib().or_verify(target, U, E_in, W_out, anchor, dt, vl, temp, rid, B, G, V, r, seed,
                         out["accept_len"], out["out_tokens"], out["num_out"], out["target_lse"],
                         out["logp"], out["logq"], out["accept_margin"], out["final_gap"],
                         out["final_top"], out["final_kind"])
    if rc != 0:
        raise ValueError("or_verify failed: %d" % rc)
    return out


# ---------------------------------------------------------------------------
# request-parallel drivers (the oracle's loops are independent per request)
# ---------------------------------------------------------------------------

def _chunks(B, n):
    n = max(1, min(n, B))
    step = (B + n - 1) // n
    return [(i, min(B, i + step)) for i in range(0, B, step)]


def _merge(parts):
    out = {}
    for k in parts[0]:
        if isinstance(parts[0][k], np.ndarray):
            out[k] = np.concatenate([p[k] for p in parts], axis=0)
    return out


def _rid_or_default(rid, B):
    if rid is None:
        return np.arange(B, dtype=np.uint32)
    return _u32(rid)


def draft_sample_parallel(U, E_in, W_out, anchor, temp, rid=None, seed=0, threads=None):
    """``draft_sample`` over request chunks on ``threads`` host threads."""
    U = _f64(U); E_in = _f64(E_in); W_out = _f64(W_out)
    anchor = _i32(anchor); temp = _f64(temp)
    B = U.shape[0]
    rid = _rid_or_default(rid, B)
    threads = threads or os.cpu_count() or 1
    parts = _chunks(B, threads)
    with ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(lambda ab: draft_sample(U[ab[0]:ab[1]], E_in, W_out, anchor[ab[0]:ab[1]],
                                                  temp[ab[0]:ab[1]], rid[ab[0]:ab[1]], seed), parts))
    return _merge(res)


def draft_sample_rnn_parallel(U, E_in, W_h, W_out, anchor, temp, rid=None, seed=0, threads=None,
                              want_z=False):
    """``draft_sample_rnn`` over request chunks on ``threads`` host threads."""
    U = _f64(U); E_in = _f64(E_in); W_h = _f64(W_h); W_out = _f64(W_out)
    anchor = _i32(anchor); temp = _f64(temp)
    B = U.shape[0]
    rid = _rid_or_default(rid, B)
    threads = threads or os.cpu_count() or 1
    parts = _chunks(B, threads)
    with ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(lambda ab: draft_sample_rnn(U[ab[0]:ab[1]], E_in, W_h, W_out, anchor[ab[0]:ab[1]],
                                                      temp[ab[0]:ab[1]], rid[ab[0]:ab[1]], seed,
                                                      want_z=want_z), parts))
    return _merge(res)


def verify_parallel(target, U, E_in, W_out, anchor, draft_tokens, verify_len, temp, rid=None,
                    seed=0, threads=None):
    """``verify`` over request chunks on ``threads`` host threads."""
    target = _f64(target); U = _f64(U); E_in = _f64(E_in); W_out = _f64(W_out)
    anchor = _i32(anchor); dt = _i32(draft_tokens); temp = _f64(temp)
    B = U.shape[0]
    vl = None if verify_len is None else _i32(verify_len)
    rid = _rid_or_default(rid, B)
    threads = threads or os.cpu_count() or 1
    parts = _chunks(B, threads)

    def one(ab):
        a, b = ab
        return verify(target[a:b], U[a:b], E_in, W_out, anchor[a:b], dt[a:b],
                      None if vl is None else vl[a:b], temp[a:b], rid[a:b], seed)

    with ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(one, parts))
    return _merge(res)
