"""The C-ABI library loads, exports every declared symbol and rejects bad
host-side arguments before touching the GPU (no compute calls here)."""
import ctypes
import glob
import os
import re

import pytest

from speculative_decoding_draft_head_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"DSPARK_API\s+[\w\s\*]*?\b(dspark_\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_library_builds_and_exports_every_declared_symbol():
    path = build.build_library()
    lib = ctypes.CDLL(path)
    declared = _declared_symbols()
    assert declared == set(binding.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_workspace_sizes():
    lib = binding.load()
    assert lib.dspark_version() >= 100
    for which in (0, 1, 2):
        assert binding.workspace_bytes(which, 256, 5, 129280, 256) >= 256
    assert binding.workspace_bytes(0, 0, 5, 129280, 256) == 0
    assert binding.workspace_bytes(2, 4, 5, 1001, 16) == 0     # V % 8 != 0
    assert binding.workspace_bytes(7, 4, 5, 1024, 16) == 0


def _call_draft(**over):
    lib = binding.load()
    args = dict(base=1 << 12, e_in=1 << 12, w_out=1 << 12, anchor=1 << 12, temp=1 << 12, rid=None,
                B=4, G=4, V=1024, r=16, dt=1, seed=0, tok=1 << 12, lse=1 << 12, logq=1 << 12,
                logits=None, ws=1 << 12, wsb=0, stream=None)
    args.update(over)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    st = lib.dspark_draft_sample(vp(args["base"]), vp(args["e_in"]), vp(args["w_out"]),
                                 vp(args["anchor"]), vp(args["temp"]), vp(args["rid"]),
                                 args["B"], args["G"], args["V"], args["r"], args["dt"], args["seed"],
                                 vp(args["tok"]), vp(args["lse"]), vp(args["logq"]),
                                 vp(args["logits"]), vp(args["ws"]), args["wsb"], vp(args["stream"]))
    return st, lib.dspark_last_error().decode()


@pytest.mark.parametrize("over,needle", [
    (dict(B=0), "B must be"),
    (dict(G=0), "G must be"),
    (dict(G=65), "G must be"),
    (dict(V=1001), "multiple of 8"),
    (dict(r=0), "r must be"),
    (dict(dt=0, r=24), "r % 16"),
    (dict(dt=5), "unknown dtype"),
    (dict(dt=1, r=6), "r % 4"),
    (dict(base=None), "NULL"),
    (dict(base=(1 << 12) + 4), "aligned"),
    (dict(ws=None), "workspace is NULL"),
    (dict(ws=(1 << 12) + 16), "256-byte"),
    (dict(wsb=16), "too small"),
])
def test_draft_rejects_bad_host_arguments(over, needle):
    st, msg = _call_draft(**over)
    assert st == 1 and needle in msg, (st, msg)


def test_schedule_and_verify_reject_bad_host_arguments():
    lib = binding.load()
    vp = ctypes.c_void_p
    p = vp(1 << 12)
    st = lib.dspark_schedule_prefix(p, p, p, 10, 4, 4, 3, 2, p, p, p, None, p, 4096, None)
    assert st == 1 and "L_min" in lib.dspark_last_error().decode()
    st = lib.dspark_schedule_prefix(p, p, p, 10, 4, 4, 1, 4, p, p, p, None, p, 4096, None)
    assert st == 1 and "sps_len" in lib.dspark_last_error().decode()
    st = lib.dspark_verify(p, None, None, None, None, p, p, p, p, None, p, None,
                           4, 4, 1024, 16, 1, 0, p, p, p, None, None, p, 1 << 20, None)
    assert st == 1 and "draft_logits" in lib.dspark_last_error().decode()


def test_packed_verify_rejects_bad_host_arguments():
    """dspark_verify_packed checks the packed layout, then dspark_verify's
    arguments, on the host before any launch."""
    lib = binding.load()
    vp = ctypes.c_void_p
    p = vp(1 << 12)
    err = lambda: lib.dspark_last_error().decode()
    st = lib.dspark_verify_packed(p, p, 0, p, p, p, None, p, p, p, p, None, p, None,
                                  4, 4, 1024, 16, 1, 0, p, p, p, None, None, p, 1 << 20, None)
    assert st == 1 and "n_target_rows" in err()
    st = lib.dspark_verify_packed(p, p, 8, None, None, None, None, p, p, p, p, None, p, None,
                                  4, 4, 1024, 16, 1, 0, p, p, p, None, None, p, 1 << 20, None)
    assert st == 1 and "draft_logits" in err()


def test_pack_target_rejects_bad_host_arguments():
    lib = binding.load()
    vp = ctypes.c_void_p
    p = vp(1 << 12)
    err = lambda: lib.dspark_last_error().decode()
    cases = [
        ((p, None, 0, 4, 1024, 0, p, p, p, None), "bad B"),
        ((p, None, 4, 65, 1024, 0, p, p, p, None), "bad B"),
        ((p, None, 4, 4, 1001, 0, p, p, p, None), "multiple of 8"),
        ((p, None, 4, 4, 1024, 7, p, p, p, None), "unknown dtype"),
        ((None, None, 4, 4, 1024, 0, p, p, p, None), "NULL"),
        ((p, None, 4, 4, 1024, 0, vp((1 << 12) + 8), p, p, None), "aligned"),
    ]
    for args, needle in cases:
        st = lib.dspark_pack_target(*args)
        assert st == 1 and needle in err(), (args, st, err())


def test_recurrent_draft_rejects_bad_host_arguments():
    lib = binding.load()
    vp = ctypes.c_void_p
    p = vp(1 << 12)
    err = lambda: lib.dspark_last_error().decode()

    def call(dt=0, r=16, wh=p, ws=p, wsb=1 << 24, hs=None):
        return lib.dspark_draft_sample_rnn(p, p, wh, p, p, p, None, 4, 3, 1024, r, dt, 0, p, p, p, None, hs,
                                           ws, wsb, None)
    assert call(dt=1, r=16) == 2 and "bf16" in err()          # fp32 weights: unsupported
    assert call(r=24) == 1 and "r % 16" in err()
    assert call(wh=None) == 1 and "NULL" in err()
    assert call(wh=vp((1 << 12) + 8)) == 1 and "aligned" in err()
    assert call(hs=vp((1 << 12) + 1)) == 1 and "aligned" in err()
    assert call(wsb=16) == 1 and "too small" in err()


def test_selftest_and_noalloc_reject_on_the_host():
    lib = binding.load()
    vp = ctypes.c_void_p
    p = vp(1 << 12)
    err = lambda: lib.dspark_last_error().decode()
    res = ctypes.cast(vp(1 << 12), ctypes.POINTER(ctypes.c_uint32))
    assert lib.dspark_selftest_bounded_wait(0, res, None) == 1 and "limit_us" in err()
    assert lib.dspark_selftest_bounded_wait(2000000, res, None) == 1 and "limit_us" in err()
    assert lib.dspark_selftest_bounded_wait(10, None, None) == 1 and "NULL" in err()
    # a verification whose scratch exceeds the fixed array: unsupported, no launch
    args = [p] * 12 + [20096, 16, 129280, 256, 0, 0] + [p] * 6
    assert lib.dspark_verify_noalloc(*args) == 2 and "fixed" in err()
    # an invalid size is reported as dspark_verify reports it
    args = [p] * 12 + [4, 0, 1024, 16, 0, 0] + [p] * 6
    assert lib.dspark_verify_noalloc(*args) == 1 and "G must be" in err()
    # argument errors come before the scratch-size check, as in dspark_verify
    args = [p] * 5 + [None] + [p] * 6 + [20096, 16, 129280, 256, 0, 0] + [p] * 6
    assert lib.dspark_verify_noalloc(*args) == 1 and "NULL" in err()
    args = [vp((1 << 12) + 4)] + [p] * 11 + [20096, 16, 129280, 256, 0, 0] + [p] * 6
    assert lib.dspark_verify_noalloc(*args) == 1 and "aligned" in err()
    # the flag reader wants somewhere to put the word
    assert lib.dspark_read_noalloc_flags(None, None) == 1 and "NULL" in err()
    # the Philox rate probe checks its arguments before any launch
    rate = ctypes.c_double(0.0)
    assert lib.dspark_selftest_philox_rate(p, 1 << 16, 16, None, None) == 1 and "NULL" in err()
    assert lib.dspark_selftest_philox_rate(p, 1 << 16, 0, ctypes.byref(rate), None) == 1 and "iters" in err()
