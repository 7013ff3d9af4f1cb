"""dspark_verify_noalloc against dspark_verify (collected last on purpose).

The no-allocation entry point serves callers that cannot allocate device
memory (runtimes with pre-planned memory, plugins inside other frameworks,
foreign-function callers without an allocator).  It must give the same
results as the workspace entry point, call after call, although every call
reuses one fixed scratch array inside the library.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_draft_head_gb300 import binding
from speculative_decoding_draft_head_gb300.synth import WORKLOADS, make_inputs

REL = 1e-5  # the tolerance of the parity tests for log-sum-exps and log-probabilities


def _same(a, b):
    for k in ("accept_len", "out_tokens", "num_out"):
        assert torch.equal(a[k], b[k]), k
    for k in ("target_lse", "logp"):
        x, y = a[k].cpu().numpy(), b[k].cpu().numpy()
        assert np.array_equal(np.isnan(x), np.isnan(y)), k
        m = ~np.isnan(x) & np.isfinite(y)
        np.testing.assert_allclose(x[m], y[m], rtol=REL, atol=REL)


@pytest.mark.gpu
@pytest.mark.parametrize("name,scale", [("dspark5", dict(B=64, V=8200)), ("largev", dict(B=16, V=16392)),
                                        ("tiny", {})])
def test_noalloc_verify_matches_workspace_verify_twice(name, scale):
    w = WORKLOADS[name].scaled(**scale)
    inp = make_inputs(w, 21, device="cuda")
    d = binding.draft_sample(inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], inp["temperature"],
                             inp["request_id"], 21)
    vl = None
    if w.scheduler:
        vl = binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], inp["sps"], w.L_min, w.G)["verify_len"]
    args = (inp["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d, vl, inp["temperature"],
            inp["request_id"], 21)
    ref = binding.verify(*args)
    for _ in range(2):  # the second call finds the first call's scratch contents
        got = binding.verify_noalloc(*args)
        torch.cuda.synchronize()
        _same(got, ref)
    # a different seed through the same scratch still matches its own reference
    args2 = args[:-1] + (22,)
    _same(binding.verify_noalloc(*args2), binding.verify(*args2))


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_the_fixed_array():
    lib = binding.load()
    p = ctypes.c_void_p(1 << 20)
    st = lib.dspark_verify_noalloc(p, p, p, p, None, p, p, p, p, None, p, None,
                                   4096, 64, 1024, 16, 1, 0, p, p, p, None, None, None)
    assert st == 2
    assert "scratch" in lib.dspark_last_error().decode()


@pytest.mark.gpu
def test_noalloc_flag_word_reports_invalid_device_inputs():
    """An out-of-range verify length raises its bit in the fixed array's flag
    word, which dspark_read_noalloc_flags returns; the next valid call clears
    it."""
    w = WORKLOADS["dspark5"].scaled(B=8, V=2056, scheduler=False)
    inp = make_inputs(w, 5, device="cuda")
    d = binding.draft_sample(inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], inp["temperature"],
                             inp["request_id"], 5)
    vl = torch.full((w.B,), w.G, dtype=torch.int32, device="cuda")
    vl[3] = w.G + 7
    args = (inp["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d)
    got = binding.verify_noalloc(*args, vl, inp["temperature"], inp["request_id"], 5)
    assert binding.read_noalloc_flags() & binding.FLAG_BAD_VERIFY_LEN
    assert int(got["accept_len"][3]) == -1
    vl[3] = w.G
    binding.verify_noalloc(*args, vl, inp["temperature"], inp["request_id"], 5)
    assert binding.read_noalloc_flags() == 0
