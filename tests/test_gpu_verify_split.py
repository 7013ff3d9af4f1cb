"""Verification split in two calls (dspark_verify_rows + dspark_verify_finish)
against the single call (dspark_verify / dspark_verify_packed).

The target-row statistics of the rejection test (the log-sum-exp of every
tested target row at its temperature, or its argmax for a greedy request)
depend only on the target logits and the verify lengths ("DSpark, la bozza
che sa quando fermarsi", section "Verificare meglio, non di piu'"), so they may
run before the draft exists, beside the draft kernel on another stream.  The
split must give the single call's results bit for bit (the single call is
itself parity-tested against the oracle), whatever runs beside it.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_draft_head_gb300 import binding
from speculative_decoding_draft_head_gb300.synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _same(a, b):
    a, b = a.cpu().numpy(), b.cpu().numpy()
    return np.array_equal(a, b, equal_nan=True) if a.dtype.kind == "f" else np.array_equal(a, b)


def _draft(inp, seed, stream=None, out=None, ws=None):
    return binding.draft_sample(inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], inp["temperature"],
                                inp["request_id"], seed, out=out, workspace=ws, stream=stream)


def _split(inp, d, vl, seed, w, target=None, row0=None, stream=None):
    target = inp["target"] if target is None else target
    ws = binding.verify_rows(target, vl, inp["temperature"], w.G, target_row0=row0, r=w.r, stream=stream,
                             workspace=binding.default_workspace(binding.WS_VERIFY, w.B, w.G, w.V, w.r,
                                                                 target.device).clone())
    return binding.verify(target, inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d, vl,
                          inp["temperature"], inp["request_id"], seed, target_row0=row0, rows_done=True,
                          workspace=ws, stream=stream), ws


@pytest.mark.parametrize("name,B,V,dtype", [("dspark5", 64, 8200, "bf16"), ("highconc", 150, 4104, "bf16"),
                                            ("largev", 16, 16392, "f32")])
def test_split_equals_single_call(name, B, V, dtype):
    w = WORKLOADS[name].scaled(B=B, V=V, dtype=dtype)
    for seed in range(2):
        inp = make_inputs(w, seed, device="cuda")
        gen = torch.Generator().manual_seed(seed)
        vl = torch.randint(-1 if seed else 0, w.G + 1, (w.B,), generator=gen, dtype=torch.int32).cuda()
        d = _draft(inp, seed)
        one = binding.verify(inp["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d, vl,
                             inp["temperature"], inp["request_id"], seed)
        two, ws = _split(inp, d, vl, seed, w)
        torch.cuda.synchronize()
        for k in one:
            assert _same(one[k], two[k]), k
        # an invalid length is flagged by the finishing half, as by the single call
        if seed:
            assert bool(binding.read_device_flags(ws) & binding.FLAG_BAD_VERIFY_LEN) == bool((vl < 0).any())


def test_split_beside_the_draft_full_size_packed():
    """The bench's order: schedule, then the rows half on a side stream while
    the draft runs, then the finishing half on the packed target."""
    w = WORKLOADS["dspark5"]
    inp = make_inputs(w, 6, device="cuda")
    sch = binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], inp["sps"], w.L_min, w.G)
    vl = sch["verify_len"]
    d_ref = _draft(inp, 6)
    pk = binding.pack_target(inp["target"], vl)
    one = binding.verify(pk["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d_ref, vl,
                         inp["temperature"], inp["request_id"], 6, target_row0=pk["row0"])
    torch.cuda.synchronize()

    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    d_out = {k: torch.empty_like(v) for k, v in d_ref.items()}
    ws_v = binding.default_workspace(binding.WS_VERIFY, w.B, w.G, w.V, w.r, inp["target"].device).clone()
    for _ in range(3):
        ev0, ev1 = torch.cuda.Event(), torch.cuda.Event()
        ev0.record(main)
        side.wait_event(ev0)
        binding.verify_rows(pk["target"], vl, inp["temperature"], w.G, target_row0=pk["row0"], r=w.r,
                            workspace=ws_v, stream=side)
        ev1.record(side)
        _draft(inp, 6, stream=main, out=d_out)
        main.wait_event(ev1)
        two = binding.verify(pk["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d_out, vl,
                             inp["temperature"], inp["request_id"], 6, target_row0=pk["row0"],
                             rows_done=True, workspace=ws_v, stream=main)
        torch.cuda.synchronize()
        for k in d_ref:
            assert _same(d_ref[k], d_out[k]), k
        for k in one:
            assert _same(one[k], two[k]), k
        assert binding.read_device_flags(ws_v) == 0


def test_rows_half_rejects_bad_arguments():
    lib = binding.load()
    f = torch.zeros(64, device="cuda")
    p = binding._ptr(f)
    st = lib.dspark_verify_rows(p, None, 0, None, None, 1, 1, 8, 16, 0, p, 1 << 20, None)
    assert st != 0 and b"NULL" in lib.dspark_last_error()
    st = lib.dspark_verify_rows(p, p, 0, None, p, 1, 1, 8, 16, 0, p, 1 << 20, None)
    assert st != 0 and b"n_target_rows" in lib.dspark_last_error()
    st = lib.dspark_verify_rows(p, None, 0, None, p, 1, 1, 8, 16, 0, p, 16, None)
    assert st != 0
