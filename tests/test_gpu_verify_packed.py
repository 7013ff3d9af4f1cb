"""Verification on a packed target (dspark_verify_packed) against the dense form.

"DSpark, la bozza che sa quando fermarsi" (paithon.it), section "Verificare
meglio, non di piu'": the scheduler's verify lengths size the target's batch,
so a serving engine holds target logits only for rows 0 .. L_b of each
request.  The packed call reads exactly those rows and must give the dense
call's results bit for bit (the dense form is itself parity-tested against the
oracle); rows outside the array are flagged and never read.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_draft_head_gb300 import binding
from speculative_decoding_draft_head_gb300.synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _pack(target, vl, order, gap):
    """Rows 0 .. L_b of each request, requests placed in ``order`` with ``gap``
    unused rows between them.  Returns (packed [n, V], row0 [B] int64)."""
    B = target.shape[0]
    row0 = torch.empty(B, dtype=torch.int64)
    pieces, pos = [], 0
    vl_h = vl.cpu().tolist()
    for b in order:
        if gap:
            pieces.append(torch.full((gap, target.shape[2]), 7.0, dtype=target.dtype, device=target.device))
            pos += gap
        row0[b] = pos
        pieces.append(target[b, : vl_h[b] + 1])
        pos += vl_h[b] + 1
    return torch.cat(pieces).contiguous(), row0.to(target.device)


def _same(a, b):
    a, b = a.cpu().numpy(), b.cpu().numpy()
    return np.array_equal(a, b, equal_nan=True) if a.dtype.kind == "f" else np.array_equal(a, b)


def _compare(inp, w, seed, vl, order, gap):
    d = binding.draft_sample(inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], inp["temperature"],
                             inp["request_id"], seed)
    dense = binding.verify(inp["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d, vl,
                           inp["temperature"], inp["request_id"], seed)
    packed_t, row0 = _pack(inp["target"], vl, order, gap)
    packed = binding.verify(packed_t, inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d, vl,
                            inp["temperature"], inp["request_id"], seed, target_row0=row0)
    torch.cuda.synchronize()
    for k in dense:
        assert _same(dense[k], packed[k]), k
    return dense, packed_t.shape[0]


@pytest.mark.parametrize("name,B,V", [("dspark5", 64, 8200), ("largev", 16, 16392), ("highconc", 160, 4104)])
def test_packed_equals_dense_scaled(name, B, V):
    w = WORKLOADS[name].scaled(B=B, V=V)
    for seed in range(2):
        inp = make_inputs(w, seed, device="cuda")
        gen = torch.Generator().manual_seed(seed)
        vl = torch.randint(0, w.G + 1, (w.B,), generator=gen, dtype=torch.int32).cuda()
        order = torch.randperm(w.B, generator=gen).tolist()
        _compare(inp, w, seed, vl, order, gap=seed)


def test_packed_equals_dense_full_size_with_scheduled_lengths():
    w = WORKLOADS["dspark5"]
    inp = make_inputs(w, 2, device="cuda")
    sch = binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], inp["sps"], w.L_min, w.G)
    vl = sch["verify_len"].clone()
    dense, rows = _compare(inp, w, 2, vl, list(range(w.B)), gap=0)
    # only the scheduled rows exist: sum_b (L_b + 1) of B (G + 1)
    assert rows == int((vl.long() + 1).sum()) < w.B * (w.G + 1)
    assert int(dense["accept_len"].min()) >= 0


def test_rows_outside_the_packed_array_are_flagged_not_read():
    w = WORKLOADS["dspark5"].scaled(B=8, V=2056)
    inp = make_inputs(w, 0, device="cuda")
    vl = torch.full((w.B,), 3, dtype=torch.int32, device="cuda")
    d = binding.draft_sample(inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], inp["temperature"],
                             inp["request_id"], 0)
    packed_t, row0 = _pack(inp["target"], vl, list(range(w.B)), gap=0)
    row0[2] = packed_t.shape[0] - 2       # rows 0 .. 3 would run past the end
    row0[5] = -1
    ws = binding.default_workspace(binding.WS_VERIFY, w.B, w.G, w.V, w.r, packed_t.device)
    v = binding.verify(packed_t, inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d, vl,
                       inp["temperature"], inp["request_id"], 0, target_row0=row0, workspace=ws)
    assert binding.read_device_flags(ws) & binding.FLAG_BAD_TARGET_ROW
    acc = v["accept_len"].cpu().numpy()
    assert acc[2] == -1 and acc[5] == -1
    assert np.all(np.delete(acc, [2, 5]) >= 0)
    lib = binding.load()
    st = lib.dspark_verify_packed(binding._ptr(packed_t), None, 4, *([None] * 11), 1, 1, 8, 16, 0, 0,
                                  *([None] * 5), None, 0, None)
    assert st != 0 and b"target_row0" in lib.dspark_last_error()


@pytest.mark.parametrize("where", ["device", "pinned host"])
def test_pack_target_gathers_the_scheduled_rows(where):
    w = WORKLOADS["dspark5"].scaled(B=48, V=4104)
    inp = make_inputs(w, 3, device="cuda")
    gen = torch.Generator().manual_seed(3)
    vl = torch.randint(0, w.G + 1, (w.B,), generator=gen, dtype=torch.int32)
    vl[5], vl[9] = -1, w.G + 1          # invalid lengths contribute no row
    vl = vl.cuda()
    src = inp["target"] if where == "device" else inp["target"].cpu().pin_memory()
    pk = binding.pack_target(src, vl)
    torch.cuda.synchronize()
    vh = vl.cpu().numpy()
    rows = np.where((vh < 0) | (vh > w.G), 0, vh + 1)
    assert int(pk["n_rows"].item()) == int(rows.sum())
    assert np.array_equal(pk["row0"].cpu().numpy(), np.concatenate([[0], np.cumsum(rows)[:-1]]))
    want = torch.cat([inp["target"][b, : rows[b]] for b in range(w.B) if rows[b] > 0])
    assert torch.equal(pk["target"][: int(rows.sum())], want)


def test_pack_then_verify_packed_equals_dense_full_size():
    w = WORKLOADS["dspark5"]
    inp = make_inputs(w, 4, device="cuda")
    d = binding.draft_sample(inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], inp["temperature"],
                             inp["request_id"], 4)
    sch = binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], inp["sps"], w.L_min, w.G)
    vl = sch["verify_len"]
    dense = binding.verify(inp["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d, vl,
                           inp["temperature"], inp["request_id"], 4)
    pk = binding.pack_target(inp["target"].cpu().pin_memory(), vl)
    packed = binding.verify(pk["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d, vl,
                            inp["temperature"], inp["request_id"], 4, target_row0=pk["row0"])
    torch.cuda.synchronize()
    for k in dense:
        assert _same(dense[k], packed[k]), k
