"""CUDA path vs the oracle, element by element, through the C ABI.

Sizes: the tiny workload in full; every other workload scaled down in B and V
(the oracle finishes in seconds, the vocabulary still spans several segments
and a ragged tail); and every workload at full size with the oracle on a
sample of requests plus properties that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_head_gb300 import binding
from speculative_decoding_draft_head_gb300.synth import WORKLOADS, make_inputs

from parity import (REL, Tally, compare_draft, compare_verify, full_parity, gpu_round, host_inputs,
                    logq_tolerance_low_temperature, oracle_round)

pytestmark = pytest.mark.gpu

SCALED = {
    "tiny": WORKLOADS["tiny"],
    "qwen3": WORKLOADS["qwen3"].scaled(B=12, V=8200),
    "dspark5": WORKLOADS["dspark5"].scaled(B=64, V=8200),
    "largev": WORKLOADS["largev"].scaled(B=16, V=16392),
    "highconc": WORKLOADS["highconc"].scaled(B=160, V=4104),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load()
    oracle.build()


@pytest.mark.parametrize("name", list(SCALED))
def test_scaled_workload_matches_oracle(name):
    w = SCALED[name]
    total = Tally()
    for seed in range(3):
        tally, g, o, _ = full_parity(w, seed)
        total.add(tally)
    total.check()
    assert total.exempt <= total.allowed_exempt()


def test_tiny_many_seeds():
    w = SCALED["tiny"]
    total = Tally()
    for seed in range(40):
        tally, *_ = full_parity(w, 1000 + seed)
        total.add(tally)
    total.check()
    assert total.decisions > 600


def _properties(w, g, inp):
    d, v = g["draft"], g["verify"]
    V, G, B = w.V, w.G, w.B
    tok = d["tokens"].numpy()
    assert tok.min() >= 0 and tok.max() < V
    acc, out, n = v["accept_len"].numpy(), v["out_tokens"].numpy(), v["num_out"].numpy()
    vl = g["sched"]["verify_len"].numpy() if g["sched"] is not None else np.full(B, G)
    assert np.all(n == acc + 1) and np.all(acc >= 0) and np.all(acc <= vl)
    for b in range(B):
        assert np.array_equal(out[b, :acc[b]], tok[b, :acc[b]])
        assert 0 <= out[b, acc[b]] < V
        assert np.all(out[b, acc[b] + 1:] == -1)
    if g["sched"] is not None:
        assert vl.min() >= w.L_min and vl.max() <= G
    lse = d["lse"].numpy()
    assert np.all(np.isfinite(lse))
    logq = d["logq"].numpy()
    assert np.all(logq <= 1e-6)


def _spanning_sample(B, n, seed):
    """n requests (all of them if B <= n), spread over every 128-request row
    block of the tensor-core kernel and, inside each, drawn at random."""
    if B <= n:
        return np.arange(B)
    rng = np.random.default_rng(seed)
    blocks = [np.arange(a, min(B, a + 128)) for a in range(0, B, 128)]
    per = -(-n // len(blocks))
    picks = [rng.choice(blk, size=min(per, len(blk)), replace=False) for blk in blocks]
    return np.sort(np.concatenate(picks))


@pytest.mark.parametrize("name", ["qwen3", "dspark5", "largev", "highconc"])
def test_full_size_sampled_requests(name):
    """Full-size workloads, 32 or more requests against the oracle, spread over
    every row block (all 32 requests of largev: both temperature groups)."""
    w = WORKLOADS[name]
    reqs = _spanning_sample(w.B, 32, 5)
    assert len(reqs) >= 32 and len({int(r) // 128 for r in reqs}) == -(-w.B // 128)
    tally, g, o, inp = full_parity(w, 7, reqs=reqs)
    tally.check()
    assert tally.exempt <= tally.allowed_exempt()
    _properties(w, g, inp)
    del inp
    torch.cuda.empty_cache()


def test_draft_one_launch_per_position():
    """More 128-request row blocks than SMs: the grid cannot be resident at
    once, so the draft runs one launch per block position (each reading the
    previous position's draws from the workspace) and must still match."""
    w = WORKLOADS["qwen3"].scaled(B=157 * 128, G=3, V=1024, r=16)
    reqs = np.array([0, 1, 5000, 12345, 20000, w.B - 1])
    tally, g, o, inp = full_parity(w, 9, reqs=reqs)
    tally.check()
    del inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("G", [1, 2])
def test_short_blocks(G):
    """A block of one position (a single launch) and of two."""
    w = SCALED["qwen3"].scaled(G=G)
    total = Tally()
    for seed in range(3):
        tally, *_ = full_parity(w, 40 + seed)
        total.add(tally)
    total.check()


def test_verify_alone_on_oracle_drafts():
    """Feed the oracle's draft to the CUDA verify, compare with the oracle verify."""
    for name in ("tiny", "dspark5", "largev"):
        w = SCALED[name]
        inp = make_inputs(w, 3, device="cuda")
        h = host_inputs(inp)
        o = oracle_round(h, w, 3)
        d = dict(tokens=torch.from_numpy(o["draft"]["tokens"]).cuda(),
                 lse=torch.from_numpy(o["draft"]["lse"].astype(np.float32)).cuda(),
                 logq=torch.from_numpy(o["draft"]["logq"].astype(np.float32)).cuda())
        vl = None
        if w.scheduler:
            vl = torch.from_numpy(o["sched"]["verify_len"]).cuda()
        v = binding.verify(inp["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d,
                           vl, inp["temperature"], inp["request_id"], 3)
        torch.cuda.synchronize()
        g = {k: t.cpu() for k, t in v.items()}
        t = compare_verify(g, o["verify"], h["temperature"].numpy(), np.arange(w.B),
                           np.zeros(w.B, bool))
        t.check()


def test_stored_draft_logits_match_oracle_and_recompute_path():
    w = SCALED["dspark5"]
    inp = make_inputs(w, 4, device="cuda")
    d = binding.draft_sample(inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], inp["temperature"],
                             inp["request_id"], 4, store_logits=True)
    h = host_inputs(inp)
    o = oracle.draft_sample(h["base"][:4], h["e_in"], h["w_out"], h["anchor"][:4],
                            h["temperature"][:4], h["request_id"][:4].numpy().astype(np.uint32), 4,
                            want_z=True)
    z = d["logits"][:4].cpu().double().numpy()
    same = (d["tokens"][:4].cpu().numpy() == o["tokens"]).all(axis=1)
    for b in range(4):
        if same[b]:
            np.testing.assert_allclose(z[b], o["z"][b], rtol=REL, atol=REL)
    v1 = binding.verify(inp["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d, None,
                        inp["temperature"], inp["request_id"], 4)
    v2 = binding.verify(inp["target"], None, inp["e_in"], None, inp["anchor"], d, None,
                        inp["temperature"], inp["request_id"], 4, draft_logits=d["logits"])
    torch.cuda.synchronize()
    for k in ("accept_len", "out_tokens", "num_out"):
        assert torch.equal(v1[k], v2[k]), k


def test_edge_cases_lengths_and_greedy():
    w = SCALED["dspark5"].scaled(B=9, G=5, V=1032, scheduler=False)
    inp = make_inputs(w, 11, device="cuda")
    h = host_inputs(inp)
    for vl_np in (np.zeros(w.B, np.int32), np.full(w.B, w.G, np.int32),
                  np.arange(w.B, dtype=np.int32) % (w.G + 1)):
        for greedy in (False, True):
            temp = inp["temperature"].clone()
            if greedy:
                temp.zero_()
            inp2 = dict(inp, temperature=temp)
            d = binding.draft_sample(inp2["base"], inp2["e_in"], inp2["w_out"], inp2["anchor"], temp,
                                     inp2["request_id"], 11)
            vl = torch.from_numpy(vl_np).cuda()
            v = binding.verify(inp2["target"], inp2["base"], inp2["e_in"], inp2["w_out"], inp2["anchor"],
                               d, vl, temp, inp2["request_id"], 11)
            torch.cuda.synchronize()
            h2 = dict(h, temperature=temp.cpu())
            o = oracle_round(h2, w, 11, verify_len=vl_np)
            td, div = compare_draft({k: t.cpu() for k, t in d.items()}, o["draft"], h2["temperature"].numpy(),
                                    np.arange(w.B))
            td.check()
            tv = compare_verify({k: t.cpu() for k, t in v.items()}, o["verify"], h2["temperature"].numpy(),
                                np.arange(w.B), div)
            tv.check()


def test_minimal_sizes():
    w = WORKLOADS["tiny"].scaled(B=1, G=1, V=8, r=4)
    tally, *_ = full_parity(w, 0)
    tally.check()
    w2 = WORKLOADS["dspark5"].scaled(B=1, G=1, V=8, r=16, scheduler=False)
    tally, *_ = full_parity(w2, 0)
    tally.check()


# temperatures far from 1: per-request T spread geometrically over
# [0.02, 20] (very peaked to nearly flat draws), every 16th request greedy.
# Tokens, acceptance and residual draws stay exact against the oracle; log q
# is held to 1e-5 plus the fp32 representation of the logits over T
# (logq_tolerance_low_temperature), which passes 1e-5 below T of about 0.1.
@pytest.mark.parametrize("name", ["dspark5", "tiny"])
def test_extreme_temperatures(name):
    w = WORKLOADS[name].scaled(B=64, V=4104) if name != "tiny" else WORKLOADS["tiny"].scaled(B=64)

    def edit(inp):
        T = torch.logspace(np.log10(0.02), np.log10(20.0), w.B, dtype=torch.float64)
        T[::16] = 0.0
        inp["temperature"].copy_(T.to(torch.float32))

    total = Tally()
    for seed in range(3):
        tally, *_ = full_parity(w, 70 + seed, edit=edit, logq_tol=logq_tolerance_low_temperature)
        total.add(tally)
    total.check_rate()


# the longest block the entry points take (G = 64): 64 positions in one
# cooperative launch (or one SIMT launch), verification over 65 target rows,
# the scheduler over 63 candidates per request
@pytest.mark.parametrize("name,B,sched", [("dspark5", 16, True),    # scheduled lengths
                                          ("dspark5", 100, False),  # every request verifies all 64
                                          ("tiny", 4, False)])
def test_longest_block(name, B, sched):
    w = WORKLOADS[name].scaled(B=B, G=64, V=2056, r=16, scheduler=sched)
    total = Tally()
    for seed in range(2):
        tally, *_ = full_parity(w, 60 + seed)
        total.add(tally)
    total.check_rate()


# ranks r whose last 64-wide K block is partial (tensor path: W_out boxes
# zero-filled past r, a partial A-operand block, UMMA steps skipped past r),
# and an fp32 rank that is not a multiple of 16
@pytest.mark.parametrize("name,r", [("dspark5", 80), ("dspark5", 208), ("tiny", 52)])
def test_ranks_with_partial_k_blocks(name, r):
    w = (WORKLOADS[name].scaled(B=64, V=2056, r=r) if name != "tiny"
         else WORKLOADS["tiny"].scaled(B=32, r=r))
    total = Tally()
    for seed in range(2):
        tally, *_ = full_parity(w, 80 + seed)
        total.add(tally)
    total.check_rate()


# the largest vocabulary the entry points take: token ids fill the 20-bit
# field of the 64-bit key words (ids up to 2^20 - 1)
MAX_V = 1 << 20


@pytest.mark.parametrize("name,B,reqs", [("dspark5", 4, None),             # bf16, four replicas
                                         ("dspark5", 40, [0, 13, 27, 39]),  # bf16, two replicas
                                         ("tiny", 4, None)])                # fp32 weights, SIMT path
def test_maximum_vocabulary(name, B, reqs):
    w = WORKLOADS[name].scaled(B=B, G=2, V=MAX_V, r=16)
    tally, g, o, _ = full_parity(w, 3, reqs=reqs)
    tally.check_rate()
    # every drafted token is a valid id, the top ones included
    toks = g["draft"]["tokens"].numpy()
    assert toks.min() >= 0 and toks.max() < MAX_V
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["tiny", "dspark5"])
def test_invalid_device_inputs_are_flagged_not_read(name):
    """fp32 weights (SIMT draft writing its rows itself) and bf16 weights
    (tensor-core draft + finalize): flagged requests get token -1 and NaN lse
    and log q at every position, the others are drawn."""
    w = SCALED[name].scaled(B=4, scheduler=False)
    inp = make_inputs(w, 0, device="cuda")
    anchor = inp["anchor"].clone()
    anchor[1] = w.V + 5
    temp = inp["temperature"].clone()
    temp[2] = -1.0
    ws = binding.default_workspace(binding.WS_DRAFT, w.B, w.G, w.V, w.r, anchor.device)
    d = binding.draft_sample(inp["base"], inp["e_in"], inp["w_out"], anchor, temp, None, 0, workspace=ws)
    flags = binding.read_device_flags(ws)
    assert flags & binding.FLAG_BAD_TOKEN and flags & binding.FLAG_BAD_TEMPERATURE
    tok = d["tokens"].cpu().numpy()
    assert np.all(tok[1] == -1) and np.all(tok[2] == -1)
    assert np.all(tok[0] >= 0) and np.all(tok[3] >= 0)
    lse, logq = d["lse"].cpu().numpy(), d["logq"].cpu().numpy()
    assert np.all(np.isnan(lse[1:3])) and np.all(np.isnan(logq[1:3]))
    assert np.all(np.isfinite(lse[[0, 3]])) and np.all(np.isfinite(logq[[0, 3]]))
    vl = torch.tensor([2, 9, 1, 0], dtype=torch.int32, device="cuda")
    wsv = binding.default_workspace(binding.WS_VERIFY, w.B, w.G, w.V, w.r, anchor.device)
    v = binding.verify(inp["target"], inp["base"], inp["e_in"], inp["w_out"], anchor, d, vl, temp, None, 0,
                       workspace=wsv)
    flags = binding.read_device_flags(wsv)
    assert flags & binding.FLAG_BAD_VERIFY_LEN
    acc = v["accept_len"].cpu().numpy()
    assert acc[1] == -1 and acc[2] == -1 and acc[0] >= 0 and acc[3] == 0
    cl = inp["conf_logits"]
    pt = torch.ones(w.G, device="cuda")
    pt[1] = 0.0  # a position temperature must be > 0
    wss = binding.default_workspace(binding.WS_SCHEDULE, w.B, w.G, 8, 1, anchor.device)
    binding.schedule_prefix(cl, pt, inp["sps"], 1, w.G, workspace=wss)
    assert binding.read_device_flags(wss) & binding.FLAG_BAD_POS_TEMP
