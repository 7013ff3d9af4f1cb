"""Helpers that run the CUDA path and the oracle on the same inputs and compare
them under the parity contract.

Contract (fp32 device arithmetic against a double-precision oracle):
  - token ids, accepted lengths and verify lengths are bit-exact, except for a
    decision the oracle itself places on a near-tie: a Gumbel (or greedy)
    top-two gap <= TIE_GUMBEL * max(1, |top key|), an acceptance uniform
    within TIE_ACCEPT of min(1, p/q), or a scheduler step whose Theta change
    or candidate order is within TIE_THETA (relative).  Such mismatches are
    counted (``exempt``, out of ``decisions``); everything after a divergence
    in the same request is skipped.  A mismatch on any other decision fails.
  - log-sum-exps and calibrated confidences agree within REL (relative, with
    a floor of 1 on the scale); log-probabilities within REL absolute (that is,
    probabilities within REL relative) down to log p = -64, and within
    REL |log p| / 64 below (p < 2^-92, masked tokens), where the spacing of
    fp32 numbers near log p itself exceeds REL.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

import oracle
from speculative_decoding_draft_head_gb300 import binding
from speculative_decoding_draft_head_gb300.synth import make_inputs

REL = 1e-5
TIE_GUMBEL = 1e-5
TIE_ACCEPT = 1e-6
TIE_THETA = 1e-6
# exempt (near-tie) mismatches allowed per decision: the parity bar
EXEMPT_RATE = 1e-6


@dataclasses.dataclass
class Tally:
    decisions: int = 0
    exempt: int = 0
    failures: list = dataclasses.field(default_factory=list)

    def add(self, other: "Tally"):
        self.decisions += other.decisions
        self.exempt += other.exempt
        self.failures += other.failures

    def check(self):
        assert not self.failures, "\n".join(self.failures[:20])

    def allowed_exempt(self):
        """Exempt mismatches a test of this many decisions may see at the
        parity bar (EXEMPT_RATE per decision): the count below which a
        Poisson count at that rate stays with probability 1 - 1e-3."""
        lam = EXEMPT_RATE * self.decisions
        k, p, cdf = 0, math.exp(-lam), math.exp(-lam)
        while cdf < 1.0 - 1e-3:
            k += 1
            p *= lam / k
            cdf += p
        return k

    def check_rate(self):
        self.check()
        assert self.exempt <= self.allowed_exempt(), (
            "%d exempt near-tie mismatches in %d decisions (allowed %d at %.0e per decision)"
            % (self.exempt, self.decisions, self.allowed_exempt(), EXEMPT_RATE))


def to_host(d):
    return {k: (v.detach().cpu() if torch.is_tensor(v) else v) for k, v in d.items()}


def gpu_round(inp, w, seed, scheduler=None, store_logits=False):
    """draft -> schedule (if the workload uses it) -> verify on the GPU; the
    device flag words of the calls must stay clear (no invalid input, no
    bounded wait that ran out)."""
    scheduler = w.scheduler if scheduler is None else scheduler
    dev = inp["base"].device
    ws_d = binding.default_workspace(binding.WS_DRAFT, w.B, w.G, w.V, w.r, dev)
    ws_v = binding.default_workspace(binding.WS_VERIFY, w.B, w.G, w.V, w.r, dev)
    d = binding.draft_sample(inp["base"], inp["e_in"], inp["w_out"], inp["anchor"],
                             inp["temperature"], inp["request_id"], seed, store_logits=store_logits,
                             workspace=ws_d)
    assert binding.read_device_flags(ws_d) == 0, "draft flags %d" % binding.read_device_flags(ws_d)
    sch = None
    vl = None
    if scheduler:
        sch = binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], inp["sps"], w.L_min, w.G)
        vl = sch["verify_len"]
    v = binding.verify(inp["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d, vl,
                       inp["temperature"], inp["request_id"], seed, workspace=ws_v)
    torch.cuda.synchronize()
    assert binding.read_device_flags(ws_v) == 0, "verify flags %d" % binding.read_device_flags(ws_v)
    return dict(draft=to_host(d), sched=None if sch is None else to_host(sch), verify=to_host(v))


def oracle_round(hinp, w, seed, reqs=None, verify_len=None, threads=None):
    """The oracle on the requests ``reqs`` (all when None)."""
    B = w.B
    reqs = np.arange(B) if reqs is None else np.asarray(reqs)
    base = hinp["base"][reqs]
    target = hinp["target"][reqs]
    anchor = hinp["anchor"][reqs]
    temp = hinp["temperature"][reqs]
    rid = hinp["request_id"].numpy().astype(np.uint32)[reqs]
    d = oracle.draft_sample_parallel(base, hinp["e_in"], hinp["w_out"], anchor, temp, rid, seed,
                                     threads=threads)
    sch = None
    if w.scheduler and verify_len is None:
        sch = oracle.schedule(hinp["conf_logits"], hinp["pos_temp"], hinp["sps"], w.L_min, w.G)
        vl_all = sch["verify_len"]
    else:
        vl_all = verify_len
    vl = None if vl_all is None else np.asarray(vl_all)[reqs]
    v = oracle.verify_parallel(target, base, hinp["e_in"], hinp["w_out"], anchor, d["tokens"], vl,
                               temp, rid, seed, threads=threads)
    return dict(draft=d, sched=sch, verify=v, reqs=reqs)


def _close(a, b, scale_floor=1.0, rel=REL):
    return abs(a - b) <= rel * max(scale_floor, abs(b))


def compare_draft(g, o, temps, reqs, logq_tol=None):
    """g: GPU draft (host tensors, all B rows); o: oracle draft on ``reqs``.
    logq_tol: per-request absolute tolerance of log q (default REL)."""
    t = Tally()
    G = o["tokens"].shape[1]
    diverged = np.zeros(len(reqs), bool)
    gt, gl, gq = g["tokens"].numpy(), g["lse"].numpy(), g["logq"].numpy()
    for i, b in enumerate(reqs):
        T = float(temps[b])
        for j in range(G):
            t.decisions += 1
            if gt[b, j] != o["tokens"][i, j]:
                gap, top = o["gap"][i, j], o["top"][i, j]
                if gap <= TIE_GUMBEL * max(1.0, abs(top)):
                    t.exempt += 1
                    diverged[i] = True
                    break
                t.failures.append("draft token b=%d j=%d gpu=%d oracle=%d gap=%.3g" %
                                  (b, j, gt[b, j], o["tokens"][i, j], gap))
                diverged[i] = True
                break
            if not _close(gl[b, j], o["lse"][i, j]):
                t.failures.append("draft lse b=%d j=%d gpu=%.9g oracle=%.9g" % (b, j, gl[b, j], o["lse"][i, j]))
            tq = REL if logq_tol is None else float(logq_tol[b])
            if T > 0 and abs(gq[b, j] - o["logq"][i, j]) > tq:
                t.failures.append("draft logq b=%d j=%d gpu=%.9g oracle=%.9g" % (b, j, gq[b, j], o["logq"][i, j]))
            if T == 0 and gq[b, j] != 0.0:
                t.failures.append("greedy logq b=%d j=%d is %g" % (b, j, gq[b, j]))
    return t, diverged


def compare_schedule(g, o):
    t = Tally()
    c, a = g["conf"].numpy(), g["cum_conf"].numpy()
    if not np.allclose(c, o["conf"], rtol=REL, atol=0):
        t.failures.append("calibrated confidences differ: max rel %.3g" %
                          np.max(np.abs(c - o["conf"]) / np.abs(o["conf"])))
    if not np.allclose(a, o["cum_conf"], rtol=REL, atol=0):
        t.failures.append("cumulative confidences differ")
    t.decisions += int(o["n_admitted"]) + 1
    gl = g["verify_len"].numpy()
    if not np.array_equal(gl, o["verify_len"]):
        if min(o["min_margin"], o["min_tie"]) <= TIE_THETA:
            t.exempt += 1
        else:
            t.failures.append("verify lengths differ (%d requests)" % int((gl != o["verify_len"]).sum()))
    theta = float(g["theta"].numpy()[0])
    if not _close(theta, o["theta"]):
        t.failures.append("theta gpu=%.12g oracle=%.12g" % (theta, o["theta"]))
    return t


def compare_verify(g, o, temps, reqs, skip):
    """Compare verification outputs of requests whose drafts matched."""
    t = Tally()
    ga, go, gn = g["accept_len"].numpy(), g["out_tokens"].numpy(), g["num_out"].numpy()
    glse, glp = g["target_lse"].numpy(), g["logp"].numpy()
    for i, b in enumerate(reqs):
        if skip[i]:
            continue
        T = float(temps[b])
        ka, ko = int(ga[b]), int(o["accept_len"][i])
        t.decisions += min(ka, ko) + 1
        if ka != ko:
            row = min(ka, ko)
            m = o["accept_margin"][i, row] if T > 0 else np.nan
            if T > 0 and not np.isnan(m) and m <= TIE_ACCEPT:
                t.exempt += 1
            else:
                t.failures.append("accept_len b=%d gpu=%d oracle=%d margin=%s" % (b, ka, ko, m))
            continue
        t.decisions += 1
        if gn[b] != o["num_out"][i]:
            t.failures.append("num_out b=%d" % b)
        if not np.array_equal(go[b, :ka], o["out_tokens"][i, :ko]):
            t.failures.append("accepted prefix b=%d" % b)
        if go[b, ka] != o["out_tokens"][i, ko]:
            gap, top = o["final_gap"][i], o["final_top"][i]
            if gap <= TIE_GUMBEL * max(1.0, abs(top)):
                t.exempt += 1
            else:
                t.failures.append("final token b=%d gpu=%d oracle=%d kind=%d gap=%.3g" %
                                  (b, go[b, ka], o["out_tokens"][i, ko], o["final_kind"][i], gap))
        if np.any(go[b, ka + 1:] != -1):
            t.failures.append("padding b=%d" % b)
        for j in range(o["target_lse"].shape[1]):
            ol = o["target_lse"][i, j]
            if not np.isnan(ol) and not _close(glse[b, j], ol):
                t.failures.append("target lse b=%d j=%d gpu=%.9g oracle=%.9g" % (b, j, glse[b, j], ol))
        for j in range(o["logp"].shape[1]):
            ol = o["logp"][i, j]
            # absolute below |log p| = 64; beyond (p < 2^-92, a masked token) the
            # fp32 spacing of log p itself passes REL, so the bound scales with it
            if np.isfinite(ol) and abs(glp[b, j] - ol) > REL * max(1.0, abs(ol) / 64.0):
                t.failures.append("logp b=%d j=%d gpu=%.9g oracle=%.9g" % (b, j, glp[b, j], ol))
    return t


def host_inputs(inp):
    return {k: v.detach().cpu() for k, v in inp.items()}


def logq_tolerance_low_temperature(inp):
    """Per-request tolerance of log q for temperatures far below 1: REL plus
    the fp32 representation of the draft logits scaled by 1/T.  The device
    holds z = U + bias in fp32 (one rounding, at most half an ulp of |z|),
    and log q = z(x)/T - lse moves by at most an ulp of the row's largest |z|
    over T; the oracle's z is exact.  Bound on |z|: the row's largest |U|
    plus r max|E_in| max|W_out|."""
    U = inp["base"].float().abs().amax(dim=(1, 2)).cpu().double()
    r = inp["e_in"].shape[1]
    bias = r * float(inp["e_in"].float().abs().max()) * float(inp["w_out"].float().abs().max())
    T = inp["temperature"].cpu().double()
    zmax = U + bias
    ulp = torch.pow(2.0, torch.floor(torch.log2(zmax.clamp_min(1e-30))) - 23)
    return (REL + torch.where(T > 0, ulp / T.clamp_min(1e-30), torch.zeros_like(T))).numpy()


def full_parity(w, seed, reqs=None, device="cuda", threads=None, edit=None, logq_tol=None):
    """Generate inputs, run both sides, compare everything; returns the Tally.
    edit(inputs), if given, changes the generated inputs in place first (the
    same inputs then go to both sides); logq_tol(inputs), if given, gives the
    per-request tolerance of log q (default REL)."""
    inp = make_inputs(w, seed, device=device)
    if edit is not None:
        edit(inp)
    g = gpu_round(inp, w, seed)
    h = host_inputs(inp)
    o = oracle_round(h, w, seed, reqs=reqs, threads=threads)
    temps = h["temperature"].numpy()
    tally = Tally()
    if w.scheduler:
        tally.add(compare_schedule(g["sched"], o["sched"]))
    td, diverged = compare_draft(g["draft"], o["draft"], temps, o["reqs"],
                                 None if logq_tol is None else logq_tol(inp))
    tally.add(td)
    skip = diverged.copy()
    if w.scheduler:
        gl = g["sched"]["verify_len"].numpy()
        skip |= gl[o["reqs"]] != o["sched"]["verify_len"][o["reqs"]]
    tally.add(compare_verify(g["verify"], o["verify"], temps, o["reqs"], skip))
    return tally, g, o, inp
