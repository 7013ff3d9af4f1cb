"""Seeded synthetic workloads for the draft-sample / schedule / verify path.

This module only draws inputs; it holds none of the method's arithmetic.  The
same tensors feed the CUDA path and the CPU oracle.  Shapes and value
distributions follow the five workloads the library is measured on:

  tiny       B=4    G=4   V=1024    r=16   fp32  U~N(0,2^2), t=U+N(0,0.5^2), T=1
  qwen3      B=64   G=16  V=151936  r=256  bf16  U~N(0,3^2)+8 spike, t=U+N(0,1), T=1
  dspark5    B=256  G=5   V=129280  r=256  bf16  as qwen3, confidences + scheduler
  largev     B=32   G=8   V=262144  r=256  bf16  t=U+N(0,0.7^2), T=0 (b<16) / 0.7
  highconc   B=1024 G=4   V=129280  r=256  bf16  T~U[0.3,1.2], t=U+N(0,sigma_b^2),
                                                  sigma_b~U[0.2,2], scheduler on

E_in and W_out (both V x r; W_out row v scores token v) are N(0, 0.02^2).  The
recurrent head (make_rnn_head) draws its own, larger weights so that its state
moves the logits: E_in ~ N(0, 0.5^2), W_h ~ N(0, (0.9 / sqrt(r))^2) (a
contracting recurrence), W_out ~ N(0, 0.05^2), all rounded to bf16; the bias
then has a spread of about 0.3 nats against the base logits' 3.  Confidence logits are
N(1, 1); the per-position calibration temperatures are evenly spaced in
[1, 2]; the batch-token throughput table is SPS(n) = 1 / (1 + n / 512).
"""
from __future__ import annotations

import dataclasses
import zlib

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    G: int
    V: int
    r: int
    dtype: str            # "f32" or "bf16"
    u_sigma: float        # std of the base draft logits
    spike: float          # +spike on one uniformly drawn token per (b, j); 0 = none
    noise: str            # "const" or "per_request"
    noise_sigma: float    # target noise std ("const")
    temp: str             # "one", "mix_greedy", "uniform"
    temp_value: float = 1.0
    scheduler: bool = False
    L_min: int = 1

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 4, 4, 1024, 16, "f32", 2.0, 0.0, "const", 0.5, "one"),
    "qwen3": Workload("qwen3", 64, 16, 151936, 256, "bf16", 3.0, 8.0, "const", 1.0, "one"),
    "dspark5": Workload("dspark5", 256, 5, 129280, 256, "bf16", 3.0, 8.0, "const", 1.0, "one",
                        scheduler=True),
    "largev": Workload("largev", 32, 8, 262144, 256, "bf16", 3.0, 8.0, "const", 0.7,
                       "mix_greedy", temp_value=0.7),
    "highconc": Workload("highconc", 1024, 4, 129280, 256, "bf16", 3.0, 8.0, "per_request", 0.0,
                         "uniform", scheduler=True),
}


def torch_dtype(w: Workload):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def sps_table(n_max: int, capacity: float = 512.0, device="cpu") -> torch.Tensor:
    """SPS(n) for n = 0 .. n_max batch tokens: 1 / (1 + n / capacity)."""
    n = torch.arange(n_max + 1, dtype=torch.float64, device=device)
    return (1.0 / (1.0 + n / capacity)).to(torch.float32)


def make_inputs(w: Workload, seed: int = 0, device="cpu", request_id_base: int = 0) -> dict:
    """Draw one block's inputs for every request of workload ``w``.

    Returns a dict of tensors on ``device``:
      base [B,G,V], target [B,G+1,V], e_in [V,r], w_out [V,r] (workload dtype),
      anchor [B] i32, temperature [B] f32, request_id [B] u32 (as int32 storage),
      conf_logits [B,G] f32, pos_temp [G] f32, sps [B*(G+1)+1] f32.
    """
    B, G, V, r = w.B, w.G, w.V, w.r
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + zlib.crc32(w.name.encode()) % 997)
    dt = torch_dtype(w)
    f32 = torch.float32

    base_ext = torch.randn((B, G + 1, V), generator=g, device=device, dtype=f32) * w.u_sigma
    if w.spike:
        idx = torch.randint(0, V, (B, G + 1, 1), generator=g, device=device)
        base_ext.scatter_add_(2, idx, torch.full((B, G + 1, 1), w.spike, device=device, dtype=f32))
    base = base_ext[:, :G, :].to(dt).contiguous()
    if w.noise == "const":
        sig = torch.full((B, 1, 1), w.noise_sigma, device=device, dtype=f32)
    else:
        sig = (0.2 + 1.8 * torch.rand((B, 1, 1), generator=g, device=device, dtype=f32))
    # the target sees the stored (rounded) draft base plus noise
    target = base_ext.to(dt).to(f32)
    target += torch.randn((B, G + 1, V), generator=g, device=device, dtype=f32) * sig
    target = target.to(dt).contiguous()
    del base_ext

    e_in = (torch.randn((V, r), generator=g, device=device, dtype=f32) * 0.02).to(dt).contiguous()
    w_out = (torch.randn((V, r), generator=g, device=device, dtype=f32) * 0.02).to(dt).contiguous()
    anchor = torch.randint(0, V, (B,), generator=g, device=device, dtype=torch.int32)

    if w.temp == "one":
        temperature = torch.full((B,), w.temp_value, device=device, dtype=f32)
    elif w.temp == "mix_greedy":
        temperature = torch.full((B,), w.temp_value, device=device, dtype=f32)
        temperature[: B // 2] = 0.0
    else:
        temperature = 0.3 + 0.9 * torch.rand((B,), generator=g, device=device, dtype=f32)

    request_id = (torch.arange(B, device=device, dtype=torch.int64) + request_id_base).to(torch.int32)
    conf_logits = 1.0 + torch.randn((B, G), generator=g, device=device, dtype=f32)
    pos_temp = torch.linspace(1.0, 2.0, G, device=device, dtype=f32)
    sps = sps_table(B * (G + 1), device=device)
    return dict(base=base, target=target, e_in=e_in, w_out=w_out, anchor=anchor,
                temperature=temperature, request_id=request_id, conf_logits=conf_logits,
                pos_temp=pos_temp, sps=sps)


def make_rnn_head(w: Workload, seed: int = 0, device="cpu") -> dict:
    """Weights of a recurrent draft head for workload ``w`` (bf16):
    e_in [V,r], w_h [r,r] (row n: weights of state unit n), w_out [V,r]."""
    V, r = w.V, w.r
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000033 + 7 + zlib.crc32(w.name.encode()) % 991)
    f32 = torch.float32
    e_in = (torch.randn((V, r), generator=g, device=device, dtype=f32) * 0.5).to(torch.bfloat16)
    w_h = (torch.randn((r, r), generator=g, device=device, dtype=f32) * (0.9 / r ** 0.5)).to(torch.bfloat16)
    w_out = (torch.randn((V, r), generator=g, device=device, dtype=f32) * 0.05).to(torch.bfloat16)
    return dict(e_in=e_in.contiguous(), w_h=w_h.contiguous(), w_out=w_out.contiguous())
