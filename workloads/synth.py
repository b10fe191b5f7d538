"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random tensors with the shapes and distributions of the
workloads; it holds none of the layer's arithmetic (no gating, no dispatch, no
expert FFN, no combine).  Both the CUDA path and the CPU oracle are fed from it.

Workloads (the shapes of the MoE layer studied in "Enabling trillion-parameter
models on AWS EFA", section "Evaluation": hidden size 7168, token batches up to
a few thousand per rank, top-R routing over E experts):

    tiny      T=256    d=512  E=8   R=2 f=1024  plain router
    mid       T=4096   d=2048 E=64  R=6 f=1408  Zipf(s=1.0) per-expert router bias
    large     T=8192   d=7168 E=384 R=8 f=2048  unbiased router ("uniform")
    large_hot                                    + bias on 4 hot experts (25% of assignments)
    dispatch  T=128..65536 d=7168 E=256 R=8     routing drawn directly, identity experts
    train     T=16384  d=4096 E=128 R=8 f=1536  fwd+bwd, loss = sum(y * g)

Seeds are ``workload_index * 1000 + tensor_id`` so every tensor is reproducible
on its own.  x, W_g, the router bias and g always come from torch's CPU
generator.  The expert weights come from the generator of ``weight_device``
(torch's CUDA generator is a different stream than the CPU one for the same
seed); the large workloads draw them on the GPU because drawing 17e9 weights on
the host takes minutes.

Weight layout (the usual ``nn.Linear`` [out, in] convention):
    W1, W3: bf16 [E, f, d]   (a = x @ W1[e].T,  b = x @ W3[e].T)
    W2:     bf16 [E, d, f]   (o = h @ W2[e].T)
    W_g:    fp32 [d, E]      (logits = x @ W_g + bias)
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass, field, replace

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOT_BIAS_FILE = os.path.join(os.path.dirname(_HERE), "tests", "golden", "hot_bias.json")


@dataclass(frozen=True)
class Workload:
    name: str
    index: int          # position in the workload list; seeds derive from it
    T: int
    d: int
    E: int
    R: int
    f: int = 0          # 0 = identity experts (dispatch + combine only)
    router: str = "plain"   # plain | zipf | hot | drawn
    zipf_s: float = 0.0
    hot_experts: int = 0
    train: bool = False
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny": Workload("tiny", 0, T=256, d=512, E=8, R=2, f=1024),
    "mid": Workload("mid", 1, T=4096, d=2048, E=64, R=6, f=1408, router="zipf", zipf_s=1.0),
    "large": Workload("large", 2, T=8192, d=7168, E=384, R=8, f=2048),
    "large_hot": Workload("large_hot", 2, T=8192, d=7168, E=384, R=8, f=2048, router="hot",
                          hot_experts=4),
    "dispatch": Workload("dispatch", 3, T=8192, d=7168, E=256, R=8, f=0, router="drawn"),
    "dispatch_zipf": Workload("dispatch_zipf", 3, T=8192, d=7168, E=256, R=8, f=0,
                              router="drawn", zipf_s=1.2),
    "train": Workload("train", 4, T=16384, d=4096, E=128, R=8, f=1536, train=True),
}

DISPATCH_T_SWEEP = [2 ** k for k in range(7, 17)]   # 128 .. 65536

# tensor ids
_X, _WG, _W1, _W3, _W2, _BIAS, _G, _ROUTE, _RW = range(1, 10)


def workload(name: str, **overrides) -> Workload:
    """A named workload, optionally with some fields replaced (e.g. a smaller T)."""
    return replace(WORKLOADS[name], **overrides)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(shape, std, device, seed, chunk_rows=None):
    """N(0, std^2) values rounded to bf16 by torch, drawn in leading-dim chunks."""
    g = _gen(device, seed)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    n0 = shape[0]
    step = chunk_rows or n0
    for i in range(0, n0, step):
        j = min(n0, i + step)
        tmp = torch.randn((j - i,) + tuple(shape[1:]), generator=g, device=device,
                          dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        out[i:j].copy_(tmp)
        del tmp
    return out


def hot_bias_value(wl: Workload) -> float:
    """Bias added to the hot experts' logits; stored by tests/golden/make_hot_bias.py."""
    with open(_HOT_BIAS_FILE) as fh:
        table = json.load(fh)
    return float(table[wl.name]["beta"])


def hot_experts(wl: Workload):
    """The seeded set of hot experts of a ``hot`` workload."""
    g = _gen("cpu", wl.index * 1000 + _BIAS)
    return torch.randperm(wl.E, generator=g)[: wl.hot_experts]


def router_bias(wl: Workload, device="cpu"):
    """Per-expert router bias (fp32 [E]) or None.

    zipf: b_e = -s * ln(k_e), k a seeded permutation of 1..E; the E/8 experts of
          largest rank k are switched off (b = -30) so zero-row experts always occur.
    hot:  +beta on ``hot_experts`` seeded experts, 0 elsewhere.
    """
    if wl.router == "zipf":
        g = _gen("cpu", wl.index * 1000 + _BIAS)
        k = torch.randperm(wl.E, generator=g).to(torch.float64) + 1.0
        b = -wl.zipf_s * torch.log(k)
        off = k > wl.E - wl.E // 8
        b[off] = -30.0
        return b.to(torch.float32).to(device)
    if wl.router == "hot":
        b = torch.zeros(wl.E, dtype=torch.float32)
        b[hot_experts(wl)] = hot_bias_value(wl)
        return b.to(device)
    return None


def router_inputs(wl: Workload):
    """x bf16 [T,d], W_g fp32 [d,E] and the router bias, all on the host."""
    base = wl.index * 1000
    x = _normal_bf16((wl.T, wl.d), 1.0, "cpu", base + _X)
    w_gate = torch.randn((wl.d, wl.E), generator=_gen("cpu", base + _WG),
                         dtype=torch.float32) * 0.02
    return x, w_gate, router_bias(wl)


def layer_inputs(wl: Workload, device="cpu", weight_device=None, with_grad=None):
    """x, W_g, bias, W1, W3, W2 (and g for training) for a layer workload."""
    assert wl.f > 0
    base = wl.index * 1000
    wdev = weight_device or device
    chunk = max(1, (1 << 28) // max(1, wl.f * wl.d))   # ~1 GiB fp32 temporaries at most
    x, w_gate, bias = router_inputs(wl)
    out = {
        "x": x.to(device),
        "w_gate": w_gate.to(device),
        "bias": None if bias is None else bias.to(device),
        "W1": _normal_bf16((wl.E, wl.f, wl.d), 0.02, wdev, base + _W1, chunk).to(device),
        "W3": _normal_bf16((wl.E, wl.f, wl.d), 0.02, wdev, base + _W3, chunk).to(device),
        "W2": _normal_bf16((wl.E, wl.d, wl.f), 0.02, wdev, base + _W2, chunk).to(device),
    }
    if wl.train if with_grad is None else with_grad:
        out["g"] = _normal_bf16((wl.T, wl.d), 1.0, "cpu", base + _G).to(device)
    return out


def shared_expert_inputs(wl: Workload, fs: int, device="cpu"):
    """Seeded weights of one shared expert: W1, W3 bf16 [fs, d], W2 bf16 [d, fs],
    ~N(0, 0.02) like the routed experts'."""
    base = wl.index * 1000 + 500
    return {"W1": _normal_bf16((fs, wl.d), 0.02, device, base + _W1),
            "W3": _normal_bf16((fs, wl.d), 0.02, device, base + _W3),
            "W2": _normal_bf16((wl.d, fs), 0.02, device, base + _W2)}


def drawn_routing(wl: Workload, device="cpu"):
    """Routing drawn directly (dispatch-only workloads): idx int32 [T,R], w fp32 [T,R].

    Each token picks R distinct experts without replacement with probability
    proportional to k_e^{-s} (k a seeded permutation of 1..E; s=0 is uniform),
    by the Gumbel-top-R construction.  The R weights are positive and normalised
    to sum to 1.
    """
    g = _gen("cpu", wl.index * 1000 + _ROUTE)
    k = torch.randperm(wl.E, generator=g).to(torch.float64) + 1.0
    logp = -wl.zipf_s * torch.log(k)
    idx = torch.empty((wl.T, wl.R), dtype=torch.int32)
    step = 8192
    for i in range(0, wl.T, step):
        j = min(wl.T, i + step)
        u = torch.rand((j - i, wl.E), generator=g, dtype=torch.float64).clamp_(1e-300, 1.0)
        keys = logp - torch.log(-torch.log(u))
        idx[i:j] = torch.topk(keys, wl.R, dim=1).indices.to(torch.int32)
    u = torch.rand((wl.T, wl.R), generator=_gen("cpu", wl.index * 1000 + _RW),
                   dtype=torch.float64) + 0.5
    w = (u / u.sum(dim=1, keepdim=True)).to(torch.float32)
    x = _normal_bf16((wl.T, wl.d), 1.0, "cpu", wl.index * 1000 + _X)
    return {"x": x.to(device), "topk_idx": idx.to(device), "topk_w": w.to(device)}


def bf16_bits(t: torch.Tensor):
    """A bf16 tensor's raw bit patterns as a numpy uint16 array (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def flops_fwd(wl: Workload) -> float:
    """Algorithmic FLOPs of the expert FFN forward (gate-up + down), real rows only."""
    n = wl.T * wl.R
    return 6.0 * n * wl.d * wl.f


def flops_gate(wl: Workload) -> float:
    return 2.0 * wl.T * wl.d * wl.E


def describe(wl: Workload) -> str:
    s = f"{wl.name} T={wl.T} d={wl.d} E={wl.E} R={wl.R}"
    if wl.f:
        s += f" f={wl.f}"
    if wl.router == "zipf":
        s += f" zipf_s={wl.zipf_s}"
    if wl.router == "hot":
        s += f" hot_experts={wl.hot_experts}"
    if wl.router == "drawn":
        s += f" drawn_routing zipf_s={wl.zipf_s}"
    return s


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["Workload", "WORKLOADS", "DISPATCH_T_SWEEP", "workload", "layer_inputs",
           "router_inputs", "hot_experts",
           "drawn_routing", "router_bias", "bf16_bits", "flops_fwd", "flops_gate", "describe",
           "ceil_div"]
