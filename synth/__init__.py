"""Seeded synthetic inputs for the fp8 MoE verify layer.

This module feeds both the CUDA path and the CPU oracle and holds none of the
layer's arithmetic.  It builds what a GLM-5.2-FP8-class checkpoint and a verify
batch look like:

* activations x: bf16, N(0, 1); pad rows filled with NaN;
* router weight Wr: fp32 [E, H], N(0, 1/H), so logits are about N(0, 1);
* correction bias: fp32 [E], U(-0.1, 0.1) plus a routing skew per workload;
* expert weights: N(0, 0.02) in fp32, then per 128x128 block
  scale = amax / 448 and codes = torch's float8_e4m3fn cast of w / scale
  (a synthetic block-fp8 checkpoint: e4m3 codes + fp32 block scales);
  gate/up [E, I, H], down [E, H, I], output-major; shared expert(s) likewise.

Every tensor draws from its own torch generator seeded with
fnv1a64(name) ^ seed, so tensors are independent of one another and of the
order they are made in.  The same call on the same device and torch build
gives the same bytes; CPU and CUDA generators give different streams, so a
test generates once and hands the same bytes to both sides.

The pages quote their numbers on the real GLM-5.2-FP8 checkpoint and real
prompts; neither is available here, so these seeded draws of the same shapes
stand in for them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class LayerShape:
    hidden: int
    inter: int
    n_experts: int
    n_groups: int
    topk_groups: int
    topk: int
    n_shared: int = 1
    routed_scaling: float = 2.5


GLM52 = LayerShape(hidden=6144, inter=2048, n_experts=256, n_groups=8, topk_groups=4,
                   topk=8, n_shared=1, routed_scaling=2.5)
# GLM-5.2 router shape (hidden 6144, 256 experts, top-8 of top-4 groups) with
# 128-wide experts: the small kernels at their real size, for profiler captures
GLM52_ROUTER = LayerShape(hidden=6144, inter=128, n_experts=256, n_groups=8, topk_groups=4,
                          topk=8, n_shared=1, routed_scaling=2.5)
# GLM-5.2 expert shape with 32 experts: the small case for full profiler captures
# (about 1.2 GB of weights: above L2, a few GB on the device at most)
GLM52_E32 = LayerShape(hidden=6144, inter=2048, n_experts=32, n_groups=4, topk_groups=2,
                       topk=8, n_shared=1, routed_scaling=2.5)
TINY = LayerShape(hidden=256, inter=128, n_experts=16, n_groups=4, topk_groups=2, topk=4,
                  n_shared=1, routed_scaling=2.5)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    rows: int
    routing: str = "uniform"          # uniform | hot | zipf
    pads: tuple = ()                  # pad row indices (x = NaN, not routed)
    hot_per_group: int = 0            # routing == "hot": hot experts per group
    hot_delta: float = 0.0            # routing == "hot": bias lift of hot experts
    zipf_s: float = 1.1               # routing == "zipf": exponent
    zipf_tau: float = 0.1             # routing == "zipf": bias = tau * ln(p) + U
    seed: int = 0
    note: str = ""


WORKLOADS = {
    "tiny": Workload("tiny", TINY, rows=8, note="CPU-oracle scale, 8 rows"),
    "verify8": Workload("verify8", GLM52, rows=8, routing="hot", hot_per_group=10,
                        hot_delta=1.0,
                        note="single-request verify: 1 committed + 7 drafts; skewed "
                             "router so about 40 distinct experts are hit"),
    "verify64": Workload("verify64", GLM52, rows=64, pads=(7, 23, 39, 55),
                         note="batched verify: 8 requests x span 8, 4 pad rows"),
    "decode512": Workload("decode512", GLM52, rows=512, routing="zipf",
                          note="mixed decode batch, Zipf(1.1) expert popularity"),
    "prefill4096": Workload("prefill4096", GLM52, rows=4096,
                            note="prefill chunk, uniform routing"),
    "profile8": Workload("profile8", GLM52_E32, rows=8,
                         note="8 rows on 32 experts of the GLM-5.2 shape, for profiler "
                              "captures"),
    "profile8r": Workload("profile8r", GLM52_ROUTER, rows=8, routing="hot", hot_per_group=10,
                          hot_delta=1.0,
                          note="verify8's routing at 128-wide experts, for profiler captures of "
                               "the router, union, dispatch and combine kernels"),
    "profile128": Workload("profile128", GLM52_E32, rows=128,
                           note="128 rows on 32 experts of the GLM-5.2 shape (about 32 rows per "
                                "expert, the 32-row tile of mixed decode batches): profiler "
                                "captures"),
    "profile1024": Workload("profile1024", GLM52_E32, rows=1024,
                            note="1024 rows on 32 experts of the GLM-5.2 shape (256 rows per "
                                 "expert, the 64-row tile): prefill-like profiler captures"),
    "profile512": Workload("profile512", GLM52_E32, rows=512,
                           note="512 rows on 32 experts of the GLM-5.2 shape (128 rows per "
                                "expert, the 64-row tile with the deeper ring of calls of at "
                                "most 512 rows): decode-batch-like profiler captures"),
    "profile4096r": Workload("profile4096r", GLM52_ROUTER, rows=4096,
                             note="prefill4096's routing at 128-wide experts: the large-R "
                                  "router at its real size, for profiler captures"),
}


def _fnv1a64(s: str) -> int:
    h = 0xCBF29CE484222325
    for b in s.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _gen(name: str, seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((_fnv1a64(name) ^ (seed & 0xFFFFFFFFFFFFFFFF)) & 0x7FFFFFFFFFFFFFFF)
    return g


def _randn(shape, name, seed, device, dtype=torch.float32):
    return torch.randn(shape, generator=_gen(name, seed, device), device=device, dtype=dtype)


def _rand(shape, name, seed, device):
    return torch.rand(shape, generator=_gen(name, seed, device), device=device,
                      dtype=torch.float32)


def quantize_blocks(w: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """[..., N, K] fp32 -> (e4m3 codes uint8 [..., N, K], fp32 scales [..., N/128, K/128]).

    Synthetic-checkpoint quantisation (not a step of the layer): scale =
    amax/448 per 128x128 block (1 for an all-zero block), codes from torch's
    float8_e4m3fn cast.
    """
    *lead, N, K = w.shape
    b = w.reshape(*lead, N // 128, 128, K // 128, 128)
    amax = b.abs().amax(dim=(-3, -1))
    s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (b / s[..., :, None, :, None]).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).reshape(*lead, N, K).contiguous(), s.contiguous()


def make_router_inputs(wl: Workload, device="cpu") -> dict:
    """x (bf16 [R,H]), row_valid (uint8 [R]), wr (fp32 [E,H]), bias (fp32 [E])."""
    sh, R, seed = wl.shape, wl.rows, wl.seed
    H, E, G = sh.hidden, sh.n_experts, sh.n_groups
    x = _randn((R, H), "x", seed, device).to(torch.bfloat16)
    valid = torch.ones(R, dtype=torch.uint8, device=device)
    for p in wl.pads:
        x[p] = float("nan")
        valid[p] = 0
    wr = _randn((E, H), "router.weight", seed, device) * (1.0 / math.sqrt(H))
    bias = (_rand((E,), "router.bias", seed, device) * 0.2 - 0.1)
    if wl.routing == "hot":
        epg = E // G
        # hot_per_group experts of every group, picked by a seeded permutation
        perm = torch.argsort(_rand((G, epg), "router.hot", seed, "cpu"), dim=1)
        hot = (perm[:, :wl.hot_per_group] + torch.arange(G)[:, None] * epg).flatten()
        lift = torch.zeros(E)
        lift[hot] = wl.hot_delta
        bias = bias + lift.to(device)
    elif wl.routing == "zipf":
        # popularity p_rank ~ rank^-s over a seeded permutation of the experts
        ranks = torch.argsort(_rand((E,), "router.zipf_perm", seed, "cpu")) + 1
        p = ranks.double() ** (-wl.zipf_s)
        p = p / p.sum()
        bias = bias + (wl.zipf_tau * torch.log(p)).float().to(device)
    elif wl.routing != "uniform":
        raise ValueError(f"unknown routing {wl.routing}")
    return {"x": x.contiguous(), "row_valid": valid, "wr": wr.contiguous(),
            "bias": bias.contiguous()}


def make_expert_weights(wl: Workload, device="cpu", chunk: int = 16) -> dict:
    """Routed and shared expert tensors (codes + block scales)."""
    sh, seed = wl.shape, wl.seed
    E, S, H, I = sh.n_experts, sh.n_shared, sh.hidden, sh.inter
    out = {}
    for prefix, n in (("", E), ("sh_", S)):
        for proj, (N, K) in (("gate", (I, H)), ("up", (I, H)), ("down", (H, I))):
            codes = torch.empty((n, N, K), dtype=torch.uint8, device=device)
            scales = torch.empty((n, N // 128, K // 128), dtype=torch.float32, device=device)
            for e0 in range(0, n, chunk):
                e1 = min(n, e0 + chunk)
                w = _randn((e1 - e0, N, K), f"{prefix}{proj}[{e0}:{e1}]", seed, device) * 0.02
                q, s = quantize_blocks(w)
                codes[e0:e1] = q
                scales[e0:e1] = s
                del w, q, s
            key_w = f"{prefix}{proj}" if prefix else f"w_{proj}"
            key_s = f"{prefix}s_{proj}" if prefix else f"s_{proj}"
            out[key_w] = codes
            out[key_s] = scales
    return out


def make_layer(wl: Workload, device="cpu") -> dict:
    t = make_router_inputs(wl, device)
    t.update(make_expert_weights(wl, device))
    return t


def to_numpy(t: dict) -> dict:
    """Host numpy view of a layer dict (bf16 as uint16 bit patterns)."""
    out = {}
    for k, v in t.items():
        if v is None:
            out[k] = None
        elif v.dtype == torch.bfloat16:
            out[k] = v.detach().cpu().view(torch.int16).numpy().view("uint16")
        else:
            out[k] = v.detach().cpu().numpy()
    return out


def variant(wl: Workload, **kw) -> Workload:
    return replace(wl, **kw)
