"""Seeded synthetic workloads shaped like the source pages' MoE layers.

This module only draws inputs (activations, BF16 weight stacks, routing ids and
scores).  It holds none of the layer's arithmetic, so both the CUDA path and
the CPU oracle can take their inputs from it.

The routing ids and scores stand in for the router that sits upstream of the
expert layer: softmax over N(0,1) logits and top-k, renormalised (the pages'
plain top-k router, "Performance" section of Megatron-LM PR #8262), except
where a workload asks for Zipf-skewed or uniform expert choice.
"""
from dataclasses import dataclass, field

import torch

BASE_SEED = 1234


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    K: int
    act: str            # "relu2" or "swiglu"
    x_dist: str = "outliers"       # "outliers" | "logspread" | "normal"
    routing: str = "softmax_topk"  # "softmax_topk" | "zipf" | "uniform"
    empty_experts: int = 0

    @property
    def N1(self):
        return 2 * self.I if self.act == "swiglu" else self.I

    def with_T(self, T):
        d = dict(self.__dict__)
        d["T"] = T
        d["name"] = f"{self.name.split('@')[0]}@T{T}"
        return Workload(**d)

    def with_E(self, E):
        d = dict(self.__dict__)
        d["E"] = E
        d["name"] = f"{self.name}@E{E}"
        return Workload(**d)


# The five workload shapes (tiny squared-ReLU; SwiGLU E64; mid-scale Zipf; DeepSeek-like
# H7168/I2048/E256; the pages' benchmark shape H7168/I3072/E384 on one GPU).
TINY_RELU2 = Workload("tiny_relu2_T16_H256_I512_E8_K2", 16, 256, 512, 8, 2, "relu2")
SWIGLU_E64 = Workload("swiglu_T128_H2048_I1024_E64_K8", 128, 2048, 1024, 64, 8, "swiglu")
MID_ZIPF = Workload("relu2_T2048_H4096_I2048_E128_K6_zipf", 2048, 4096, 2048, 128, 6, "relu2",
                    x_dist="logspread", routing="zipf", empty_experts=4)
DSV3_LIKE = Workload("swiglu_H7168_I2048_E256_K8", 128, 7168, 2048, 256, 8, "swiglu",
                     x_dist="normal", routing="uniform")
PAGES_E384 = Workload("swiglu_H7168_I3072_E384_K6", 512, 7168, 3072, 384, 6, "swiglu",
                      x_dist="normal")
# The squared-ReLU layer of the GB300 table in Megatron-LM PR #8262, "Performance":
# H7168 / I2048 / 256 experts / plain top-8 over N(0,1) activations.
PAGES_GB300_RELU2 = Workload("relu2_H7168_I2048_E256_K8", 128, 7168, 2048, 256, 8, "relu2",
                             x_dist="normal")

# A compute-regime probe outside the pages' workloads: 8 experts of the
# H7168 / I2048 SwiGLU layer, top-2 of uniform routing over 65536 tokens gives
# ~16k routes per expert, far past the ~530 at which the grouped GEMMs stop
# being weight-streaming bound, so it measures the tensor pipe.
COMPUTE_PROBE = Workload("swiglu_H7168_I2048_E8_K2_compute", 65536, 7168, 2048, 8, 2, "swiglu",
                         x_dist="normal", routing="uniform")

ALL = {w.name: w for w in [TINY_RELU2, SWIGLU_E64, MID_ZIPF, DSV3_LIKE, PAGES_E384,
                             PAGES_GB300_RELU2, COMPUTE_PROBE]}


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_x(wl: Workload, device="cpu", seed=BASE_SEED + 1):
    """Token activations [T,H] bf16."""
    g = _gen(seed, device)
    x = torch.randn(wl.T, wl.H, generator=g, device=device, dtype=torch.float32)
    if wl.x_dist == "outliers":
        mask = torch.rand(wl.T, wl.H, generator=g, device=device) < 0.01
        x = torch.where(mask, x * 20.0, x)
    elif wl.x_dist == "logspread":
        u = torch.rand(wl.T, 1, generator=g, device=device) * 4.0 - 2.0
        x = x * torch.pow(10.0, u)
    return x.to(torch.bfloat16)


def make_weights(wl: Workload, device="cpu", seed=BASE_SEED):
    """BF16 FC1 [E,N1,H] (canonical [gate; up] for SwiGLU) and FC2 [E,H,I] stacks,
    N(0, 1/sqrt(fan_in)), generated one expert at a time to bound peak memory."""
    w1 = torch.empty(wl.E, wl.N1, wl.H, dtype=torch.bfloat16, device=device)
    w2 = torch.empty(wl.E, wl.H, wl.I, dtype=torch.bfloat16, device=device)
    g1 = _gen(seed + 2, device)
    g2 = _gen(seed + 3, device)
    s1 = 1.0 / wl.H ** 0.5
    s2 = 1.0 / wl.I ** 0.5
    for e in range(wl.E):
        w1[e] = (torch.randn(wl.N1, wl.H, generator=g1, device=device) * s1).to(torch.bfloat16)
        w2[e] = (torch.randn(wl.H, wl.I, generator=g2, device=device) * s2).to(torch.bfloat16)
    return w1, w2


def make_routing(wl: Workload, device="cpu", seed=BASE_SEED + 4):
    """Routing ids int32 [T,K] and fp32 scores [T,K]."""
    g = _gen(seed, device)
    T, E, K = wl.T, wl.E, wl.K
    if wl.routing == "softmax_topk":
        logits = torch.randn(T, E, generator=g, device=device)
        probs = torch.softmax(logits, dim=-1)
        # ties go to the lower expert id: stable descending sort
        order = torch.sort(probs, dim=-1, descending=True, stable=True).indices[:, :K]
        w = torch.gather(probs, 1, order)
        w = w / w.sum(dim=-1, keepdim=True)
        return order.to(torch.int32).contiguous(), w.float().contiguous()
    if wl.routing == "uniform":
        keys = torch.rand(T, E, generator=g, device=device)
        ids = torch.topk(keys, K, dim=-1).indices
        w = torch.softmax(torch.randn(T, K, generator=g, device=device), dim=-1)
        return ids.to(torch.int32).contiguous(), w.float().contiguous()
    if wl.routing == "zipf":
        perm = torch.randperm(E, generator=g, device=device)
        rank = torch.empty(E, device=device)
        rank[perm] = torch.arange(1, E + 1, device=device, dtype=torch.float32)
        p = rank.pow(-1.1)
        if wl.empty_experts:
            p[perm[E - wl.empty_experts:]] = 0.0   # the rarest experts never chosen
        logp = torch.log(p)
        gumbel = -torch.log(-torch.log(torch.rand(T, E, generator=g, device=device).clamp_min(1e-20)))
        ids = torch.topk(logp.unsqueeze(0) + gumbel, K, dim=-1).indices
        w = torch.softmax(torch.randn(T, K, generator=g, device=device), dim=-1)
        return ids.to(torch.int32).contiguous(), w.float().contiguous()
    raise ValueError(wl.routing)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (for the oracle)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
