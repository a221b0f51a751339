"""Seeded synthetic inputs for the displaced-patch layer ops.

This module is shared by the oracle tests, the GPU parity tests, the smoke
check and the benchmark.  It holds shapes and random draws only: none of the
method's arithmetic lives here.  Every tensor is drawn on the CPU with a seeded
``torch.Generator`` so that both sides of a parity test see the same values.

Workload shapes follow the SDXL U-Net levels the displaced-patch pages talk
about ("DistriFusion: Distributed Parallel Inference for High-Resolution
Diffusion Models", reader's notes, Background: SDXL at 1024x1024; Introduction
para. 5: 3840x3840 with classifier-free-guidance batch split).

Draw recipe (seed = 1000 * workload.index + 10 * step + tensor_id):
  * activations ~ N(0, 1); stale = fresh + stale_scale * N(0, 1);
  * weights ~ N(0, 1 / fan_in) (fan_in = 9 * C_in for the conv, the input
    width for a linear map);
  * GroupNorm gamma = 1 + 0.1 * N(0, 1), beta = 0.1 * N(0, 1);
  * guidance maps eps_u, eps_c i.i.d. N(0, 1) in fp32.
  For bf16 workloads every draw is rounded to bf16 (round-to-nearest-even)
  and both sides consume the rounded values.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

# tensor ids inside one (workload, step) seed block
T_FRESH, T_STALE_NOISE, T_CONV_W, T_GAMMA, T_BETA = 0, 1, 2, 3, 4
T_WQ, T_WK, T_WV, T_WO = 5, 6, 7, 8
T_CTX, T_XWK, T_XWV, T_XWQ, T_XWO = 9, 10, 11, 12, 13  # cross-attention
T_EPS_U, T_EPS_C = 14, 15
T_ATTN_X = 16


@dataclasses.dataclass(frozen=True)
class ConvShape:
    B: int
    H: int
    W: int
    C: int
    P: int


@dataclasses.dataclass(frozen=True)
class AttnShape:
    B: int
    H: int  # token grid height (patches are bands of H)
    W: int
    C: int
    heads: int
    head_dim: int
    P: int
    n_ctx: int = 0
    c_ctx: int = 0

    @property
    def N(self) -> int:
        return self.H * self.W


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    dtype: str  # "f32" or "bf16"
    conv: Optional[ConvShape] = None
    groups: int = 32
    eps: float = 1e-5
    attn: Optional[AttnShape] = None
    cfg_shape: Optional[tuple] = None
    cfg_scale: float = 7.5
    displaced_steps: int = 1
    stale_scale: float = 0.05


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_fp32", 1, "f32",
                 conv=ConvShape(1, 32, 32, 64, 2),
                 attn=AttnShape(1, 32, 32, 64, 1, 64, 2)),
        Workload("sdxl_1024_conv", 2, "bf16",
                 conv=ConvShape(1, 128, 128, 320, 4), displaced_steps=4),
        Workload("sdxl_1024_attn", 3, "bf16",
                 attn=AttnShape(1, 64, 64, 640, 10, 64, 4, n_ctx=77, c_ctx=2048)),
        Workload("sdxl_2048", 4, "bf16",
                 conv=ConvShape(1, 256, 256, 320, 8),
                 attn=AttnShape(1, 128, 128, 640, 10, 64, 8)),
        Workload("sdxl_3840_cfg", 5, "bf16",
                 conv=ConvShape(2, 480, 480, 320, 8),
                 attn=AttnShape(2, 240, 240, 640, 10, 64, 8, n_ctx=77, c_ctx=2048),
                 cfg_shape=(4, 480, 480)),
    ]
}


def torch_dtype(dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def seed_of(index: int, step: int, tensor_id: int) -> int:
    return 1000 * index + 10 * step + tensor_id


def normal(shape, seed: int, std: float = 1.0, mean: float = 0.0,
           dtype: str = "f32") -> torch.Tensor:
    """N(mean, std^2) draw on the CPU, rounded to ``dtype`` (RNE for bf16)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    t = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch_dtype(dtype))


def perturbed(base: torch.Tensor, seed: int, scale: float) -> torch.Tensor:
    """base + scale * N(0, 1), drawn in fp32 and rounded to base's dtype."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    noise = torch.randn(tuple(base.shape), generator=g, dtype=torch.float32)
    return (base.float() + scale * noise).to(base.dtype)


def activation_steps(shape, index: int, steps: int, scale: float, dtype: str,
                     tensor_id: int = T_FRESH):
    """Fresh activations for steps 0..steps: F_0 ~ N(0,1), F_s = F_{s-1} + scale*N(0,1).

    With the stale buffer at step s holding F_{s-1}, stale - fresh is
    scale * N(0,1) in distribution, as the workloads state.
    """
    out = [normal(shape, seed_of(index, 0, tensor_id), dtype=dtype)]
    for s in range(1, steps + 1):
        out.append(perturbed(out[-1], seed_of(index, s, tensor_id), scale))
    return out


def conv_weight(C_out: int, C_in: int, seed: int, dtype: str) -> torch.Tensor:
    """[C_out, C_in, 3, 3] (torch order), N(0, 1/(9*C_in))."""
    return normal((C_out, C_in, 3, 3), seed, std=(9.0 * C_in) ** -0.5, dtype=dtype)


def linear_weight(out_f: int, in_f: int, seed: int, dtype: str) -> torch.Tensor:
    """[out, in] (torch Linear order), N(0, 1/in)."""
    return normal((out_f, in_f), seed, std=float(in_f) ** -0.5, dtype=dtype)


def gn_affine(C: int, index: int):
    """(gamma, beta) fp32 [C]: gamma = 1 + 0.1 N(0,1), beta = 0.1 N(0,1)."""
    gamma = normal((C,), seed_of(index, 0, T_GAMMA), std=0.1, mean=1.0)
    beta = normal((C,), seed_of(index, 0, T_BETA), std=0.1)
    return gamma, beta


def attn_weights(a: AttnShape, index: int, dtype: str):
    C = a.C
    return {
        "wq": linear_weight(C, C, seed_of(index, 0, T_WQ), dtype),
        "wk": linear_weight(C, C, seed_of(index, 0, T_WK), dtype),
        "wv": linear_weight(C, C, seed_of(index, 0, T_WV), dtype),
        "wo": linear_weight(C, C, seed_of(index, 0, T_WO), dtype),
    }


def cross_weights(a: AttnShape, index: int, dtype: str):
    C = a.C
    return {
        "wq": linear_weight(C, C, seed_of(index, 0, T_XWQ), dtype),
        "wk": linear_weight(C, a.c_ctx, seed_of(index, 0, T_XWK), dtype),
        "wv": linear_weight(C, a.c_ctx, seed_of(index, 0, T_XWV), dtype),
        "wo": linear_weight(C, C, seed_of(index, 0, T_XWO), dtype),
    }


def context(a: AttnShape, index: int, dtype: str) -> torch.Tensor:
    return normal((a.B, a.n_ctx, a.c_ctx), seed_of(index, 0, T_CTX), dtype=dtype)


def guidance_maps(shape, index: int):
    """(eps_u, eps_c), fp32, i.i.d. N(0, 1)."""
    return (normal(shape, seed_of(index, 0, T_EPS_U)),
            normal(shape, seed_of(index, 0, T_EPS_C)))


def to_f64(t: torch.Tensor):
    """Exact upcast of a CPU tensor (fp32 or bf16) to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


# ------------------------------------------------------------ block chain
@dataclasses.dataclass(frozen=True)
class ChainShape:
    """One U-Net level stepped as a ResNet block + transformer block:
    latent B x H x W x C in P bands, G GroupNorm groups, `heads` heads of
    C / heads, text context n_ctx x c_ctx, feed-forward width ff_mult * C."""
    name: str
    index: int
    B: int
    H: int
    W: int
    C: int
    heads: int
    P: int
    G: int = 32
    n_ctx: int = 77
    c_ctx: int = 2048
    ff_mult: int = 4
    stale_scale: float = 0.05


CHAINS = {
    c.name: c
    for c in [
        # small enough for the fp64 oracle, several tiles of every kernel
        ChainShape("chain_small", 6, 2, 16, 16, 320, 5, 4, n_ctx=77, c_ctx=256),
        # SDXL at 3840px, level 2 of the down path (latent 480 -> 240 x 240 x 640)
        ChainShape("sdxl_3840_level2", 7, 2, 240, 240, 640, 10, 8),
    ]
}


def chain_weights(ch: ChainShape, dtype: str = "bf16"):
    """Weights of the chain in torch layouts (conv [C, C, 3, 3], Linear [out,
    in]; ff1 is [2 F, C]: value rows then gate rows).  Weights ~ N(0, 1/fan_in)
    in `dtype`; biases ~ 0.1 N(0, 1), affine gains 1 + 0.1 N(0, 1) and shifts
    0.1 N(0, 1), all fp32.  Seeds 1000 * index + 100 + k, k the name's rank."""
    C, F, X = ch.C, ch.ff_mult * ch.C, ch.c_ctx
    spec = [
        ("gn1_g", (C,), "gain"), ("gn1_b", (C,), "shift"), ("conv1_w", (C, C, 3, 3), 9 * C),
        ("conv1_b", (C,), "shift"), ("gn2_g", (C,), "gain"), ("gn2_b", (C,), "shift"),
        ("conv2_w", (C, C, 3, 3), 9 * C), ("conv2_b", (C,), "shift"),
        ("gn_g", (C,), "gain"), ("gn_b", (C,), "shift"), ("pi_w", (C, C), C),
        ("pi_b", (C,), "shift"), ("ln1_g", (C,), "gain"), ("ln1_b", (C,), "shift"),
        ("wq", (C, C), C), ("wk", (C, C), C), ("wv", (C, C), C), ("wo", (C, C), C),
        ("ln2_g", (C,), "gain"), ("ln2_b", (C,), "shift"), ("xq", (C, C), C),
        ("xk", (C, X), X), ("xv", (C, X), X), ("xo", (C, C), C),
        ("ln3_g", (C,), "gain"), ("ln3_b", (C,), "shift"), ("ff1_w", (2 * F, C), C),
        ("ff1_b", (2 * F,), "shift"), ("ff2_w", (C, F), F), ("ff2_b", (C,), "shift"),
        ("po_w", (C, C), C), ("po_b", (C,), "shift"),
    ]
    out = {}
    for k, (name, shape, kind) in enumerate(spec):
        seed = 1000 * ch.index + 100 + k
        if kind == "gain":
            out[name] = normal(shape, seed, std=0.1, mean=1.0)
        elif kind == "shift":
            out[name] = normal(shape, seed, std=0.1)
        else:
            out[name] = normal(shape, seed, std=float(kind) ** -0.5, dtype=dtype)
    return out


def chain_inputs(ch: ChainShape, steps: int, dtype: str = "bf16"):
    """Level inputs for steps 0..steps (F_s = F_{s-1} + stale_scale N(0, 1))
    and the text context, both in `dtype`."""
    xs = activation_steps((ch.B, ch.H, ch.W, ch.C), ch.index, steps, ch.stale_scale, dtype,
                          tensor_id=T_FRESH)
    ctx = normal((ch.B, ch.n_ctx, ch.c_ctx), seed_of(ch.index, 0, T_CTX), dtype=dtype)
    return xs, ctx
