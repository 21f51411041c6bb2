"""Seeded synthetic inputs for the streamed DiT block stack.

This module is shared by the tests, the benchmark and the CPU oracle's callers.
It draws random numbers and names tensors; it holds none of the method's
arithmetic (no normalisation, attention, GEMM, modulation or staging logic).

Workload shapes follow the five stack configurations of the layerwise-offload
workloads: a tiny DiT stack, a DiT-XL-like stack, a large video-DiT stack at
32760 tokens, the same stack with per-tensor FP8 linears at 8192 tokens, and
the staging/residency sweep at 8192 tokens.

Recipe (all seeded; seed 0 unless stated):
  * linear weights and biases: N(0, 0.02);
  * norm gains: 1 + N(0, 0.02); norm biases: N(0, 0.02);
  * video modulation table [6, D]: N(0, 0.02);
  * activations x: N(0, 1); text context: N(0, 1);
  * shared video modulation e [B, 6, D]: 0.1 * N(0, 1);
  * DiT timestep conditioning c: produced by `timestep_condition` below.
Weights that a configuration declares "bf16" are rounded to bf16 (RNE) here,
so both consumers see the same bf16-exact fp32 values.  Weights declared
"fp32 on host" are left as fp32 masters.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

KIND_DIT = 0      # DiT adaLN-zero block (self-attention only)
KIND_VIDEO = 1    # video-DiT block (self-attn, cross-attn to text, FFN)

W_BF16 = 0
W_E4M3 = 1
W_E4M3_A8 = 2     # E4M3 weights and dynamically quantised E4M3 linear inputs (W8A8)


def fp8_weights(wdtype: int) -> bool:
    return wdtype in (W_E4M3, W_E4M3_A8)


@dataclasses.dataclass(frozen=True)
class StackConfig:
    name: str
    kind: int
    n_blocks: int
    hidden: int
    heads: int
    head_dim: int
    ffn: int
    batch: int
    tokens: int
    cond_dim: int = 0          # DiT: width of the conditioning vector c
    text_dim: int = 0          # video: width of the text context
    text_tokens: int = 0       # video: number of text tokens
    wdtype: int = W_BF16
    master_fp32: bool = False  # weights kept as fp32 masters on the host
    steps: int = 1
    resident: int = 0
    seed: int = 0

    def with_(self, **kw) -> "StackConfig":
        return dataclasses.replace(self, **kw)


# The five stack workloads.
CFG_TINY = StackConfig("dit-tiny-4x256", KIND_DIT, 4, 256, 4, 64, 1024, 1, 256,
                       cond_dim=256, master_fp32=True, steps=1)
CFG_DITXL = StackConfig("dit-xl-28x1152-b2-n1024", KIND_DIT, 28, 1152, 16, 72, 4608, 2,
                        1024, cond_dim=1152, steps=10)
CFG_VIDEO = StackConfig("video-40x5120-n32760", KIND_VIDEO, 40, 5120, 40, 128, 13824, 1,
                        32760, text_dim=4096, text_tokens=512)
CFG_VIDEO_FP8 = StackConfig("video-fp8-40x5120-n8192", KIND_VIDEO, 40, 5120, 40, 128, 13824,
                            1, 8192, text_dim=4096, text_tokens=512, wdtype=W_E4M3,
                            master_fp32=True)
CFG_VIDEO_W8A8 = StackConfig("video-w8a8-40x5120-n8192", KIND_VIDEO, 40, 5120, 40, 128, 13824,
                             1, 8192, text_dim=4096, text_tokens=512, wdtype=W_E4M3_A8,
                             master_fp32=True)
CFG_SWEEP = StackConfig("video-sweep-40x5120-n8192", KIND_VIDEO, 40, 5120, 40, 128, 13824, 1,
                        8192, text_dim=4096, text_tokens=512)

CONFIGS = {c.name: c for c in (CFG_TINY, CFG_DITXL, CFG_VIDEO, CFG_VIDEO_FP8, CFG_VIDEO_W8A8,
                               CFG_SWEEP)}


@dataclasses.dataclass(frozen=True)
class MultiConfig:
    """A stack of several ordered block containers (e.g. double-stream blocks
    followed by single-stream blocks).  The parts share hidden, batch and
    tokens; part c draws its weights with its own seed, and its block j is
    block `first(c) + j` of the stack."""
    name: str
    parts: tuple
    steps: int = 1

    @property
    def n_blocks(self) -> int:
        return sum(p.n_blocks for p in self.parts)

    @property
    def hidden(self) -> int:
        return self.parts[0].hidden

    @property
    def batch(self) -> int:
        return self.parts[0].batch

    @property
    def tokens(self) -> int:
        return self.parts[0].tokens

    @property
    def video(self) -> "StackConfig | None":
        return next((p for p in self.parts if p.kind == KIND_VIDEO), None)

    def part_of(self, block: int) -> tuple[int, int]:
        for c, p in enumerate(self.parts):
            if block < p.n_blocks:
                return c, block
            block -= p.n_blocks
        raise IndexError("block out of range")


# Mixed stacks: video (cross-attention) blocks, then DiT adaLN blocks.
MULTI_TINY = MultiConfig("mixed-video2-dit3-d128", (
    StackConfig("mixed-tiny-video", KIND_VIDEO, 2, 128, 2, 64, 256, 2, 40, text_dim=64,
                text_tokens=9, seed=0),
    StackConfig("mixed-tiny-dit", KIND_DIT, 3, 128, 2, 64, 512, 2, 40, cond_dim=128, seed=7)))
MULTI_FP8_TINY = MultiConfig("mixed-video2fp8-dit2-d256", (
    StackConfig("mixed-fp8-video", KIND_VIDEO, 2, 256, 4, 64, 512, 1, 130, text_dim=128,
                text_tokens=17, wdtype=W_E4M3, master_fp32=True, seed=3),
    StackConfig("mixed-fp8-dit", KIND_DIT, 2, 256, 2, 128, 768, 1, 130, cond_dim=256, seed=5)))
MULTI_DITXL = MultiConfig("mixed-video8-dit20-d1152-b2-n1024", (
    StackConfig("mixed-xl-video", KIND_VIDEO, 8, 1152, 16, 72, 4608, 2, 1024, text_dim=4096,
                text_tokens=256, seed=0),
    StackConfig("mixed-xl-dit", KIND_DIT, 20, 1152, 16, 72, 4608, 2, 1024, cond_dim=1152,
                seed=11)), steps=10)
MULTI_CONFIGS = {c.name: c for c in (MULTI_TINY, MULTI_FP8_TINY, MULTI_DITXL)}


def multi_block_params(mc: MultiConfig, block: int) -> dict[str, np.ndarray]:
    c, j = mc.part_of(block)
    return block_params(mc.parts[c], j)


def param_specs(cfg: StackConfig):
    """Ordered (name, shape, role) of one block's tensors.

    role is one of "linear_w", "linear_b", "norm_w", "norm_b", "table".
    Linear weights are [out_features, in_features] (y = x W^T + b).
    """
    D, F = cfg.hidden, cfg.ffn
    if cfg.kind == KIND_DIT:
        C = cfg.cond_dim
        return [
            ("adaLN.weight", (6 * D, C), "linear_w"),
            ("adaLN.bias", (6 * D,), "linear_b"),
            ("attn.qkv.weight", (3 * D, D), "linear_w"),
            ("attn.qkv.bias", (3 * D,), "linear_b"),
            ("attn.proj.weight", (D, D), "linear_w"),
            ("attn.proj.bias", (D,), "linear_b"),
            ("mlp.fc1.weight", (F, D), "linear_w"),
            ("mlp.fc1.bias", (F,), "linear_b"),
            ("mlp.fc2.weight", (D, F), "linear_w"),
            ("mlp.fc2.bias", (D,), "linear_b"),
        ]
    Dt = cfg.text_dim
    return [
        ("modulation", (6, D), "table"),
        ("self_attn.q.weight", (D, D), "linear_w"),
        ("self_attn.k.weight", (D, D), "linear_w"),
        ("self_attn.v.weight", (D, D), "linear_w"),
        ("self_attn.q.bias", (D,), "linear_b"),
        ("self_attn.k.bias", (D,), "linear_b"),
        ("self_attn.v.bias", (D,), "linear_b"),
        ("self_attn.o.weight", (D, D), "linear_w"),
        ("self_attn.o.bias", (D,), "linear_b"),
        ("self_attn.norm_q.weight", (D,), "norm_w"),
        ("self_attn.norm_k.weight", (D,), "norm_w"),
        ("norm_cross.weight", (D,), "norm_w"),
        ("norm_cross.bias", (D,), "norm_b"),
        ("cross_attn.q.weight", (D, D), "linear_w"),
        ("cross_attn.q.bias", (D,), "linear_b"),
        ("cross_attn.k.weight", (D, Dt), "linear_w"),
        ("cross_attn.v.weight", (D, Dt), "linear_w"),
        ("cross_attn.k.bias", (D,), "linear_b"),
        ("cross_attn.v.bias", (D,), "linear_b"),
        ("cross_attn.o.weight", (D, D), "linear_w"),
        ("cross_attn.o.bias", (D,), "linear_b"),
        ("cross_attn.norm_q.weight", (D,), "norm_w"),
        ("cross_attn.norm_k.weight", (D,), "norm_w"),
        ("ffn.fc1.weight", (F, D), "linear_w"),
        ("ffn.fc1.bias", (F,), "linear_b"),
        ("ffn.fc2.weight", (D, F), "linear_w"),
        ("ffn.fc2.bias", (D,), "linear_b"),
    ]


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence(list(key))))


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even), returned as fp32."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def block_params(cfg: StackConfig, block: int) -> dict[str, np.ndarray]:
    """Seeded fp32 tensors of one block (bf16-exact unless `cfg.master_fp32`)."""
    out = {}
    for t, (name, shape, role) in enumerate(param_specs(cfg)):
        g = _rng(cfg.seed, 1000 + block, t)
        a = g.standard_normal(shape, dtype=np.float32) * np.float32(0.02)
        if role == "norm_w":
            a = a + np.float32(1.0)
        # fp32 masters are kept for every tensor of an fp32-master stack, and for
        # the linear weights of an FP8 stack (the quantiser's input); all other
        # tensors are bf16-exact.
        keep_master = cfg.master_fp32 and (cfg.wdtype == W_BF16 or role == "linear_w")
        if not keep_master:
            a = round_bf16(a)
        out[name] = a
    return out


def stack_params(cfg: StackConfig, threads: int = 8) -> list[dict[str, np.ndarray]]:
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda i: block_params(cfg, i), range(cfg.n_blocks)))


def activations(cfg: StackConfig, step: int = 0) -> np.ndarray:
    """x [B, N, D], N(0,1), rounded to bf16 (the stack's input type)."""
    g = _rng(cfg.seed, 1, step)
    return round_bf16(g.standard_normal((cfg.batch, cfg.tokens, cfg.hidden), dtype=np.float32))


def text_context(cfg: StackConfig, step: int = 0) -> np.ndarray:
    """ctx [B, L, Dt], N(0,1), bf16-exact (video blocks only)."""
    g = _rng(cfg.seed, 2, step)
    return round_bf16(g.standard_normal((cfg.batch, cfg.text_tokens, cfg.text_dim),
                                        dtype=np.float32))


def video_modulation(cfg: StackConfig, step: int = 0) -> np.ndarray:
    """Shared modulation e [B, 6, D] = 0.1 * N(0,1), fp32 (video blocks only)."""
    g = _rng(cfg.seed, 3, step)
    return (g.standard_normal((cfg.batch, 6, cfg.hidden), dtype=np.float32)
            * np.float32(0.1))


def timesteps(cfg: StackConfig, step: int = 0) -> np.ndarray:
    """Timesteps [B] of one denoising step: t = 500 for a single-step stack,
    else U[0, 1000) seeded per step."""
    if cfg.steps == 1 and step == 0:
        return np.full((cfg.batch,), 500.0, dtype=np.float64)
    return _rng(cfg.seed, 4, step).uniform(0.0, 1000.0, size=(cfg.batch,))


def sinusoidal(t: np.ndarray, dim: int) -> np.ndarray:
    """Standard sinusoidal timestep features [cos | sin], max period 10000."""
    half = dim // 2
    freqs = np.exp(-math.log(10000.0) * np.arange(half, dtype=np.float64) / half)
    args = np.asarray(t, dtype=np.float64)[:, None] * freqs[None, :]
    return np.concatenate([np.cos(args), np.sin(args)], axis=1)


def timestep_condition(cfg: StackConfig, step: int = 0) -> np.ndarray:
    """DiT conditioning c [B, cond_dim] (bf16-exact fp32), outside the block stack.

    For a stack whose cond_dim equals the sinusoid width (256) c is the
    sinusoidal embedding itself; otherwise c comes from a fixed, resident
    timestep embedder (sinusoidal 256 -> Linear -> SiLU -> Linear, weights
    N(0, 0.02), seed 1) that is input preparation, not part of the stack.
    """
    t = timesteps(cfg, step)
    f = sinusoidal(t, 256)
    if cfg.cond_dim == 256:
        return round_bf16(f.astype(np.float32))
    g = _rng(1, 5)
    w1 = g.standard_normal((cfg.cond_dim, 256)) * 0.02
    b1 = g.standard_normal((cfg.cond_dim,)) * 0.02
    w2 = g.standard_normal((cfg.cond_dim, cfg.cond_dim)) * 0.02
    b2 = g.standard_normal((cfg.cond_dim,)) * 0.02
    h = f @ w1.T + b1
    h = h / (1.0 + np.exp(-h))
    return round_bf16((h @ w2.T + b2).astype(np.float32))


def condition(cfg: StackConfig, step: int = 0) -> np.ndarray:
    """The per-step conditioning input of the stack (c for DiT, e for video)."""
    if cfg.kind == KIND_DIT:
        return timestep_condition(cfg, step)
    return video_modulation(cfg, step)


def staging_bytes(size: int, seed: int = 0) -> np.ndarray:
    """Random uint8 payload for the staging sweep."""
    return _rng(seed, 6, size).integers(0, 256, size=size, dtype=np.uint8)
