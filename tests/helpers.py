"""Shared helpers of the GPU tests: build an OffloadStack from a synthetic
workload, upload inputs, run the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import dit


def make_stack(cfg: synth.StackConfig, *, staging=0, host_mode="pinned", blocks=None,
               register_budget_bytes=0):
    from layerwise_weight_offload_slot_gb300.stack import OffloadStack
    st = OffloadStack(block_kind=cfg.kind, n_blocks=cfg.n_blocks, hidden=cfg.hidden,
                      heads=cfg.heads, head_dim=cfg.head_dim, ffn=cfg.ffn, cond_dim=cfg.cond_dim,
                      text_dim=cfg.text_dim, max_batch=cfg.batch, max_tokens=cfg.tokens,
                      max_text_tokens=cfg.text_tokens, wdtype=cfg.wdtype, staging=staging,
                      host_mode=host_mode, register_budget_bytes=register_budget_bytes)
    st.pack_all(blocks if blocks is not None else (lambda i: synth.block_params(cfg, i)))
    return st


def device_inputs(cfg: synth.StackConfig, step: int = 0):
    x = torch.from_numpy(synth.activations(cfg, step)).to(torch.bfloat16).cuda()
    if cfg.kind == synth.KIND_DIT:
        cond = torch.from_numpy(synth.condition(cfg, step)).to(torch.bfloat16).cuda()
        ctx = None
    else:
        cond = torch.from_numpy(synth.condition(cfg, step)).float().cuda()
        ctx = torch.from_numpy(synth.text_context(cfg, step)).to(torch.bfloat16).cuda()
    return x, cond, ctx


def oracle_blocks(cfg: synth.StackConfig, params=None):
    fp8_lin = cfg.wdtype == synth.W_E4M3
    ps = params if params is not None else [synth.block_params(cfg, i) for i in range(cfg.n_blocks)]
    return [dit.prepare_block(p, fp8_linears=fp8_lin) for p in ps]


def oracle_forward(cfg: synth.StackConfig, x_bf16: torch.Tensor, cond, ctx, blocks):
    """Oracle stack on the exact device inputs (copied back to the host)."""
    x = x_bf16.float().cpu().numpy().astype(np.float64)
    c = cond.float().cpu().numpy().astype(np.float64)
    t = ctx.float().cpu().numpy().astype(np.float64) if ctx is not None else None
    return dit.stack_forward(cfg.kind, x, c, t, blocks, cfg.heads)


def rel_l2(y, ref):
    return dit.max_rel_l2(np.asarray(y, dtype=np.float64), ref)


def bf16(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()
