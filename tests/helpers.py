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
    fp8_lin = synth.fp8_weights(cfg.wdtype)
    fp8_act = cfg.wdtype == synth.W_E4M3_A8
    ps = params if params is not None else [synth.block_params(cfg, i) for i in range(cfg.n_blocks)]
    return [dit.prepare_block(p, fp8_linears=fp8_lin, fp8_activations=fp8_act) for p in ps]


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


# ---------------------------------------------------------------- multi-container stacks

def make_multi_stack(mc: synth.MultiConfig, *, staging=0, host_mode="pinned"):
    from layerwise_weight_offload_slot_gb300.stack import OffloadStack
    v = mc.video
    conts = [dict(block_kind=p.kind, n_blocks=p.n_blocks, heads=p.heads, head_dim=p.head_dim,
                  ffn=p.ffn, cond_dim=p.cond_dim, text_dim=p.text_dim,
                  max_text_tokens=p.text_tokens, wdtype=p.wdtype) for p in mc.parts]
    st = OffloadStack(containers=conts, hidden=mc.hidden, max_batch=mc.batch, max_tokens=mc.tokens,
                      staging=staging, host_mode=host_mode)
    st.pack_all(lambda i: synth.multi_block_params(mc, i))
    return st


def multi_inputs(mc: synth.MultiConfig, step: int = 0):
    """x, one conditioning tensor per container, the text context (or None)."""
    x = torch.from_numpy(synth.activations(mc.parts[0], step)).to(torch.bfloat16).cuda()
    conds = []
    for p in mc.parts:
        c = synth.condition(p, step)
        conds.append(torch.from_numpy(c).to(torch.bfloat16 if p.kind == synth.KIND_DIT
                                            else torch.float32).cuda())
    v = mc.video
    ctx = torch.from_numpy(synth.text_context(v, step)).to(torch.bfloat16).cuda() if v else None
    return x, conds, ctx


def oracle_multi(mc: synth.MultiConfig, x_bf16, conds, ctx):
    parts = []
    for p, c in zip(mc.parts, conds):
        blocks = oracle_blocks(p)
        parts.append((p.kind, c.float().cpu().numpy().astype(np.float64), blocks, p.heads))
    x = x_bf16.float().cpu().numpy().astype(np.float64)
    t = ctx.float().cpu().numpy().astype(np.float64) if ctx is not None else None
    return dit.multi_stack_forward(parts, x, t)
