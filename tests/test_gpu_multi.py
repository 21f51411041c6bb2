"""Stacks of several ordered block containers through the C ABI: parity with
the oracle, the one circular schedule over all containers, slots shared by
blocks of different sizes, residency across the container boundary, and the
equivalence of a split container with the unsplit one."""
import numpy as np
import pytest
import torch

import synth
from oracle import schedule as osched
from tests import helpers as H

dlo = pytest.importorskip("layerwise_weight_offload_slot_gb300")

pytestmark = pytest.mark.gpu


def run(st, mc, step=0):
    x, conds, ctx = H.multi_inputs(mc, step)
    out = st.forward(x, conds, ctx)
    torch.cuda.synchronize()
    st.wait()
    return x, conds, ctx, out


@pytest.mark.parametrize("mc", [synth.MULTI_TINY, synth.MULTI_FP8_TINY], ids=lambda c: c.name)
def test_mixed_stack_matches_oracle(mc):
    st = H.make_multi_stack(mc)
    assert st.multi and len(set(st.container_bytes)) == 2
    assert st.slot_bytes >= max(st.container_bytes)
    st.attach()
    tol = 5e-2 if any(synth.fp8_weights(p.wdtype) for p in mc.parts) else 2e-2
    for step in range(2):
        x, conds, ctx, out = run(st, mc, step)
        ref = H.oracle_multi(mc, x, conds, ctx)
        err = H.rel_l2(out.float().cpu().numpy(), ref)
        print(mc.name, "step", step, "max rel L2", err)
        assert err <= tol
    st.close()


def test_mixed_stack_schedule_slots_and_sizes():
    mc = synth.MULTI_TINY
    st = H.make_multi_stack(mc)
    st.attach()
    steps = 3
    for s in range(steps):
        run(st, mc, s)
    assert st.log() == osched.schedule(mc.n_blocks, 0, steps)
    stats = st.stats()
    # each staging moves exactly that block's own bytes
    n = mc.n_blocks
    assert stats["stagings"] == steps * n + 1   # the prime, then one prefetch per execution
    expected = sum(st.block_sizes[b] for kind, b, _ in st.log() if kind == "stage")
    assert stats["staged_bytes"] == expected
    # both slots hold bit-exact copies of the blocks last staged into them,
    # also when those blocks come from different containers
    for s in (0, 1):
        assert st.verify_slot(s)
    held = st.stats()["slot_block"]
    for s in (0, 1):
        for b in range(n):
            assert st.verify_slot(s, b) == (held[s] == b), (s, b)
    st.close()


def test_residency_across_the_container_boundary_is_bit_exact():
    mc = synth.MULTI_TINY
    outs = {}
    for k in (0, 1, 2, 3, 5):
        st = H.make_multi_stack(mc)
        st.attach()
        st.set_resident(k)
        x, conds, ctx = H.multi_inputs(mc, 0)
        y = st.forward(x, conds, ctx)
        torch.cuda.synchronize()
        st.wait()
        outs[k] = y.cpu()
        if k < mc.n_blocks:
            assert st.log() == osched.schedule(mc.n_blocks, k, 1)
        st.close()
    for k in (1, 2, 3, 5):
        assert torch.equal(outs[k], outs[0]), k


def test_split_container_is_bit_identical_to_one_container():
    # the same five DiT blocks as one container and as containers of 2 + 3
    cfg = synth.StackConfig("dit-split", synth.KIND_DIT, 5, 256, 4, 64, 512, 2, 150, cond_dim=256)
    one = H.make_stack(cfg)
    one.attach()
    x, cond, _ = H.device_inputs(cfg)
    y1 = one.forward(x, cond)
    torch.cuda.synchronize()
    one.wait()
    from layerwise_weight_offload_slot_gb300.stack import OffloadStack
    part = dict(block_kind=cfg.kind, heads=cfg.heads, head_dim=cfg.head_dim, ffn=cfg.ffn,
                cond_dim=cfg.cond_dim)
    two = OffloadStack(containers=[dict(part, n_blocks=2), dict(part, n_blocks=3)], hidden=cfg.hidden,
                       max_batch=cfg.batch, max_tokens=cfg.tokens)
    two.pack_all(lambda i: synth.block_params(cfg, i))
    two.attach()
    y2 = two.forward(x, cond)             # one cond serves containers of one kind
    torch.cuda.synchronize()
    two.wait()
    assert torch.equal(y1, y2)
    y3 = two.forward(x, [cond, cond])
    torch.cuda.synchronize()
    two.wait()
    assert torch.equal(y1, y3)
    one.close()
    two.close()


def test_mixed_stack_argument_errors():
    mc = synth.MULTI_TINY
    st = H.make_multi_stack(mc)
    st.attach()
    x, conds, ctx = H.multi_inputs(mc, 0)
    # containers of different kinds need one conditioning each
    with pytest.raises(dlo.DloError) as e:
        st.forward(x, conds[1], ctx)
    assert e.value.status == dlo.EINVAL
    with pytest.raises(dlo.DloError) as e:
        st.forward(x, conds, None)      # the video container needs the text context
    assert e.value.status == dlo.EINVAL
    with pytest.raises(dlo.DloError) as e:
        st.forward_host(x.cpu().float().numpy(), conds[0].cpu().numpy(), ctx.cpu().float().numpy(),
                        np.empty(x.shape, np.uint16))
    assert e.value.status == dlo.EUNSUPPORTED
    # the context still works after the rejected calls
    y = st.forward(x, conds, ctx)
    torch.cuda.synchronize()
    st.wait()
    ref = H.oracle_multi(mc, x, conds, ctx)
    assert H.rel_l2(y.float().cpu().numpy(), ref) <= 2e-2
    st.close()


def test_mixed_stack_registered_and_pageable_hosts():
    mc = synth.MULTI_TINY
    ref = None
    for mode in ("pinned", "register", "pageable"):
        st = H.make_multi_stack(mc, host_mode=mode)
        st.attach()
        x, conds, ctx, out = run(st, mc, 0)
        if ref is None:
            ref = out.cpu()
        else:
            assert torch.equal(out.cpu(), ref), mode
        for s in (0, 1):
            assert st.verify_slot(s)
        st.close()
