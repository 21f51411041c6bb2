"""Stack-level checks through the C ABI: parity with the oracle, the circular
schedule, bit-exact slot bytes, residency invariance, staging engines,
registration rollback and lifecycle errors."""
import numpy as np
import pytest
import torch

import synth
from oracle import schedule as osched
from tests import helpers as H

dlo = pytest.importorskip("layerwise_weight_offload_slot_gb300")

pytestmark = pytest.mark.gpu

# small stacks that still span several GEMM tiles and a ragged tail
SMALL_DIT = synth.StackConfig("dit-small", synth.KIND_DIT, 6, 256, 4, 64, 512, 2, 200, cond_dim=256)
SMALL_VID = synth.StackConfig("video-small", synth.KIND_VIDEO, 4, 256, 2, 128, 512, 2, 300,
                              text_dim=192, text_tokens=77)
SMALL_VID_FP8 = SMALL_VID.with_(name="video-small-fp8", wdtype=synth.W_E4M3, master_fp32=True)
SMALL_VID_W8A8 = SMALL_VID.with_(name="video-small-w8a8", wdtype=synth.W_E4M3_A8, master_fp32=True)


def run(st, cfg, step=0):
    x, cond, ctx = H.device_inputs(cfg, step)
    out = st.forward(x, cond, ctx)
    torch.cuda.synchronize()
    st.wait()
    return x, cond, ctx, out


def test_tiny_stack_matches_oracle():
    cfg = synth.CFG_TINY
    st = H.make_stack(cfg)
    st.attach()
    x, cond, ctx, out = run(st, cfg)
    ref = H.oracle_forward(cfg, x, cond, ctx, H.oracle_blocks(cfg))
    err = H.rel_l2(out.float().cpu().numpy(), ref)
    print("tiny stack max rel L2", err)
    assert err <= 2e-2
    st.close()


@pytest.mark.parametrize("cfg", [SMALL_DIT, SMALL_VID, SMALL_VID_FP8, SMALL_VID_W8A8], ids=lambda c: c.name)
def test_small_stacks_match_oracle(cfg):
    st = H.make_stack(cfg)
    st.attach()
    x, cond, ctx, out = run(st, cfg)
    ref = H.oracle_forward(cfg, x, cond, ctx, H.oracle_blocks(cfg))
    y = out.float().cpu().numpy()
    err = H.rel_l2(y, ref)
    # the residual dominates x; also bound the error of the stack's update
    # y - x, allowing for the bf16 rounding of the output itself
    x0 = x.float().cpu().numpy().astype(np.float64)
    derr = H.rel_l2(y - x0, ref - x0)
    rounding = H.rel_l2(synth.round_bf16(ref.astype(np.float32)) - x0, ref - x0)
    print(cfg.name, "rel L2", err, "update rel L2", derr, "of which output rounding", rounding)
    tol = 5e-2 if synth.fp8_weights(cfg.wdtype) else 2e-2
    assert err <= tol and derr <= tol + 2 * rounding
    st.close()


@pytest.mark.parametrize("k", [0, 2, 5, 6])
@pytest.mark.parametrize("steps", [1, 3])
def test_schedule_log_and_slots(k, steps):
    cfg = SMALL_DIT
    st = H.make_stack(cfg)
    st.attach()
    st.set_resident(k)
    for s in range(steps):
        run(st, cfg, s)
    log = st.log()
    assert log == osched.schedule(cfg.n_blocks, k, steps)
    stats = st.stats()
    assert stats["stagings"] == (0 if k == cfg.n_blocks else 1 + steps * (cfg.n_blocks - k))
    # both slots hold the bytes of the block last staged into them
    for s in (0, 1):
        if stats["slot_block"][s] >= 0:
            assert st.verify_slot(s)
    if k < cfg.n_blocks:
        # the tail prefetch re-staged the first streamed block
        last_stage = [e for e in log if e[0] == "stage"][-1]
        assert last_stage[1] == k
    st.close()


def test_verify_slot_detects_wrong_block():
    cfg = SMALL_DIT
    st = H.make_stack(cfg)
    st.attach()
    run(st, cfg)
    s = st.stats()["slot_block"]
    other = (s[0] + 1) % cfg.n_blocks
    assert not st.verify_slot(0, other)
    assert st.verify_slot(0, s[0])
    st.close()


@pytest.mark.parametrize("cfg", [SMALL_DIT, SMALL_VID_W8A8], ids=lambda c: c.name)
def test_residency_invariance_bit_exact(cfg):
    outs = []
    for k in sorted({0, 2, cfg.n_blocks // 2 + 1, cfg.n_blocks}):
        st = H.make_stack(cfg)
        st.attach()
        st.set_resident(k)
        outs.append(run(st, cfg)[3].cpu())
        st.close()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_gather_staging_and_registered_memory_bit_exact():
    cfg = SMALL_VID
    outs = []
    for staging, mode in ((dlo.STAGE_MEMCPY, "pinned"), (dlo.STAGE_GATHER, "pinned"),
                          (dlo.STAGE_MEMCPY, "register"), (dlo.STAGE_GATHER, "register"),
                          (dlo.STAGE_PER_TENSOR, "register"), (dlo.STAGE_PER_TENSOR, "pinned"),
                          (dlo.STAGE_MEMCPY, "pageable")):
        st = H.make_stack(cfg, staging=staging, host_mode=mode)
        st.attach()
        if mode == "register":
            assert st.stats()["registered_ranges"] >= 1
        if mode == "pageable":
            assert st.stats()["registered_ranges"] == 0
        outs.append(run(st, cfg)[3].cpu())
        for s in (0, 1):
            assert st.verify_slot(s)
        stats = st.stats()
        per_stage = len(st.layout) if staging == dlo.STAGE_PER_TENSOR else 0
        if staging == dlo.STAGE_PER_TENSOR:
            assert stats["h2d_copies"] == per_stage * stats["stagings"]
        elif staging == dlo.STAGE_MEMCPY:
            assert stats["h2d_copies"] == stats["stagings"]
        st.close()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_steps_chain_and_restage():
    cfg = SMALL_DIT
    st = H.make_stack(cfg)
    st.attach()
    x, cond, ctx = H.device_inputs(cfg, 0)
    blocks = H.oracle_blocks(cfg)
    for s in range(3):
        cond = torch.from_numpy(synth.condition(cfg, s)).to(torch.bfloat16).cuda()
        out = st.forward(x, cond, ctx)
        torch.cuda.synchronize()
        ref = H.oracle_forward(cfg, x, cond, ctx, blocks)
        assert H.rel_l2(out.float().cpu().numpy(), ref) <= 2e-2
        x = out
    st.wait()
    st.close()


def test_forward_host_matches_device_forward():
    cfg = SMALL_VID
    st = H.make_stack(cfg)
    st.attach()
    x, cond, ctx, out = run(st, cfg)
    xh = x.cpu().view(torch.int16).numpy().copy()
    ch = cond.cpu().numpy().copy()
    th = ctx.cpu().view(torch.int16).numpy().copy()
    oh = np.empty_like(xh)
    st.forward_host(xh, ch, th, oh)
    np.testing.assert_array_equal(oh, out.cpu().view(torch.int16).numpy())
    st.close()


def test_registration_rollback_and_retry():
    cfg = SMALL_DIT
    st = H.make_stack(cfg, host_mode="register")
    # blocks are page-aligned and adjacent -> one merged range; force two
    # failures at the first register call, then retry succeeds
    dlo.dlo_debug_fail_register(1)
    with pytest.raises(dlo.DloError) as e:
        st.attach()
    assert e.value.status == dlo.EREGISTER
    assert st.stats()["registered_ranges"] == 0
    dlo.dlo_debug_fail_register(0)
    st.attach()
    assert st.stats()["registered_ranges"] == 1
    run(st, cfg)
    st.close()


def test_registration_budget_checked_before_mutation():
    cfg = SMALL_DIT
    st = H.make_stack(cfg, host_mode="register", register_budget_bytes=4096)
    with pytest.raises(dlo.DloError) as e:
        st.attach()
    assert e.value.status == dlo.EREGISTER and "budget" in str(e.value)
    assert st.stats()["registered_ranges"] == 0
    st.close()


def test_lifecycle_errors():
    cfg = SMALL_DIT
    st = H.make_stack(cfg)
    x, cond, ctx = H.device_inputs(cfg)
    with pytest.raises(dlo.DloError) as e:
        st.forward(x, cond, ctx)
    assert e.value.status == dlo.ESTATE
    st.attach()
    with pytest.raises(dlo.DloError) as e:
        st.attach()
    assert e.value.status == dlo.ESTATE
    with pytest.raises(dlo.DloError) as e:
        dlo.dlo_set_resident(st.ctx, [0] * 7)
    assert e.value.status == dlo.EINVAL
    st.set_resident(1)
    with pytest.raises(dlo.DloError) as e:
        st.set_resident(1)
    assert e.value.status == dlo.ESTATE
    xb = torch.zeros((cfg.batch, cfg.tokens + 1, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dlo.DloError) as e:
        st.forward(xb, cond, ctx)
    assert e.value.status == dlo.EINVAL
    run(st, cfg)
    assert st.close() == 0


def test_pageable_rejects_gather():
    cfg = SMALL_DIT
    st = H.make_stack(cfg, staging=dlo.STAGE_GATHER, host_mode="pageable")
    with pytest.raises(dlo.DloError) as e:
        st.attach()
    assert e.value.status == dlo.EINVAL
    st.close()


@pytest.mark.parametrize("cfg", [
    synth.StackConfig("dit-1block-1token", synth.KIND_DIT, 1, 128, 2, 64, 256, 1, 1, cond_dim=128),
    synth.StackConfig("dit-2blocks-ragged", synth.KIND_DIT, 2, 128, 2, 64, 256, 3, 129, cond_dim=128),
    synth.StackConfig("video-1token-1text", synth.KIND_VIDEO, 2, 128, 1, 128, 256, 1, 1, text_dim=64,
                      text_tokens=1),
    synth.StackConfig("video-hd64-ragged", synth.KIND_VIDEO, 3, 256, 4, 64, 512, 2, 257,
                      text_dim=128, text_tokens=130),
], ids=lambda c: c.name)
def test_degenerate_and_ragged_shapes(cfg):
    """One streamed block (re-staged into alternating slots every execution),
    one query token, one text token, ragged token counts past a tile edge."""
    st = H.make_stack(cfg)
    st.attach()
    for step in range(2):
        x, cond, ctx, out = run(st, cfg, step)
        ref = H.oracle_forward(cfg, x, cond, ctx, H.oracle_blocks(cfg))
        assert H.rel_l2(out.float().cpu().numpy(), ref) <= 2e-2
    log = st.log()
    assert log == osched.schedule(cfg.n_blocks, 0, 2)
    for s in (0, 1):
        assert st.verify_slot(s)
    st.close()


def test_smaller_batch_and_tokens_than_the_maximum():
    cfg = SMALL_VID
    st = H.make_stack(cfg)
    st.attach()
    small = cfg.with_(batch=1, tokens=77, text_tokens=5)
    x, cond, ctx = H.device_inputs(small)
    out = st.forward(x, cond, ctx)
    torch.cuda.synchronize()
    st.wait()
    ref = H.oracle_forward(small, x, cond, ctx, H.oracle_blocks(cfg))
    assert H.rel_l2(out.float().cpu().numpy(), ref) <= 2e-2
    st.close()


def _stack_output_digest(env_pdl: str) -> str:
    """sha256 of one small video stack's output, computed in a fresh process
    with DLO_PDL set as given (the switch is read once per process)."""
    import os
    import subprocess
    import sys
    code = (
        "import hashlib, torch, synth\n"
        "from tests import helpers as H\n"
        "cfg = synth.StackConfig('pdl', synth.KIND_VIDEO, 3, 256, 2, 128, 512, 2, 300,"
        " text_dim=192, text_tokens=77)\n"
        "st = H.make_stack(cfg); st.attach()\n"
        "x, c, t = H.device_inputs(cfg)\n"
        "y = st.forward(x, c, t); torch.cuda.synchronize(); st.wait()\n"
        "y = st.forward(y.clone(), c, t); torch.cuda.synchronize(); st.wait()\n"
        "print(hashlib.sha256(y.view(torch.int16).cpu().numpy().tobytes()).hexdigest())\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, DLO_PDL=env_pdl, PYTHONPATH=root)
    out = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    return out.stdout.strip().splitlines()[-1]


def test_programmatic_dependent_launch_changes_no_bit():
    assert _stack_output_digest("1") == _stack_output_digest("0")


def test_w8a16_widened_linears_match_oracle(tmp_path):
    """W8A16 linears with at least DLO_WIDEN_ROWS rows are widened to bf16 in
    the workspace and multiplied in bf16 (the 8192-token video block takes
    that path by default): inside the CTA-pair GEMM kernel (its CTAs widen the
    codes, meet at a grid barrier, then run the bf16 mainloop), or, where the
    tile model picks another kernel, by a separate widening kernel first.
    Forced here on the small E4M3 video stack (ragged rows, a 77-token text
    context), each in a process of its own: pairs forced (six linears widen
    inside the GEMM; the 154-row cross k|v is too short for a pair and widens
    separately), the tile model's picks (all seven widen separately), and no
    widening (the GEMMs widen each tile in their mainloop).  All three stay
    within the W8A16 stack tolerance of the oracle and of each other."""
    import os
    import subprocess
    import sys
    cfg = SMALL_VID_FP8
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import sys, numpy as np, torch\n"
        "from tests import helpers as H\n"
        "from tests.test_gpu_stack import SMALL_VID_FP8 as cfg\n"
        "import layerwise_weight_offload_slot_gb300 as dlo\n"
        "st = H.make_stack(cfg); st.attach(); st.set_timing(2)\n"
        "x, c, t = H.device_inputs(cfg)\n"
        "y = st.forward(x, c, t); torch.cuda.synchronize(); st.wait()\n"
        "np.save(sys.argv[1], y.float().cpu().numpy())\n"
        "print(st.stats()['kclass_launches'][dlo.KCLASS_NAMES.index('convert')])\n")
    runs = {"in_gemm": {"DLO_WIDEN_ROWS": "1", "DLO_GEMM_PAIR": "1", "DLO_GEMM_BN": "256"},
            "separate": {"DLO_WIDEN_ROWS": "1"},
            "mainloop": {"DLO_WIDEN_ROWS": "1000000000"}}
    outs = {}
    for name, env in runs.items():
        path = str(tmp_path / f"y_{name}.npy")
        r = subprocess.run([sys.executable, "-c", code, path], cwd=root, capture_output=True, text=True,
                           timeout=600, env=dict(os.environ, PYTHONPATH=root, **env))
        assert r.returncode == 0, r.stderr[-2000:]
        outs[name] = (np.load(path), int(r.stdout.split()[-1]))
    base = outs["mainloop"][1]
    assert outs["separate"][1] - base == 7 * cfg.n_blocks   # every linear: a widening launch
    assert outs["in_gemm"][1] - base == 1 * cfg.n_blocks    # only the cross k|v
    x, cond, ctx = H.device_inputs(cfg)
    ref = H.oracle_forward(cfg, x, cond, ctx, H.oracle_blocks(cfg))
    ym = outs["mainloop"][0]
    for name, (y, _) in outs.items():
        assert H.rel_l2(y, ref) <= 5e-2, name
        assert H.rel_l2(y, ym) <= 5e-2, name
        print(name, "vs in-mainloop widening: max |diff|", float(np.abs(y - ym).max()),
              "bit-identical", bool((y == ym).all()))


def test_device_wait_timeout_is_reported_and_the_context_survives():
    cfg = synth.CFG_TINY
    st = H.make_stack(cfg)
    st.attach()
    x, cond, ctx, out = run(st, cfg)
    dlo.dlo_debug_device_timeout(st.ctx)
    with pytest.raises(dlo.DloError) as e:
        st.wait(30000)
    assert e.value.status == dlo.ETIMEDOUT
    assert st.stats()["device_error"] == 1
    # the word was cleared; the next forward runs and matches the oracle
    x, cond, ctx, out = run(st, cfg)
    ref = H.oracle_forward(cfg, x, cond, ctx, H.oracle_blocks(cfg))
    assert H.rel_l2(out.float().cpu().numpy(), ref) <= 2e-2
    st.close()
