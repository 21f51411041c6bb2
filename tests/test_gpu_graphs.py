"""Whole-forward CUDA graphs (dlo_set_graphs): a graph-launched forward gives
the same bits, staging order, slot contents, log and counters as the same
forward enqueued directly, across steps whose first streamed block sits in
either slot, argument changes, timing switches (and per-kernel timing inside
the graphs), residency, several
containers, the host-buffer entry point and opaque byte blocks."""
import numpy as np
import pytest
import torch

import synth
from oracle import schedule as osched
from tests import helpers as H

dlo = pytest.importorskip("layerwise_weight_offload_slot_gb300")

pytestmark = pytest.mark.gpu

DIT5 = synth.StackConfig("dit-graph", synth.KIND_DIT, 5, 256, 4, 64, 512, 2, 200, cond_dim=256)
VID3 = synth.StackConfig("video-graph", synth.KIND_VIDEO, 3, 256, 2, 128, 512, 2, 150,
                         text_dim=192, text_tokens=40)

COUNTERS = ("forwards", "stagings", "staged_bytes", "streamed_execs", "kernel_launches", "h2d_copies",
            "slot_block")


def _stack(cfg, graphs, k=0, **kw):
    st = H.make_stack(cfg, **kw)
    st.attach()
    if k:
        st.set_resident(k)
    st.set_graphs(graphs)
    return st


def _steps(st, cfg, steps, chain=True):
    """Forwards on fixed input/output buffers (as a sampler loop would),
    each step's output copied out; the next step's input is that output."""
    x, cond, ctx = H.device_inputs(cfg, 0)
    out = torch.empty_like(x)
    outs = []
    for s in range(steps):
        st.forward(x, cond, ctx, out=out)
        torch.cuda.synchronize()
        outs.append(out.clone())
        if chain:
            x.copy_(out)
    st.wait()
    return outs


@pytest.mark.parametrize("k", [0, 1, 2], ids=["k0-odd", "k1-even", "k2-odd"])
def test_graph_steps_are_bit_identical_to_direct_steps(k):
    cfg = DIT5
    steps = 5
    a = _stack(cfg, False, k)
    b = _stack(cfg, True, k)
    oa = _steps(a, cfg, steps)
    ob = _steps(b, cfg, steps)
    for s in range(steps):
        assert torch.equal(oa[s], ob[s]), s
    assert b.log() == a.log() == osched.schedule(cfg.n_blocks, k, steps)
    sa, sb = a.stats(), b.stats()
    for f in COUNTERS:
        assert sa[f] == sb[f], f
    # first forward direct; an odd number of streamed blocks alternates the
    # parity, so two graphs are captured, an even number needs one
    n_graphs = 2 if (cfg.n_blocks - k) % 2 else 1
    assert sb["graph_captures"] == n_graphs
    assert sb["graph_launches"] == steps - 1
    assert sa["graph_captures"] == sa["graph_launches"] == 0
    for s in (0, 1):
        assert b.verify_slot(s)
    a.close()
    b.close()


def test_graph_output_matches_oracle():
    cfg = VID3
    st = _stack(cfg, True)
    x, cond, ctx = H.device_inputs(cfg, 0)
    out = torch.empty_like(x)
    ref = H.oracle_forward(cfg, x, cond, ctx, H.oracle_blocks(cfg))
    for _ in range(3):
        st.forward(x, cond, ctx, out=out)
        torch.cuda.synchronize()
        assert H.rel_l2(out.float().cpu().numpy(), ref) <= 2e-2
    st.wait()
    assert st.stats()["graph_launches"] >= 1
    st.close()


@pytest.mark.parametrize("n", [4, 5])
def test_ping_pong_buffers_keep_their_graphs(n):
    """x -> y, y -> x, ... (one graph per buffer direction and parity), and
    a fifth argument set evicts the least recently used of four graphs."""
    cfg = DIT5.with_(n_blocks=n)
    a = _stack(cfg, False)
    b = _stack(cfg, True)
    x0, cond, _ = H.device_inputs(cfg, 0)
    bufs = {m: [x0.clone(), torch.empty_like(x0)] for m in ("a", "b")}
    for i in range(8):
        for m, st in (("a", a), ("b", b)):
            p, q = bufs[m][i % 2], bufs[m][(i + 1) % 2]
            st.forward(p, cond, out=q)
        torch.cuda.synchronize()
        assert torch.equal(bufs["a"][(i + 1) % 2], bufs["b"][(i + 1) % 2]), i
    sb = b.stats()
    assert sb["graph_captures"] == 2 and sb["graph_launches"] == 7
    # more argument sets than the cache holds: still the same bits
    extra = [torch.empty_like(x0) for _ in range(5)]
    for i in range(10):
        for m, st in (("a", a), ("b", b)):
            st.forward(bufs[m][0], cond, out=extra[i % 5] if m == "b" else bufs[m][1])
        torch.cuda.synchronize()
        assert torch.equal(extra[i % 5], bufs["a"][1]), i
    a.wait()
    b.wait()
    assert a.log() == b.log()
    assert b.stats()["graph_captures"] == 2 + 10   # more keys than entries, cycling: all miss
    a.close()
    b.close()


def test_new_arguments_are_captured_again():
    cfg = DIT5.with_(n_blocks=4)
    a = _stack(cfg, False)
    b = _stack(cfg, True)
    x, cond, _ = H.device_inputs(cfg, 0)
    x2, cond2, _ = H.device_inputs(cfg, 1)
    B2, N2 = 1, 137
    x3 = x2[:B2, :N2].contiguous()
    c3 = cond2[:B2].contiguous()
    seq = [(x, cond), (x, cond), (x2, cond), (x2, cond2), (x3, c3), (x3, c3), (x, cond)]
    for xi, ci in seq:
        ya = a.forward(xi, ci)
        yb = b.forward(xi, ci)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb)
    a.wait()
    b.wait()
    assert a.log() == b.log()
    assert b.stats()["graph_captures"] >= 4
    a.close()
    b.close()


def test_timing_switch_between_graph_and_direct_forwards():
    cfg = DIT5
    a = _stack(cfg, False)
    b = _stack(cfg, True)
    x, cond, _ = H.device_inputs(cfg, 0)
    out_a, out_b = torch.empty_like(x), torch.empty_like(x)
    for s in range(6):
        level = 1 if s in (2, 3) else 0
        b.set_timing(level)
        a.forward(x, cond, out=out_a)
        b.forward(x, cond, out=out_b)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b), s
        for slot in (0, 1):
            assert b.verify_slot(slot)
    b.wait()
    assert a.log() == b.log()
    sb = b.stats()
    assert sb["graph_launches"] >= 2 and sb["timed_execs"] == 2 * cfg.n_blocks
    # turning graphs off frees them; forwards continue directly
    b.set_graphs(False)
    y = b.forward(x, cond)
    ya = a.forward(x, cond)
    torch.cuda.synchronize()
    assert torch.equal(y, ya)
    a.close()
    b.close()


def test_kernel_timing_inside_graphs():
    """Timing level 3 keeps graphs on: per-kernel event pairs are nodes of the
    captured graph.  Each forward is counted once per kernel, as the direct
    level-2 forward counts it; results stay bit-identical."""
    cfg = DIT5
    a = _stack(cfg, False)
    b = _stack(cfg, True)
    a.set_timing(2)
    b.set_timing(3)
    x, cond, _ = H.device_inputs(cfg, 0)
    out_a, out_b = torch.empty_like(x), torch.empty_like(x)
    steps = 6
    for s in range(steps):
        if s == 4:
            b.set_timing(0)      # a graph captured at another level is not reused
        a.forward(x, cond, out=out_a)
        b.forward(x, cond, out=out_b)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b), s
    b.set_timing(3)
    b.forward(x, cond, out=out_b)   # the level-3 graph again: reads the last launch first
    a.forward(x, cond, out=out_a)
    torch.cuda.synchronize()
    a.wait()
    b.wait()
    assert torch.equal(out_a, out_b)
    sa, sb = a.stats(), b.stats()
    assert sb["graph_launches"] >= 5 and sb["graph_captures"] >= 2
    assert a.log() == b.log()
    # b timed 5 forwards (steps 0-3 and the last), a all 7
    for j, name in enumerate(dlo.KCLASS_NAMES):
        na, nb = sa["kclass_launches"][j], sb["kclass_launches"][j]
        assert na % 7 == 0 and nb * 7 == na * 5, name
        if nb:
            assert sb["kclass_ms"][j] > 0
            assert sb["kclass_flops"][j] * 7 == pytest.approx(sa["kclass_flops"][j] * 5)
            assert sb["kclass_bytes"][j] * 7 == pytest.approx(sa["kclass_bytes"][j] * 5)
    assert sb["timed_execs"] == 0      # level 3 times kernels only
    a.close()
    b.close()


def test_graphs_with_several_containers():
    mc = synth.MULTI_TINY
    ref = None
    for graphs in (False, True):
        st = H.make_multi_stack(mc)
        st.attach()
        st.set_graphs(graphs)
        x, conds, ctx = H.multi_inputs(mc, 0)
        out = torch.empty_like(x)
        outs = []
        for _ in range(4):
            st.forward(x, conds, ctx, out=out)
            torch.cuda.synchronize()
            outs.append(out.clone())
        st.wait()
        if ref is None:
            ref = (outs, st.log())
        else:
            assert all(torch.equal(p, q) for p, q in zip(ref[0], outs))
            assert st.log() == ref[1]
            assert st.stats()["graph_launches"] == 3
        for s in (0, 1):
            assert st.verify_slot(s)
        st.close()


def test_graphs_with_host_buffers_and_registered_memory():
    cfg = VID3
    res = []
    for graphs in (False, True):
        st = _stack(cfg, graphs, host_mode="register")
        x, cond, ctx = H.device_inputs(cfg, 0)
        xh = x.cpu().view(torch.int16).numpy().copy()
        ch = cond.cpu().numpy().copy()
        th = ctx.cpu().view(torch.int16).numpy().copy()
        outs = []
        for _ in range(3):
            oh = np.empty_like(xh)
            st.forward_host(xh, ch, th, oh)
            outs.append(oh)
        res.append(outs)
        if graphs:
            assert st.stats()["graph_launches"] == 2
        st.close()
    for p, q in zip(*res):
        np.testing.assert_array_equal(p, q)


def test_graphs_with_byte_blocks_and_gather_staging():
    from layerwise_weight_offload_slot_gb300.stack import OffloadStack
    size, n = 4 << 20, 3
    for staging in (0, 1):
        st = OffloadStack(block_kind=dlo.BLOCK_BYTES, n_blocks=n, bytes_block=size, staging=staging)
        sums = []
        for i in range(n):
            v = st.host.view(i)
            v[:] = synth.staging_bytes(size, seed=10 + i)
            sums.append(int(v.view(np.uint64).sum(dtype=np.uint64)))
        st.attach()
        st.set_graphs(True)
        got = torch.zeros(n, dtype=torch.int64, device="cuda")
        for _ in range(4):
            got.zero_()
            st.forward_bytes(got)
            torch.cuda.synchronize()
            assert [int(s) % (1 << 64) for s in got.cpu().numpy().view(np.uint64)] == sums
        st.wait()
        assert st.stats()["graph_launches"] == 3
        for s in (0, 1):
            assert st.verify_slot(s)
        st.close()


_WIDEN_GRAPHS = """
import sys, numpy as np, torch
from tests import helpers as H
from tests.test_gpu_stack import SMALL_VID_FP8 as cfg

def steps(graphs, k, n=4):
    st = H.make_stack(cfg)
    st.attach()
    if k:
        st.set_resident(k)
    st.set_graphs(graphs)
    x, c, t = H.device_inputs(cfg)
    out = torch.empty_like(x)
    outs = []
    for s in range(n):
        st.forward(x, c, t, out=out)
        torch.cuda.synchronize()
        outs.append(out.clone())
        x.copy_(out)
    st.wait()
    stats = st.stats()
    st.close()
    return outs, stats

direct, _ = steps(False, 0)
graph, sg = steps(True, 0)
resident, _ = steps(True, 2)
assert sg["graph_launches"] >= 2, sg["graph_launches"]
for s in range(len(direct)):
    assert torch.equal(direct[s], graph[s]), ("graph", s)
    assert torch.equal(direct[s], resident[s]), ("resident", s)
print("ok", sg["graph_launches"])
"""


def test_w8a16_widening_inside_the_gemm_in_graphs_and_with_residency():
    """The W8A16 GEMM that widens its codes inside the kernel (a cooperative
    launch of CTA pairs with a grid barrier), forced on the small E4M3 video
    stack: whole-forward CUDA graphs replay it, and two resident leading
    blocks change nothing; four chained steps are bit-identical to direct
    forwards with every block streamed.  In a process of its own (the
    switches are read once)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root, DLO_WIDEN_ROWS="1", DLO_GEMM_PAIR="1", DLO_GEMM_BN="256")
    r = subprocess.run([sys.executable, "-c", _WIDEN_GRAPHS], cwd=root, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    assert r.stdout.split()[-2] == "ok"
