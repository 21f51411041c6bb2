"""Host-side checks of libdlo.so that need no GPU: exported symbols, the flat
block layout, bf16 packing and the E4M3 quantiser (bit-exact against the
oracle's independent quantiser)."""
import os
import re

import numpy as np
import pytest
import torch

import synth
from oracle import fp8 as ofp8

dlo = pytest.importorskip("layerwise_weight_offload_slot_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "dlo.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dlo_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) >= 20
    for n in names:
        assert hasattr(dlo._lib, n), n
        assert n in dlo.EXPORTED, n


def desc_of(cfg, **kw):
    return dlo.make_desc(block_kind=cfg.kind, n_blocks=cfg.n_blocks, hidden=cfg.hidden,
                         heads=cfg.heads, head_dim=cfg.head_dim, ffn=cfg.ffn,
                         cond_dim=cfg.cond_dim, text_dim=cfg.text_dim, max_batch=cfg.batch,
                         max_tokens=cfg.tokens, max_text_tokens=cfg.text_tokens,
                         wdtype=cfg.wdtype, **kw)


@pytest.mark.parametrize("cfg", list(synth.CONFIGS.values()), ids=lambda c: c.name)
def test_layout_matches_param_specs(cfg):
    d = desc_of(cfg)
    lay = dlo.dlo_block_layout(d)
    bb = dlo.dlo_block_bytes(d)
    assert bb % 256 == 0
    specs = {n: s for n, s, _ in synth.param_specs(cfg)}
    src = [e for e in lay if e["source"]]
    assert {e["name"] for e in src} == set(specs)
    for e in src:
        assert tuple(e["shape"]) == tuple(specs[e["name"]])
    # non-overlapping, in bounds, 16-byte aligned, bytes = elements * size
    end = 0
    for e in lay:
        assert e["offset"] >= end and e["offset"] % 16 == 0
        n = int(np.prod(e["shape"]))
        size = {dlo.DT_BF16: 2, dlo.DT_E4M3: 1, dlo.DT_F32: 4}[e["dtype"]]
        assert e["bytes"] == n * size
        end = e["offset"] + e["bytes"]
    assert end <= bb
    # fused q|k|v weights and biases are contiguous
    by = {e["name"]: e for e in lay}
    for grp in (["attn.qkv.weight"], ["self_attn.q.weight", "self_attn.k.weight", "self_attn.v.weight"],
                ["self_attn.q.bias", "self_attn.k.bias", "self_attn.v.bias"],
                ["cross_attn.k.weight", "cross_attn.v.weight"], ["cross_attn.k.bias", "cross_attn.v.bias"]):
        if all(g in by for g in grp):
            for a, b in zip(grp, grp[1:]):
                assert by[a]["offset"] + by[a]["bytes"] == by[b]["offset"]
    if synth.fp8_weights(cfg.wdtype):
        assert not by["linear_scales"]["source"]
    assert dlo.dlo_workspace_bytes(d) > 0


def test_block_bytes_of_the_workloads():
    # hand arithmetic: parameter count x element size (+ alignment padding)
    dit = desc_of(synth.CFG_DITXL)
    D, F = 1152, 4608
    params = 6 * D * D + 6 * D + 3 * D * D + 3 * D + D * D + D + 2 * F * D + F + D
    assert params * 2 <= dlo.dlo_block_bytes(dit) < params * 2 + 4096
    vid = desc_of(synth.CFG_VIDEO)
    assert abs(dlo.dlo_block_bytes(vid) / 1e6 - 681.8) < 0.2


def test_invalid_descs_are_rejected():
    good = dict(block_kind=0, n_blocks=2, hidden=64, heads=2, head_dim=32, ffn=128, cond_dim=64,
                max_batch=1, max_tokens=16)
    assert dlo.dlo_block_bytes(dlo.make_desc(**good)) > 0
    for bad in (dict(hidden=60), dict(heads=3), dict(n_blocks=0), dict(ffn=100), dict(cond_dim=12),
                dict(head_dim=256, hidden=512, heads=2), dict(max_tokens=0), dict(block_kind=7)):
        assert dlo.dlo_block_bytes(dlo.make_desc(**{**good, **bad})) == 0, bad
    d = dlo.make_desc(**{**good, "wdtype": dlo.W_E4M3})
    with pytest.raises(dlo.DloError) as e:
        dlo.dlo_block_layout(d)
    assert e.value.status == dlo.EUNSUPPORTED


def test_pack_rounds_bf16_like_torch():
    cfg = synth.CFG_TINY.with_(n_blocks=1)
    d = desc_of(cfg)
    P = synth.block_params(cfg, 0)
    P["adaLN.bias"][:4] = [np.inf, -np.inf, 3.0e38, 1e-40]
    bb = dlo.dlo_block_bytes(d)
    flat = np.zeros(bb, dtype=np.uint8)
    dlo.dlo_pack_block(d, P, flat.ctypes.data, bb)
    for e in dlo.dlo_block_layout(d):
        got = flat[e["offset"]:e["offset"] + e["bytes"]].view(np.uint16)
        ref = torch.from_numpy(P[e["name"]].ravel()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(got, ref, err_msg=e["name"])


def test_quantizer_matches_oracle_bit_exactly():
    g = np.random.default_rng(7)
    for w in (g.standard_normal((257, 129)).astype(np.float32) * 0.02,
              g.standard_normal(4096).astype(np.float32) * 3,
              np.concatenate([g.standard_normal(1000) * 1e-4, [0.0, -0.0, 1.0]]).astype(np.float32),
              np.zeros(16, np.float32)):
        q, s = dlo.dlo_quantize_e4m3(w)
        qo, so = ofp8.quantize_per_tensor(w)
        assert np.float32(s) == so
        np.testing.assert_array_equal(q, qo)


def test_pack_fp8_block_matches_oracle():
    cfg = synth.CFG_VIDEO_FP8.with_(n_blocks=1, hidden=64, heads=2, head_dim=32, ffn=128,
                                    text_dim=48, tokens=8, text_tokens=4)
    d = desc_of(cfg)
    P = synth.block_params(cfg, 0)
    bb = dlo.dlo_block_bytes(d)
    flat = np.zeros(bb, dtype=np.uint8)
    dlo.dlo_pack_block(d, P, flat.ctypes.data, bb)
    lay = {e["name"]: e for e in dlo.dlo_block_layout(d)}
    sc = flat[lay["linear_scales"]["offset"]:][:64].view(np.float32)
    names = ["self_attn.q", "self_attn.k", "self_attn.v", "self_attn.o", "cross_attn.q",
             "cross_attn.k", "cross_attn.v", "cross_attn.o", "ffn.fc1", "ffn.fc2"]
    for i, n in enumerate(names):
        e = lay[n + ".weight"]
        assert e["dtype"] == dlo.DT_E4M3
        q, s = ofp8.quantize_per_tensor(P[n + ".weight"])
        np.testing.assert_array_equal(flat[e["offset"]:e["offset"] + e["bytes"]], q.ravel())
        assert sc[i] == s
    e = lay["ffn.fc1.bias"]
    assert e["dtype"] == dlo.DT_BF16


def _multi_descs(mc, **kw):
    return [dlo.make_desc(block_kind=p.kind, n_blocks=p.n_blocks, hidden=p.hidden, heads=p.heads,
                          head_dim=p.head_dim, ffn=p.ffn, cond_dim=p.cond_dim, text_dim=p.text_dim,
                          max_batch=p.batch, max_tokens=p.tokens, max_text_tokens=p.text_tokens,
                          wdtype=p.wdtype, **kw) for p in mc.parts]


@pytest.mark.parametrize("mc", list(synth.MULTI_CONFIGS.values()), ids=lambda c: c.name)
def test_multi_container_workspace_serves_every_container(mc):
    ds = _multi_descs(mc)
    ws = dlo.dlo_workspace_bytes_multi(ds)
    assert ws > 0 and ws % 256 == 0
    for d in ds:
        assert ws >= dlo.dlo_workspace_bytes(d)
    # one container through the multi entry point is the plain workspace
    assert dlo.dlo_workspace_bytes_multi(ds[:1]) == dlo.dlo_workspace_bytes(ds[0])


def test_multi_container_stacks_are_validated():
    mc = synth.MULTI_TINY
    ds = _multi_descs(mc)
    assert dlo.dlo_workspace_bytes_multi(ds) > 0
    assert dlo.dlo_workspace_bytes_multi([]) == 0
    def bad(i, **kw):
        out = list(ds)
        f = {name: getattr(out[i], name) for name, _ in dlo.dlo_desc._fields_}
        f.update(kw)
        out[i] = dlo.dlo_desc(**f)
        return out
    # shared fields must agree
    for kw in (dict(hidden=256, heads=4), dict(max_batch=3), dict(max_tokens=41), dict(eps=1e-5),
               dict(staging=dlo.STAGE_GATHER), dict(register_budget_bytes=1 << 20)):
        assert dlo.dlo_workspace_bytes_multi(bad(1, **kw)) == 0, kw
    # an invalid container invalidates the stack
    assert dlo.dlo_workspace_bytes_multi(bad(1, ffn=100)) == 0
    # video containers share the text fields
    v2 = bad(1, block_kind=dlo.BLOCK_VIDEO, text_dim=128, max_text_tokens=9)
    assert dlo.dlo_workspace_bytes_multi(v2) == 0
    v3 = bad(1, block_kind=dlo.BLOCK_VIDEO, text_dim=64, max_text_tokens=9)
    assert dlo.dlo_workspace_bytes_multi(v3) > 0
    # bytes blocks stand alone
    b = dlo.make_desc(block_kind=dlo.BLOCK_BYTES, n_blocks=2, hidden=0, heads=0, head_dim=0, ffn=0,
                      bytes_block=4096)
    assert dlo.dlo_workspace_bytes_multi([b]) > 0
    assert dlo.dlo_workspace_bytes_multi([b, b]) == 0


def test_multi_container_create_rejects_small_slots_before_touching_the_device():
    mc = synth.MULTI_TINY
    ds = _multi_descs(mc)
    sizes = [dlo.dlo_block_bytes(d) for d in ds]
    assert sizes[0] != sizes[1]
    ws = dlo.dlo_workspace_bytes_multi(ds)
    fake = 1 << 40
    with pytest.raises(dlo.DloError) as e:
        dlo.dlo_create_multi(ds, 0, fake, fake + (1 << 30), min(sizes), fake + (2 << 30), ws,
                             fake + 8, fake + 16)
    assert e.value.status == dlo.ENOMEM and "largest" in str(e.value)
    with pytest.raises(dlo.DloError) as e:
        dlo.dlo_create_multi(ds + [ds[0]] * 64, 0, fake, fake + (1 << 30), max(sizes),
                             fake + (2 << 30), ws, fake + 8, fake + 16)
    assert e.value.status == dlo.EINVAL
