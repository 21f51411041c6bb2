"""Pins for oracle.dit (block math in float64).

The pages print no block math; each function is pinned to torch library
routines (a different implementation of the same standard definition), to
closed forms and to invariants.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle import dit, fp8

torch.set_default_dtype(torch.float64)


def T(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def test_layernorm_vs_torch():
    x = np.random.default_rng(0).standard_normal((7, 96)) * 3 + 1
    ref = F.layer_norm(T(x), (96,), eps=1e-6).numpy()
    np.testing.assert_allclose(dit.layernorm(x), ref, rtol=1e-12, atol=1e-12)
    y = dit.layernorm(x)
    np.testing.assert_allclose(y.mean(-1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(-1), 1, atol=1e-5)   # eps shifts it by ~1e-6


def test_rmsnorm_vs_torch():
    g = np.random.default_rng(1)
    x = g.standard_normal((5, 64))
    w = 1 + 0.1 * g.standard_normal(64)
    ref = F.rms_norm(T(x), (64,), weight=T(w), eps=1e-6).numpy()
    np.testing.assert_allclose(dit.rmsnorm(x, w), ref, rtol=1e-12, atol=1e-12)


def test_activations_vs_torch():
    x = np.linspace(-8, 8, 1001)
    np.testing.assert_allclose(dit.gelu_tanh(x), F.gelu(T(x), approximate="tanh").numpy(),
                               rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dit.silu(x), F.silu(T(x)).numpy(), rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("nq,nk,heads,hd", [(9, 9, 2, 8), (5, 13, 3, 72), (16, 7, 1, 16)])
def test_attention_vs_torch_sdpa(nq, nk, heads, hd):
    g = np.random.default_rng(nq * 31 + nk)
    q = g.standard_normal((nq, heads * hd))
    k = g.standard_normal((nk, heads * hd))
    v = g.standard_normal((nk, heads * hd))
    th = lambda a, n: T(a).reshape(n, heads, hd).transpose(0, 1)
    ref = F.scaled_dot_product_attention(th(q, nq), th(k, nk), th(v, nk))
    ref = ref.transpose(0, 1).reshape(nq, heads * hd).numpy()
    np.testing.assert_allclose(dit.attention(q, k, v, heads), ref, rtol=1e-12, atol=1e-12)


def test_attention_equal_keys_is_mean_of_v():
    g = np.random.default_rng(3)
    k = np.tile(g.standard_normal((1, 32)), (11, 1))
    v = g.standard_normal((11, 32))
    q = g.standard_normal((4, 32))
    out = dit.attention(q, k, v, heads=4)
    np.testing.assert_allclose(out, np.tile(v.mean(0), (4, 1)), rtol=1e-12, atol=1e-12)


def _tiny(kind, **kw):
    if kind == synth.KIND_DIT:
        base = synth.StackConfig("t", kind, 2, 32, 2, 16, 64, 2, 10, cond_dim=24, **kw)
    else:
        base = synth.StackConfig("t", kind, 2, 32, 2, 16, 64, 2, 10, text_dim=48,
                                 text_tokens=6, **kw)
    return base


def _inputs(cfg):
    x = synth.activations(cfg)
    cond = synth.condition(cfg) if cfg.kind == synth.KIND_VIDEO else \
        np.random.default_rng(9).standard_normal((cfg.batch, cfg.cond_dim))
    ctx = synth.text_context(cfg) if cfg.kind == synth.KIND_VIDEO else None
    return x, cond, ctx


def _big_weights(P, scale=10.0):
    """Larger weights so every term of the block visibly moves the output."""
    return {k: (v * scale if k.endswith("weight") and "norm" not in k else v)
            for k, v in P.items()}


def test_dit_block_vs_torch_modules():
    cfg = _tiny(synth.KIND_DIT)
    P = _big_weights(dit.prepare_block(synth.block_params(cfg, 0)))
    x, c, _ = _inputs(cfg)
    D, H = cfg.hidden, cfg.heads
    ln = torch.nn.LayerNorm(D, eps=1e-6, elementwise_affine=False)
    mha = torch.nn.MultiheadAttention(D, H, batch_first=True)
    with torch.no_grad():
        mha.in_proj_weight.copy_(T(P["attn.qkv.weight"]))
        mha.in_proj_bias.copy_(T(P["attn.qkv.bias"]))
        mha.out_proj.weight.copy_(T(P["attn.proj.weight"]))
        mha.out_proj.bias.copy_(T(P["attn.proj.bias"]))
        ada = torch.nn.Sequential(torch.nn.SiLU(), torch.nn.Linear(cfg.cond_dim, 6 * D))
        ada[1].weight.copy_(T(P["adaLN.weight"]))
        ada[1].bias.copy_(T(P["adaLN.bias"]))
        mlp = torch.nn.Sequential(torch.nn.Linear(D, cfg.ffn), torch.nn.GELU(approximate="tanh"),
                                  torch.nn.Linear(cfg.ffn, D))
        mlp[0].weight.copy_(T(P["mlp.fc1.weight"]))
        mlp[0].bias.copy_(T(P["mlp.fc1.bias"]))
        mlp[2].weight.copy_(T(P["mlp.fc2.weight"]))
        mlp[2].bias.copy_(T(P["mlp.fc2.bias"]))
        xt, ct = T(x), T(c)
        sh1, sc1, g1, sh2, sc2, g2 = ada(ct).unsqueeze(1).chunk(6, dim=-1)
        h = ln(xt) * (1 + sc1) + sh1
        xt = xt + g1 * mha(h, h, h, need_weights=False)[0]
        h = ln(xt) * (1 + sc2) + sh2
        ref = (xt + g2 * mlp(h)).numpy()
    out = dit.dit_block(x, c, P, H)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-10)
    # the check is not vacuous: the block moves x by O(1)
    assert np.abs(out - x).mean() > 0.1


def test_video_block_vs_torch_primitives():
    cfg = _tiny(synth.KIND_VIDEO)
    P = _big_weights(dit.prepare_block(synth.block_params(cfg, 1)))
    x, e, ctx = _inputs(cfg)
    H, hd = cfg.heads, cfg.head_dim
    t = {k: T(v) for k, v in P.items()}

    def mha(q, k, v):
        sp = lambda a: a.reshape(a.shape[0], a.shape[1], H, hd).transpose(1, 2)
        o = F.scaled_dot_product_attention(sp(q), sp(k), sp(v))
        return o.transpose(1, 2).reshape(q.shape)

    D = cfg.hidden
    xt, et, ct = T(x), T(e), T(ctx)
    m = (et + t["modulation"][None]).unsqueeze(2)   # [B, 6, 1, D]
    ln = lambda a: F.layer_norm(a, (D,), eps=1e-6)
    rms = lambda a, w: F.rms_norm(a, (D,), weight=w, eps=1e-6)
    lin = lambda a, n: F.linear(a, t[n + ".weight"], t[n + ".bias"])
    h = ln(xt) * (1 + m[:, 1]) + m[:, 0]
    q = rms(lin(h, "self_attn.q"), t["self_attn.norm_q.weight"])
    k = rms(lin(h, "self_attn.k"), t["self_attn.norm_k.weight"])
    xt = xt + m[:, 2] * lin(mha(q, k, lin(h, "self_attn.v")), "self_attn.o")
    hc = F.layer_norm(xt, (D,), t["norm_cross.weight"], t["norm_cross.bias"], eps=1e-6)
    q = rms(lin(hc, "cross_attn.q"), t["cross_attn.norm_q.weight"])
    k = rms(lin(ct, "cross_attn.k"), t["cross_attn.norm_k.weight"])
    xt = xt + lin(mha(q, k, lin(ct, "cross_attn.v")), "cross_attn.o")
    h = ln(xt) * (1 + m[:, 4]) + m[:, 3]
    ref = (xt + m[:, 5] * lin(F.gelu(lin(h, "ffn.fc1"), approximate="tanh"), "ffn.fc2")).numpy()
    out = dit.video_block(x, e, ctx, P, H)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-10)
    assert np.abs(out - x).mean() > 0.1


def test_zero_gates_give_identity():
    cfg = _tiny(synth.KIND_DIT)
    P = dit.prepare_block(synth.block_params(cfg, 0))
    D = cfg.hidden
    for chunk in (2, 5):                       # gate_msa, gate_mlp
        P["adaLN.weight"][chunk * D:(chunk + 1) * D] = 0
        P["adaLN.bias"][chunk * D:(chunk + 1) * D] = 0
    x, c, _ = _inputs(cfg)
    np.testing.assert_array_equal(dit.dit_block(x, c, P, cfg.heads), x)

    cfgv = _tiny(synth.KIND_VIDEO)
    Pv = dit.prepare_block(synth.block_params(cfgv, 0))
    Pv["modulation"][[2, 5]] = 0
    Pv["cross_attn.o.weight"][:] = 0
    Pv["cross_attn.o.bias"][:] = 0
    x, e, ctx = _inputs(cfgv)
    e = e.copy()
    e[:, [2, 5]] = 0
    np.testing.assert_array_equal(dit.video_block(x, e, ctx, Pv, cfgv.heads), x)


@pytest.mark.parametrize("kind", [synth.KIND_DIT, synth.KIND_VIDEO])
def test_token_permutation_and_batch_independence(kind):
    cfg = _tiny(kind)
    P = _big_weights(dit.prepare_block(synth.block_params(cfg, 0)))
    x, cond, ctx = _inputs(cfg)
    out = dit.block_forward(kind, x, cond, ctx, P, cfg.heads)
    perm = np.random.default_rng(5).permutation(cfg.tokens)
    outp = dit.block_forward(kind, x[:, perm], cond, ctx, P, cfg.heads)
    np.testing.assert_allclose(outp, out[:, perm], rtol=1e-11, atol=1e-11)
    x2 = x.copy()
    x2[1] += 1.0
    out2 = dit.block_forward(kind, x2, cond, ctx, P, cfg.heads)
    np.testing.assert_array_equal(out2[0], out[0])
    assert not np.allclose(out2[1], out[1])


@pytest.mark.parametrize("kind", [synth.KIND_DIT, synth.KIND_VIDEO])
def test_rows_subset_matches_full(kind):
    cfg = _tiny(kind)
    P = dit.prepare_block(synth.block_params(cfg, 0))
    x, cond, ctx = _inputs(cfg)
    full = dit.block_forward(kind, x, cond, ctx, P, cfg.heads)
    rows = [0, 3, 9]
    sub = dit.block_forward(kind, x, cond, ctx, P, cfg.heads, rows=rows)
    np.testing.assert_allclose(sub, full[:, rows], rtol=1e-12, atol=1e-12)


def test_fp8_prepare_uses_decoded_weights():
    cfg = _tiny(synth.KIND_VIDEO, wdtype=synth.W_E4M3, master_fp32=True)
    raw = synth.block_params(cfg, 0)
    P = dit.prepare_block(raw, fp8_linears=True)
    q, s = fp8.quantize_per_tensor(raw["ffn.fc1.weight"])
    np.testing.assert_array_equal(P["ffn.fc1.codes"], q)
    np.testing.assert_array_equal(P["ffn.fc1.weight"], fp8.decode_e4m3(q) * np.float64(s))
    # non-linear tensors are bf16-exact in an FP8 stack
    b = raw["ffn.fc1.bias"]
    np.testing.assert_array_equal(synth.round_bf16(b), b)


def test_max_rel_l2():
    ref = np.ones((2, 3, 4))
    y = ref.copy()
    y[1] *= 1.1
    assert abs(dit.max_rel_l2(y, ref) - 0.1) < 1e-12
    assert dit.max_rel_l2(ref, ref) == 0.0


def _multi_parts(mc, step=0):
    parts = []
    for p in mc.parts:
        blocks = [dit.prepare_block(synth.block_params(p, j), fp8_linears=p.wdtype == synth.W_E4M3)
                  for j in range(p.n_blocks)]
        parts.append((p.kind, synth.condition(p, step).astype(np.float64), blocks, p.heads))
    x = synth.activations(mc.parts[0], step).astype(np.float64)
    v = mc.video
    ctx = synth.text_context(v, step).astype(np.float64) if v else None
    return parts, x, ctx


def test_multi_stack_split_of_one_container_is_the_same_stack():
    # one DiT container of 3 blocks == containers of 1 + 2 of the same blocks
    mc = synth.MULTI_TINY
    parts, x, ctx = _multi_parts(mc)
    kind, c, blocks, heads = parts[1]
    whole = dit.stack_forward(kind, x, c, None, blocks, heads)
    split = dit.multi_stack_forward([(kind, c, blocks[:1], heads), (kind, c, blocks[1:], heads)], x, ctx)
    np.testing.assert_array_equal(split, whole)


def test_multi_stack_identity_container_and_order():
    # a trailing DiT container whose gates are all zero leaves the video
    # container's output unchanged; swapping the order of two non-identity
    # containers changes the result (they do not commute)
    mc = synth.MULTI_TINY
    parts, x, ctx = _multi_parts(mc)
    kv, e, bv, hv = parts[0]
    kd, c, bd, hd = parts[1]
    D = mc.hidden
    ident = []
    for P in bd:
        Q = dict(P)
        Q["adaLN.weight"] = P["adaLN.weight"].copy()
        Q["adaLN.bias"] = P["adaLN.bias"].copy()
        for chunk in (2, 5):
            Q["adaLN.weight"][chunk * D:(chunk + 1) * D] = 0
            Q["adaLN.bias"][chunk * D:(chunk + 1) * D] = 0
        ident.append(Q)
    video_only = dit.stack_forward(kv, x, e, ctx, bv, hv)
    np.testing.assert_array_equal(dit.multi_stack_forward([parts[0], (kd, c, ident, hd)], x, ctx),
                                  video_only)
    fwd = dit.multi_stack_forward(parts, x, ctx)
    rev = dit.multi_stack_forward([parts[1], parts[0]], x, ctx)
    assert dit.max_rel_l2(rev, fwd) > 1e-7
    # each container sees its own conditioning: feeding the DiT container a
    # different c changes only what follows it
    c2 = c + 0.5
    other = dit.multi_stack_forward([parts[0], (kd, c2, bd, hd)], x, ctx)
    assert dit.max_rel_l2(other, fwd) > 1e-7


# ---------------------------------------------------------------- W8A8 linears

def _w8a8_linear_params(out_f=24, in_f=40, seed=3):
    g = np.random.default_rng(seed)
    w = g.standard_normal((out_f, in_f)).astype(np.float32) * 0.05
    b = g.standard_normal(out_f).astype(np.float32) * 0.01
    q, s = fp8.quantize_per_tensor(w)
    P = {"l.weight": fp8.dequantize(q, s), "l.bias": b.astype(np.float64), "act_e4m3": True}
    return P


def test_w8a8_linear_is_exact_on_representable_inputs():
    # x = 2^-3 * decode(codes) with a code of magnitude 448 present: the
    # per-tensor scale is exactly 2^-3 and the codes come back unchanged, so
    # the W8A8 product equals the product with the unquantised input
    P = _w8a8_linear_params()
    g = np.random.default_rng(0)
    codes = g.integers(0, 0x7F, size=(2, 7, 40)).astype(np.uint8)
    codes[0, 0, 0] = 0x7E                                   # 448
    codes |= (g.integers(0, 2, size=codes.shape) << 7).astype(np.uint8)
    x = fp8.decode_e4m3(codes) * 2.0 ** -3
    q, s = fp8.quantize_activation(x)
    assert s == np.float32(2.0 ** -3)
    np.testing.assert_array_equal(q, codes)
    y = dit._linear(P, "l", x)
    np.testing.assert_array_equal(y, dit.linear(x, P["l.weight"], P["l.bias"]))


def test_w8a8_linear_scale_invariance_and_error_bound():
    P = _w8a8_linear_params()
    P0 = dict(P, **{"l.bias": np.zeros_like(P["l.bias"])})
    g = np.random.default_rng(1)
    x = g.standard_normal((2, 9, 40)) * np.array([1.0, 3.0])[:, None, None]
    y = dit._linear(P0, "l", x)
    # powers of two move the scale, not the codes
    np.testing.assert_array_equal(dit._linear(P0, "l", x * 8.0), y * 8.0)
    # error against the exact input: at most half a quantum per element,
    # relative 2^-4 in the normal range, 2^-10 s among the subnormals
    x32 = x.astype(np.float32).astype(np.float64)
    _, s = fp8.quantize_activation(x)
    per = np.maximum(np.abs(x32) * 2.0 ** -4, float(s) * 2.0 ** -10) + np.abs(x32) * 2.0 ** -21
    bound = per @ np.abs(P0["l.weight"]).T
    ref = dit.linear(x32, P0["l.weight"], P0["l.bias"])
    assert np.all(np.abs(y - ref) <= bound * (1 + 1e-9))
    assert np.abs(y - ref).max() > 0                        # it does quantise


def test_w8a8_scale_spans_the_whole_tensor():
    # one scale for all batch elements and rows: enlarging batch element 1
    # changes the codes, hence the result, of batch element 0
    P = _w8a8_linear_params()
    g = np.random.default_rng(2)
    x = g.standard_normal((2, 9, 40))
    y = dit._linear(P, "l", x)
    x2 = x.copy()
    x2[1] *= 5.0
    y2 = dit._linear(P, "l", x2)
    assert not np.array_equal(y2[0], y[0])
    # ... while the W8A16 linear keeps batch elements independent
    Pw = {k: v for k, v in P.items() if k != "act_e4m3"}
    np.testing.assert_array_equal(dit._linear(Pw, "l", x2)[0], dit._linear(Pw, "l", x)[0])
    # rows are taken after quantising the whole tensor
    rows = [0, 4, 8]
    np.testing.assert_array_equal(dit._linear(P, "l", x, rows), y[:, rows])


def test_w8a8_video_block_near_w8a16():
    cfg = _tiny(synth.KIND_VIDEO)
    prm = synth.block_params(cfg, 0)
    P16 = dit.prepare_block(prm, fp8_linears=True)
    P8 = dit.prepare_block(prm, fp8_linears=True, fp8_activations=True)
    x, e, ctx = _inputs(cfg)
    y16 = dit.video_block(x, e, ctx, P16, cfg.heads)
    y8 = dit.video_block(x, e, ctx, P8, cfg.heads)
    d = dit.max_rel_l2(y8 - x, y16 - x)        # the block's update, not the residual
    assert 1e-4 < d < 0.1
    with pytest.raises(ValueError):
        dit.video_block(x, e, ctx, P8, cfg.heads, rows=[0, 1])
