"""DiT block-stack forward in float64 -- oracle (test infrastructure only).

The pages describe the offload orchestration only; they print no block math.
The streamed blocks are "transformer blocks" of diffusion transformers ("CPU
Offloading for Diffusion Models", section "Layerwise (Blockwise)
Offloading": "Compute block-i" in the Execution Flow table; Wan2.2 video
DiTs are the recommended case).  The block definitions below are the plain
standard readings (not on the pages):

DiT adaLN-zero block (`dit_block`):
  m = SiLU(c) W_ada^T + b_ada, chunks (shift_msa, scale_msa, gate_msa,
      shift_mlp, scale_mlp, gate_mlp), each of width D
  h = LN(x) (1 + scale_msa) + shift_msa          LN: no affine, biased variance
  q, k, v = split(h W_qkv^T + b_qkv)              head-major [H, hd] per token
  a = softmax(q k^T / sqrt(hd)) v                 per head, non-causal
  x = x + gate_msa (a W_o^T + b_o)
  h = LN(x) (1 + scale_mlp) + shift_mlp
  x = x + gate_mlp (GELU_tanh(h W_1^T + b_1) W_2^T + b_2)

Video-DiT block (`video_block`):
  m = e + T_mod                                    e [B, 6, D] shared, T_mod per block
  self-attention on LN(x)(1 + scale1) + shift1 with RMSNorm (over D, with a
  gain) on q and on k; x = x + gate1 * o
  cross-attention: q from LN_affine(x), k and v from the text context,
  RMSNorm on q and k; x = x + o (no gate)
  FFN on LN(x)(1 + scale2) + shift2 with GELU_tanh; x = x + gate2 * ffn
Both: eps = 1e-6 for every norm; softmax max-subtracted.

Per-tensor FP8 linears ("Distributed Layerwise Offload", Feature
compatibility table, row "Per-tensor online FP8 linears") use the weight
s * decode(q) of `oracle.fp8`; y = x (s q)^T + b equals s (x q^T) + b.
"""
from __future__ import annotations

import numpy as np

from . import fp8

EPS = 1e-6
KIND_DIT = 0
KIND_VIDEO = 1

MOD_CHUNKS = ("shift_msa", "scale_msa", "gate_msa", "shift_mlp", "scale_mlp", "gate_mlp")


# ---------------------------------------------------------------- primitives

def layernorm(x, eps=EPS):
    """(x - mean) / sqrt(var + eps) over the last axis; biased variance, no affine."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def rmsnorm(x, w, eps=EPS):
    """x / sqrt(mean(x^2) + eps) * w over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * w


def gelu_tanh(x):
    """0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def silu(x):
    return x / (1.0 + np.exp(-x))


def linear(x, w, b):
    """y = x w^T + b; w is [out, in]."""
    return x @ w.T + b


def attention(q, k, v, heads):
    """Multi-head softmax attention of one batch element.

    q [Nq, H*hd], k and v [Nk, H*hd]; head h uses columns h*hd .. h*hd+hd-1.
    Returns [Nq, H*hd].
    """
    nq, d = q.shape
    hd = d // heads
    o = np.empty((nq, d), dtype=np.float64)
    # one head at a time: the scores of one head are [Nq, Nk]
    for h in range(heads):
        c = slice(h * hd, (h + 1) * hd)
        s = q[:, c] @ k[:, c].T / np.sqrt(hd)
        s = s - s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=-1, keepdims=True)
        o[:, c] = p @ v[:, c]
    return o


# ---------------------------------------------------------------- parameters

_LINEARS_VIDEO = ("self_attn.q", "self_attn.k", "self_attn.v", "self_attn.o",
                  "cross_attn.q", "cross_attn.k", "cross_attn.v", "cross_attn.o",
                  "ffn.fc1", "ffn.fc2")
_LINEARS_DIT = ("adaLN", "attn.qkv", "attn.proj", "mlp.fc1", "mlp.fc2")


def prepare_block(params, fp8_linears=False, fp8_activations=False):
    """float64 copies of one block's tensors.

    With fp8_linears every linear weight W is replaced by s * decode(q) where
    (q, s) = quantize_per_tensor(W); the codes and scales are also returned
    under "<name>.codes" / "<name>.scale" for byte-level comparisons.
    With fp8_activations as well (W8A8, video blocks), every linear's input is
    quantised the same way, per tensor, when the block runs (`_linear`).
    """
    if fp8_activations and not fp8_linears:
        raise ValueError("W8A8 quantises the weights too")
    out = {k: np.asarray(v, dtype=np.float64) for k, v in params.items()}
    if fp8_activations:
        out["act_e4m3"] = True
    if fp8_linears:
        names = _LINEARS_VIDEO if "modulation" in params else _LINEARS_DIT
        for n in names:
            q, s = fp8.quantize_per_tensor(params[n + ".weight"])
            out[n + ".codes"] = q
            out[n + ".scale"] = s
            out[n + ".weight"] = fp8.dequantize(q, s)
    return out


# ---------------------------------------------------------------- blocks

def dit_block(x, c, P, heads, eps=EPS, rows=None):
    """DiT adaLN-zero block.  x [B, N, D], c [B, C].

    rows: optional token indices; when given, keys/values use every token but
    only those query rows are computed and returned ([B, len(rows), D]).
    """
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    B, N, D = x.shape
    m = linear(silu(c), P["adaLN.weight"], P["adaLN.bias"])            # [B, 6D]
    shift_msa, scale_msa, gate_msa, shift_mlp, scale_mlp, gate_mlp = np.split(m, 6, axis=-1)
    sel = np.arange(N) if rows is None else np.asarray(rows)
    out = np.empty((B, len(sel), D))
    for b in range(B):
        h = layernorm(x[b], eps) * (1.0 + scale_msa[b]) + shift_msa[b]
        wq, wk, wv = np.split(P["attn.qkv.weight"], 3, axis=0)
        bq, bk, bv = np.split(P["attn.qkv.bias"], 3)
        q = linear(h[sel], wq, bq)
        k = linear(h, wk, bk)
        v = linear(h, wv, bv)
        a = attention(q, k, v, heads)
        xb = x[b, sel] + gate_msa[b] * linear(a, P["attn.proj.weight"], P["attn.proj.bias"])
        h2 = layernorm(xb, eps) * (1.0 + scale_mlp[b]) + shift_mlp[b]
        f = gelu_tanh(linear(h2, P["mlp.fc1.weight"], P["mlp.fc1.bias"]))
        out[b] = xb + gate_mlp[b] * linear(f, P["mlp.fc2.weight"], P["mlp.fc2.bias"])
    return out


def _linear(P, name, x, rows=None):
    """x w^T + b of the named linear on a whole activation x [B, M, K]
    (rows: keep only those rows of the result, [B, len(rows), out]).

    W8A8 (P["act_e4m3"]): the input is first replaced by s_x * decode(q_x),
    (q_x, s_x) = fp8.quantize_activation(x) over the WHOLE tensor, all batch
    elements and rows, in float32 -- one dynamic scale per linear input, as
    the weights have one per tensor ("Distributed Layerwise Offload", Feature
    compatibility, row "Per-tensor online FP8 linears", extended to the
    inputs).  Then y = s_x s_w (q_x q_w^T) + b up to float64 rounding.
    """
    if P.get("act_e4m3"):
        q, s = fp8.quantize_activation(x)
        x = fp8.dequantize(q, s)
    if rows is not None:
        x = x[:, rows]
    return linear(x, P[name + ".weight"], P[name + ".bias"])


def video_block(x, e, ctx, P, heads, eps=EPS, rows=None):
    """Video-DiT block.  x [B, N, D], e [B, 6, D], ctx [B, L, Dt].

    rows: as in `dit_block` (not with W8A8: the output projection's input
    scale needs every row of the attention output).
    """
    x = np.asarray(x, dtype=np.float64)
    e = np.asarray(e, dtype=np.float64)
    ctx = np.asarray(ctx, dtype=np.float64)
    B, N, D = x.shape
    if rows is not None and P.get("act_e4m3"):
        raise ValueError("W8A8 blocks are computed for all rows")
    m = e + P["modulation"][None]                                        # [B, 6, D]
    shift1, scale1, gate1, shift2, scale2, gate2 = (m[:, i][:, None, :] for i in range(6))
    sel = np.arange(N) if rows is None else np.asarray(rows)
    h = layernorm(x, eps) * (1.0 + scale1) + shift1
    q = rmsnorm(_linear(P, "self_attn.q", h, sel), P["self_attn.norm_q.weight"], eps)
    k = rmsnorm(_linear(P, "self_attn.k", h), P["self_attn.norm_k.weight"], eps)
    v = _linear(P, "self_attn.v", h)
    a = np.stack([attention(q[b], k[b], v[b], heads) for b in range(B)])
    xb = x[:, sel] + gate1 * _linear(P, "self_attn.o", a)
    hc = layernorm(xb, eps) * P["norm_cross.weight"] + P["norm_cross.bias"]
    qc = rmsnorm(_linear(P, "cross_attn.q", hc), P["cross_attn.norm_q.weight"], eps)
    kc = rmsnorm(_linear(P, "cross_attn.k", ctx), P["cross_attn.norm_k.weight"], eps)
    vc = _linear(P, "cross_attn.v", ctx)
    ac = np.stack([attention(qc[b], kc[b], vc[b], heads) for b in range(B)])
    xb = xb + _linear(P, "cross_attn.o", ac)
    h2 = layernorm(xb, eps) * (1.0 + scale2) + shift2
    f = gelu_tanh(_linear(P, "ffn.fc1", h2))
    return xb + gate2 * _linear(P, "ffn.fc2", f)


def block_forward(kind, x, cond, ctx, P, heads, eps=EPS, rows=None):
    if kind == KIND_DIT:
        return dit_block(x, cond, P, heads, eps, rows)
    return video_block(x, cond, ctx, P, heads, eps, rows)


def stack_forward(kind, x, cond, ctx, blocks, heads, eps=EPS):
    """Blocks 0..n-1 in order; blocks is a list of prepared parameter dicts."""
    for P in blocks:
        x = block_forward(kind, x, cond, ctx, P, heads, eps)
    return x


def multi_stack_forward(parts, x, ctx, eps=EPS):
    """A stack of several ordered block containers ("CPU Offloading for
    Diffusion Models", Layerwise (Blockwise) Offloading: a model may list more
    than one attribute holding transformer blocks, offloaded as one ordered
    sequence).  parts = [(kind, cond, blocks, heads), ...]: the containers run
    in order on the one hidden state; ctx feeds every video container."""
    for kind, cond, blocks, heads in parts:
        x = stack_forward(kind, x, cond, ctx if kind == KIND_VIDEO else None, blocks, heads, eps)
    return x


def max_rel_l2(y, ref):
    """max over batch b of ||y_b - ref_b||_2 / ||ref_b||_2 over all other axes."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    B = ref.shape[0]
    d = (y - ref).reshape(B, -1)
    r = ref.reshape(B, -1)
    return float(np.max(np.linalg.norm(d, axis=1) / np.linalg.norm(r, axis=1)))
