"""Python binding of libdlo.so: layerwise weight offload of a DiT block stack
through two device slots on one GB300 (sm_103a).

The functions below carry the names of the C ABI in include/dlo.h and only
marshal arguments; every step of the offload path runs in the library.  The
library must have been built (`python layerwise_weight_offload_slot_gb300/build.py`,
or `__graft_entry__.build()`); importing this package without it raises
ImportError -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdlo.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python layerwise_weight_offload_slot_gb300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)

ABI_VERSION = 3
K_COUNT = 16
QUANT_SCRATCH = 1024
OK, EINVAL, ESTATE, ENOMEM, ECUDA, EREGISTER, ETIMEDOUT, EUNSUPPORTED, EMISMATCH = \
    0, -1, -2, -3, -4, -5, -6, -7, -8
BLOCK_DIT, BLOCK_VIDEO, BLOCK_BYTES = 0, 1, 2
W_BF16, W_E4M3, W_E4M3_A8 = 0, 1, 2
STAGE_MEMCPY, STAGE_GATHER, STAGE_PER_TENSOR = 0, 1, 2
HOST_PINNED, HOST_REGISTER, HOST_PAGEABLE = 1, 2, 4
DT_BF16, DT_E4M3, DT_F32, DT_U8 = 0, 1, 2, 3
EPI_BIAS, EPI_GELU, EPI_RESIDUAL = 0, 1, 2

STATUS_NAMES = {0: "OK", -1: "EINVAL", -2: "ESTATE", -3: "ENOMEM", -4: "ECUDA",
                -5: "EREGISTER", -6: "ETIMEDOUT", -7: "EUNSUPPORTED", -8: "EMISMATCH"}


class DloError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class dlo_desc(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_int), ("block_kind", ctypes.c_int),
                ("wdtype", ctypes.c_int), ("n_blocks", ctypes.c_int), ("hidden", ctypes.c_int),
                ("heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("cond_dim", ctypes.c_int), ("text_dim", ctypes.c_int),
                ("max_batch", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("max_text_tokens", ctypes.c_int), ("eps", ctypes.c_float),
                ("staging", ctypes.c_int), ("register_budget_bytes", ctypes.c_ulonglong),
                ("bytes_block", ctypes.c_ulonglong)]


class dlo_tensor_info(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 40), ("offset", ctypes.c_ulonglong),
                ("bytes", ctypes.c_ulonglong), ("dtype", ctypes.c_int), ("ndim", ctypes.c_int),
                ("shape", ctypes.c_longlong * 2), ("source", ctypes.c_int)]


class dlo_stats(ctypes.Structure):
    _fields_ = [("forwards", ctypes.c_ulonglong), ("stagings", ctypes.c_ulonglong),
                ("staged_bytes", ctypes.c_ulonglong), ("streamed_execs", ctypes.c_ulonglong),
                ("kernel_launches", ctypes.c_ulonglong), ("resident", ctypes.c_int),
                ("slot_block", ctypes.c_int * 2), ("registered_ranges", ctypes.c_int),
                ("registered_read_only", ctypes.c_int), ("device_error", ctypes.c_int),
                ("timed_execs", ctypes.c_int), ("copy_ms", ctypes.c_double),
                ("compute_ms", ctypes.c_double), ("exposed_wait_ms", ctypes.c_double),
                ("kclass_ms", ctypes.c_double * K_COUNT), ("kclass_flops", ctypes.c_double * K_COUNT),
                ("kclass_bytes", ctypes.c_double * K_COUNT),
                ("kclass_launches", ctypes.c_ulonglong * K_COUNT),
                ("h2d_copies", ctypes.c_ulonglong), ("graph_captures", ctypes.c_ulonglong),
                ("graph_launches", ctypes.c_ulonglong)]

    def as_dict(self) -> dict:
        d = {}
        for name, _ in self._fields_:
            v = getattr(self, name)
            d[name] = list(v) if isinstance(v, ctypes.Array) else v
        return d


KCLASS_NAMES = ("gemm_bf16", "gemm_e4m3", "attention", "layernorm", "rmsnorm", "modulation",
                "convert", "gather", "gemm_fp8", "quant")


_vp, _sz, _int, _uint, _f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint, ctypes.c_float
_P = ctypes.POINTER


def _decl(name, restype, *argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)
    return f


_c = {
    "dlo_block_bytes": _decl("dlo_block_bytes", _sz, _P(dlo_desc)),
    "dlo_block_layout": _decl("dlo_block_layout", _int, _P(dlo_desc), _P(dlo_tensor_info), _int, _P(_int)),
    "dlo_workspace_bytes": _decl("dlo_workspace_bytes", _sz, _P(dlo_desc)),
    "dlo_workspace_bytes_multi": _decl("dlo_workspace_bytes_multi", _sz, _P(dlo_desc), _int),
    "dlo_pack_block": _decl("dlo_pack_block", _int, _P(dlo_desc), _P(_vp), _int, _vp, _sz),
    "dlo_quantize_e4m3": _decl("dlo_quantize_e4m3", _int, _vp, _sz, _vp, _P(_f32)),
    "dlo_create": _decl("dlo_create", _int, _P(dlo_desc), _int, _vp, _vp, _sz, _vp, _sz, _vp, _vp, _P(_vp)),
    "dlo_create_multi": _decl("dlo_create_multi", _int, _P(dlo_desc), _int, _int, _vp, _vp, _sz, _vp, _sz,
                              _vp, _vp, _P(_vp)),
    "dlo_register_host_blocks": _decl("dlo_register_host_blocks", _int, _vp, _int, _P(_vp), _sz, _uint),
    "dlo_set_resident": _decl("dlo_set_resident", _int, _vp, _int, _P(_vp)),
    "dlo_forward": _decl("dlo_forward", _int, _vp, _vp, _vp, _vp, _int, _int, _int, _vp),
    "dlo_forward_multi": _decl("dlo_forward_multi", _int, _vp, _vp, _P(_vp), _vp, _int, _int, _int, _vp),
    "dlo_forward_host": _decl("dlo_forward_host", _int, _vp, _vp, _vp, _vp, _int, _int, _int, _vp, _int),
    "dlo_wait": _decl("dlo_wait", _int, _vp, _int),
    "dlo_destroy": _decl("dlo_destroy", _int, _vp),
    "dlo_last_error": _decl("dlo_last_error", ctypes.c_char_p, _vp),
    "dlo_get_stats": _decl("dlo_get_stats", _int, _vp, _P(dlo_stats)),
    "dlo_get_log": _decl("dlo_get_log", _int, _vp, _P(_int), _P(_int), _P(_int), _int, _P(_int)),
    "dlo_reset_log": _decl("dlo_reset_log", _int, _vp),
    "dlo_set_timing": _decl("dlo_set_timing", _int, _vp, _int),
    "dlo_set_graphs": _decl("dlo_set_graphs", _int, _vp, _int),
    "dlo_verify_slot": _decl("dlo_verify_slot", _int, _vp, _int, _int),
    "dlo_debug_fail_register": _decl("dlo_debug_fail_register", None, _int),
    "dlo_op_gemm": _decl("dlo_op_gemm", _int, _vp, _vp, _int, _vp, _int, _vp, _int, _int, _int, _int,
                         _vp, _int, _vp, _int, _int, _vp, _vp),
    "dlo_op_gemm_noalloc": _decl("dlo_op_gemm_noalloc", _int, _vp, _vp, _int, _vp, _int, _vp, _int, _int,
                                 _int, _int, _vp, _int, _vp, _int, _int, _vp),
    "dlo_op_wait_selftest": _decl("dlo_op_wait_selftest", _int, _vp, _vp),
    "dlo_debug_device_timeout": _decl("dlo_debug_device_timeout", _int, _vp),
    "dlo_op_quantize_act": _decl("dlo_op_quantize_act", _int, _vp, _int, _int, _int, _vp, _vp, _vp, _vp),
    "dlo_op_gemm_w8a8": _decl("dlo_op_gemm_w8a8", _int, _vp, _vp, _vp, _vp, _int, _vp, _int, _int, _int,
                              _int, _vp, _int, _vp, _int, _int, _vp, _vp),
    "dlo_op_attention": _decl("dlo_op_attention", _int, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int,
                              _int, _int, _int, _int, _vp),
    "dlo_op_layernorm": _decl("dlo_op_layernorm", _int, _vp, _int, _int, _int, _vp, _vp, _int, _vp, _vp,
                              _f32, _vp, _vp),
    "dlo_op_rmsnorm": _decl("dlo_op_rmsnorm", _int, _vp, _int, _int, _int, _int, _vp, _f32, _vp),
    "dlo_op_adaln": _decl("dlo_op_adaln", _int, _vp, _int, _int, _vp, _vp, _int, _vp, _vp),
    "dlo_op_stage": _decl("dlo_op_stage", _int, _vp, _vp, _sz, _int, _vp),
}

EXPORTED = tuple(_c)


def _err(ctx) -> str:
    m = _c["dlo_last_error"](ctx)
    return m.decode() if m else ""


def _check(st: int, ctx=None):
    if st != OK:
        raise DloError(st, _err(ctx))


# ------------------------------------------------------------------ layout

def make_desc(*, block_kind, n_blocks, hidden, heads, head_dim, ffn, cond_dim=0, text_dim=0,
              max_batch=1, max_tokens=1, max_text_tokens=0, wdtype=W_BF16, eps=1e-6,
              staging=STAGE_MEMCPY, register_budget_bytes=0, bytes_block=0) -> dlo_desc:
    return dlo_desc(ABI_VERSION, block_kind, wdtype, n_blocks, hidden, heads, head_dim, ffn,
                    cond_dim, text_dim, max_batch, max_tokens, max_text_tokens, eps, staging,
                    register_budget_bytes, bytes_block)


def dlo_block_bytes(desc: dlo_desc) -> int:
    return int(_c["dlo_block_bytes"](ctypes.byref(desc)))


def dlo_workspace_bytes(desc: dlo_desc) -> int:
    return int(_c["dlo_workspace_bytes"](ctypes.byref(desc)))


def dlo_workspace_bytes_multi(descs) -> int:
    arr = (dlo_desc * len(descs))(*descs)
    return int(_c["dlo_workspace_bytes_multi"](arr, len(descs)))


def dlo_block_layout(desc: dlo_desc) -> list[dict]:
    n = _int(0)
    _check(_c["dlo_block_layout"](ctypes.byref(desc), None, 0, ctypes.byref(n)))
    arr = (dlo_tensor_info * n.value)()
    _check(_c["dlo_block_layout"](ctypes.byref(desc), arr, n.value, ctypes.byref(n)))
    out = []
    for t in arr:
        shape = (t.shape[0],) if t.ndim == 1 else (t.shape[0], t.shape[1])
        out.append({"name": t.name.decode(), "offset": t.offset, "bytes": t.bytes,
                    "dtype": t.dtype, "shape": shape, "source": t.source})
    return out


def dlo_pack_block(desc: dlo_desc, tensors: dict, flat_ptr: int, flat_bytes: int) -> None:
    """tensors: name -> C-contiguous float32 numpy array, for every source entry."""
    import numpy as np
    lay = dlo_block_layout(desc)
    ptrs = (_vp * len(lay))()
    keep = []
    for i, e in enumerate(lay):
        if not e["source"]:
            continue
        a = np.ascontiguousarray(tensors[e["name"]], dtype=np.float32)
        if tuple(a.shape) != tuple(e["shape"]):
            raise ValueError(f"{e['name']}: shape {a.shape} != layout {e['shape']}")
        keep.append(a)
        ptrs[i] = a.ctypes.data
    _check(_c["dlo_pack_block"](ctypes.byref(desc), ptrs, len(lay), flat_ptr, flat_bytes))


def dlo_quantize_e4m3(w):
    """(codes uint8 array, scale float) of one fp32 tensor."""
    import numpy as np
    a = np.ascontiguousarray(w, dtype=np.float32)
    codes = np.empty(a.shape, dtype=np.uint8)
    s = _f32(0.0)
    _check(_c["dlo_quantize_e4m3"](a.ctypes.data, a.size, codes.ctypes.data, ctypes.byref(s)))
    return codes, s.value


# ------------------------------------------------------------------ lifecycle

def dlo_create(desc: dlo_desc, device: int, slot0: int, slot1: int, slot_bytes: int,
               workspace: int, ws_bytes: int, compute_stream: int, copy_stream: int) -> int:
    out = _vp(0)
    st = _c["dlo_create"](ctypes.byref(desc), device, slot0, slot1, slot_bytes, workspace, ws_bytes,
                          compute_stream, copy_stream, ctypes.byref(out))
    _check(st, None)
    return out.value


def dlo_create_multi(descs, device: int, slot0: int, slot1: int, slot_bytes: int, workspace: int,
                     ws_bytes: int, compute_stream: int, copy_stream: int) -> int:
    arr = (dlo_desc * len(descs))(*descs)
    out = _vp(0)
    st = _c["dlo_create_multi"](arr, len(descs), device, slot0, slot1, slot_bytes, workspace, ws_bytes,
                                compute_stream, copy_stream, ctypes.byref(out))
    _check(st, None)
    return out.value


def dlo_register_host_blocks(ctx: int, host_ptrs, block_bytes: int, flags: int) -> None:
    arr = (_vp * len(host_ptrs))(*host_ptrs)
    _check(_c["dlo_register_host_blocks"](ctx, len(host_ptrs), arr, block_bytes, flags), ctx)


def dlo_set_resident(ctx: int, device_ptrs) -> None:
    arr = (_vp * max(1, len(device_ptrs)))(*device_ptrs)
    _check(_c["dlo_set_resident"](ctx, len(device_ptrs), arr), ctx)


def dlo_forward(ctx: int, x_in: int, cond: int, ctx_tokens: int | None, batch: int, tokens: int,
                text_tokens: int, x_out: int) -> None:
    _check(_c["dlo_forward"](ctx, x_in, cond, ctx_tokens, batch, tokens, text_tokens, x_out), ctx)


def dlo_forward_multi(ctx: int, x_in: int, conds, ctx_tokens: int | None, batch: int, tokens: int,
                      text_tokens: int, x_out: int) -> None:
    arr = (_vp * len(conds))(*conds)
    _check(_c["dlo_forward_multi"](ctx, x_in, arr, ctx_tokens, batch, tokens, text_tokens, x_out), ctx)


def dlo_forward_host(ctx: int, x_in: int, cond: int, ctx_tokens: int | None, batch: int,
                     tokens: int, text_tokens: int, x_out: int, timeout_ms: int = 0) -> None:
    _check(_c["dlo_forward_host"](ctx, x_in, cond, ctx_tokens, batch, tokens, text_tokens, x_out,
                                  timeout_ms), ctx)


def dlo_wait(ctx: int, timeout_ms: int = 0) -> None:
    _check(_c["dlo_wait"](ctx, timeout_ms), ctx)


def dlo_destroy(ctx: int) -> int:
    return int(_c["dlo_destroy"](ctx))


def dlo_last_error(ctx: int | None = None) -> str:
    return _err(ctx)


def dlo_get_stats(ctx: int) -> dict:
    s = dlo_stats()
    _check(_c["dlo_get_stats"](ctx, ctypes.byref(s)), ctx)
    return s.as_dict()


def dlo_get_log(ctx: int, cap: int = 65536) -> list[tuple]:
    n = _int(0)
    k = (_int * cap)()
    b = (_int * cap)()
    s = (_int * cap)()
    _check(_c["dlo_get_log"](ctx, k, b, s, cap, ctypes.byref(n)), ctx)
    m = min(n.value, cap)
    return [("stage" if k[i] == 0 else "exec", b[i], None if s[i] < 0 else s[i]) for i in range(m)]


def dlo_reset_log(ctx: int) -> None:
    _check(_c["dlo_reset_log"](ctx), ctx)


def dlo_set_timing(ctx: int, level: int) -> None:
    _check(_c["dlo_set_timing"](ctx, int(level)), ctx)


def dlo_set_graphs(ctx: int, on: bool) -> None:
    _check(_c["dlo_set_graphs"](ctx, 1 if on else 0), ctx)


def dlo_verify_slot(ctx: int, slot: int, block: int = -1) -> int:
    """Returns OK or EMISMATCH; raises on other errors."""
    st = _c["dlo_verify_slot"](ctx, slot, block)
    if st not in (OK, EMISMATCH):
        _check(st, ctx)
    return st


def dlo_debug_fail_register(nth: int) -> None:
    _c["dlo_debug_fail_register"](nth)


# ------------------------------------------------------------------ unit ops

def dlo_op_gemm(A, W, w_dtype, scales, scale_seg, bias, M, N, K, epilogue, out, ldo, gate, gate_ld,
                rows_per_batch, err, stream) -> None:
    _check(_c["dlo_op_gemm"](A, W, w_dtype, scales, scale_seg, bias, M, N, K, epilogue, out, ldo,
                             gate, gate_ld, rows_per_batch, err, stream))


def dlo_op_gemm_noalloc(A, W, w_dtype, scales, scale_seg, bias, M, N, K, epilogue, out, ldo, gate,
                        gate_ld, rows_per_batch, stream) -> None:
    _check(_c["dlo_op_gemm_noalloc"](A, W, w_dtype, scales, scale_seg, bias, M, N, K, epilogue, out,
                                     ldo, gate, gate_ld, rows_per_batch, stream))


def dlo_op_wait_selftest(err, stream) -> None:
    _check(_c["dlo_op_wait_selftest"](err, stream))


def dlo_debug_device_timeout(ctx: int) -> None:
    _check(_c["dlo_debug_device_timeout"](ctx), ctx)


def dlo_op_quantize_act(x, rows, cols, ld, q, scale, scratch, stream) -> None:
    _check(_c["dlo_op_quantize_act"](x, rows, cols, ld, q, scale, scratch, stream))


def dlo_op_gemm_w8a8(A, a_scale, W, scales, scale_seg, bias, M, N, K, epilogue, out, ldo, gate,
                     gate_ld, rows_per_batch, err, stream) -> None:
    _check(_c["dlo_op_gemm_w8a8"](A, a_scale, W, scales, scale_seg, bias, M, N, K, epilogue, out, ldo,
                                  gate, gate_ld, rows_per_batch, err, stream))


def dlo_op_attention(Q, K, V, O, batch, heads, head_dim, nq, nk, ldq, ldk, ldv, ldo, stream) -> None:
    _check(_c["dlo_op_attention"](Q, K, V, O, batch, heads, head_dim, nq, nk, ldq, ldk, ldv, ldo,
                                  stream))


def dlo_op_layernorm(x, rows, D, rows_per_batch, shift, scale, mod_ld, w, b, eps, out, stream) -> None:
    _check(_c["dlo_op_layernorm"](x, rows, D, rows_per_batch, shift, scale, mod_ld, w, b, eps, out,
                                  stream))


def dlo_op_rmsnorm(x, rows, D, ld, col0, w, eps, stream) -> None:
    _check(_c["dlo_op_rmsnorm"](x, rows, D, ld, col0, w, eps, stream))


def dlo_op_adaln(c, B, C, W, bias, N, m, stream) -> None:
    _check(_c["dlo_op_adaln"](c, B, C, W, bias, N, m, stream))


def dlo_op_stage(dst, src, nbytes, mode, stream) -> None:
    _check(_c["dlo_op_stage"](dst, src, nbytes, mode, stream))
