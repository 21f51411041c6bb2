"""Torch plumbing around the C ABI: device memory, streams and host blocks.

`OffloadStack` allocates the two device slots, the workspace and the optional
resident buffers with torch, owns one compute and one copy stream, lays the
flat host blocks out in pinned (cudaHostAlloc) or anonymous-mmap memory that
the library registers itself, and calls the dlo_* functions.  No step of the
offload path runs here.
"""
from __future__ import annotations

import ctypes
import mmap
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from . import (BLOCK_BYTES, BLOCK_DIT, BLOCK_VIDEO, HOST_PAGEABLE, HOST_PINNED, HOST_REGISTER, OK, STAGE_MEMCPY, W_BF16,
               dlo_block_bytes, dlo_block_layout, dlo_create, dlo_create_multi, dlo_destroy,
               dlo_forward, dlo_forward_host, dlo_forward_multi, dlo_get_log, dlo_get_stats,
               dlo_pack_block, dlo_register_host_blocks, dlo_reset_log, dlo_set_resident,
               dlo_set_graphs, dlo_set_timing, dlo_verify_slot, dlo_wait, dlo_workspace_bytes,
               dlo_workspace_bytes_multi, make_desc)

PAGE = 4096


def _round(n: int, a: int) -> int:
    return (n + a - 1) // a * a


class HostBlocks:
    """n flat blocks of `block_bytes` (or sizes[i] <= block_bytes each), each
    page-aligned, in one allocation.

    mode "pinned": torch pinned memory (cudaHostAlloc); "register": anonymous
    mmap (pageable) for the library to register; "pageable": anonymous mmap
    that stays pageable (the library packs it through pinned host slots).
    """

    def __init__(self, n: int, block_bytes: int, mode: str, sizes=None):
        self.n = n
        self.block_bytes = block_bytes
        self.sizes = list(sizes) if sizes is not None else [block_bytes] * n
        self.stride = _round(block_bytes, PAGE)
        total = self.stride * n + PAGE
        self.mode = mode
        if mode == "pinned":
            self._t = torch.empty(total, dtype=torch.uint8, pin_memory=True)
            base = self._t.data_ptr()
            self._buf = None
        elif mode in ("register", "pageable"):
            self._buf = mmap.mmap(-1, total)
            self._anchor = ctypes.c_char.from_buffer(self._buf)
            base = ctypes.addressof(self._anchor)
            self._t = None
        else:
            raise ValueError(mode)
        self.base = _round(base, PAGE)
        self.ptrs = [self.base + i * self.stride for i in range(n)]

    def view(self, i: int) -> np.ndarray:
        """numpy uint8 view of block i (host memory)."""
        return np.ctypeslib.as_array((ctypes.c_uint8 * self.sizes[i]).from_address(self.ptrs[i]))

    def close(self):
        self._t = None
        if self._buf is not None:
            self._anchor = None
            self._buf.close()
            self._buf = None


class OffloadStack:
    """One block stack.  Either one container (block_kind, n_blocks and the
    per-block fields as keywords) or several ordered containers:
    containers = [dict(block_kind=..., n_blocks=..., heads=..., head_dim=...,
    ffn=..., cond_dim=..., text_dim=..., max_text_tokens=..., wdtype=...), ...]
    with the shared fields (hidden, max_batch, max_tokens, eps, staging,
    register_budget_bytes) given once.  Blocks are numbered across containers
    in order."""

    def __init__(self, *, block_kind: int = BLOCK_DIT, n_blocks: int = 0, hidden: int = 0,
                 heads: int = 0, head_dim: int = 0, ffn: int = 0, cond_dim: int = 0,
                 text_dim: int = 0, max_batch: int = 1, max_tokens: int = 1,
                 max_text_tokens: int = 0, wdtype: int = W_BF16, eps: float = 1e-6,
                 staging: int = STAGE_MEMCPY, host_mode: str = "pinned",
                 register_budget_bytes: int = 0, bytes_block: int = 0, device: int = 0,
                 host: "HostBlocks | None" = None, containers=None):
        shared = dict(hidden=hidden, max_batch=max_batch, max_tokens=max_tokens, eps=eps,
                      staging=staging, register_budget_bytes=register_budget_bytes)
        if containers is None:
            containers = [dict(block_kind=block_kind, n_blocks=n_blocks, heads=heads,
                               head_dim=head_dim, ffn=ffn, cond_dim=cond_dim, text_dim=text_dim,
                               max_text_tokens=max_text_tokens, wdtype=wdtype,
                               bytes_block=bytes_block)]
        self.descs = [make_desc(**{**shared, **ct}) for ct in containers]
        self.multi = len(self.descs) > 1
        self.desc = self.descs[0]
        self.container_bytes = [dlo_block_bytes(d) for d in self.descs]
        if not all(self.container_bytes):
            raise ValueError("invalid stack description")
        self.container_of = [ci for ci, d in enumerate(self.descs) for _ in range(d.n_blocks)]
        self.block_sizes = [self.container_bytes[ci] for ci in self.container_of]
        self.block_bytes = max(self.container_bytes)
        self.layouts = [dlo_block_layout(d) for d in self.descs]
        self.layout = self.layouts[0]
        self.ws_bytes = (dlo_workspace_bytes_multi(self.descs) if self.multi
                         else dlo_workspace_bytes(self.desc))
        if self.ws_bytes == 0:
            raise ValueError("invalid stack description")
        n_blocks = len(self.container_of)
        block_kind = self.desc.block_kind
        self.device = device
        self.dev = torch.device("cuda", device)
        sb = _round(self.block_bytes, 256)
        self.slot_bytes = sb
        self._slots = torch.empty(2 * sb + 256, dtype=torch.uint8, device=self.dev)
        s0 = _round(self._slots.data_ptr(), 256)
        self.slot_ptrs = (s0, s0 + sb)
        self._ws = torch.empty(self.ws_bytes + 256, dtype=torch.uint8, device=self.dev)
        self.ws_ptr = _round(self._ws.data_ptr(), 256)
        self.compute_stream = torch.cuda.Stream(device=self.dev)
        self.copy_stream = torch.cuda.Stream(device=self.dev)
        # host blocks may be shared between contexts (pinned mode only)
        self._own_host = host is None
        self.host = host if host is not None else HostBlocks(n_blocks, self.block_bytes, host_mode,
                                                             sizes=self.block_sizes)
        self.host_mode = host_mode
        self.n_blocks = n_blocks
        self.kind = block_kind
        self._resident = []
        torch.cuda.synchronize(self.dev)
        create = dlo_create_multi if self.multi else dlo_create
        self.ctx = create(self.descs if self.multi else self.desc, device, self.slot_ptrs[0],
                          self.slot_ptrs[1], sb, self.ws_ptr, self.ws_bytes,
                          self.compute_stream.cuda_stream, self.copy_stream.cuda_stream)

    # ---------------------------------------------------------------- setup
    def pack(self, i: int, params: dict) -> None:
        dlo_pack_block(self.descs[self.container_of[i]], params, self.host.ptrs[i],
                       self.block_sizes[i])

    def pack_all(self, blocks, threads: int = 8) -> None:
        """blocks: list of param dicts, or a callable i -> param dict."""
        get = blocks if callable(blocks) else (lambda i: blocks[i])
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda i: self.pack(i, get(i)), range(self.n_blocks)))

    def attach(self) -> None:
        flags = {"pinned": HOST_PINNED, "register": HOST_REGISTER,
                 "pageable": HOST_PAGEABLE}[self.host_mode]
        dlo_register_host_blocks(self.ctx, self.host.ptrs, 0 if self.multi else self.block_bytes,
                                 flags)

    def set_resident(self, k: int) -> None:
        bufs = []
        for i in range(k):
            t = torch.empty(self.block_sizes[i] + 256, dtype=torch.uint8, device=self.dev)
            bufs.append(t)
        self._resident = bufs
        dlo_set_resident(self.ctx, [_round(t.data_ptr(), 256) for t in bufs])

    # ---------------------------------------------------------------- run
    def forward_bytes(self, sums: torch.Tensor | None = None) -> torch.Tensor:
        """One pass over an opaque bytes stack; per-block uint64 checksums (as int64)."""
        if sums is None:
            sums = torch.zeros(self.n_blocks, dtype=torch.int64, device=self.dev)
        cur = torch.cuda.current_stream(self.dev)
        self.compute_stream.wait_stream(cur)
        dlo_forward(self.ctx, None, None, None, 1, 1, 0, sums.data_ptr())
        cur.wait_stream(self.compute_stream)
        return sums

    def forward(self, x: torch.Tensor, cond, ctx_tokens: torch.Tensor | None = None,
                out: torch.Tensor | None = None) -> torch.Tensor:
        """cond: one tensor for all containers, or a list with one per container."""
        B, N, _ = x.shape
        L = ctx_tokens.shape[1] if ctx_tokens is not None else 0
        if out is None:
            out = torch.empty_like(x)
        cur = torch.cuda.current_stream(self.dev)
        self.compute_stream.wait_stream(cur)
        tok = ctx_tokens.data_ptr() if ctx_tokens is not None else None
        if isinstance(cond, (list, tuple)):
            dlo_forward_multi(self.ctx, x.data_ptr(), [c.data_ptr() for c in cond], tok, B, N, L,
                              out.data_ptr())
        else:
            dlo_forward(self.ctx, x.data_ptr(), cond.data_ptr(), tok, B, N, L, out.data_ptr())
        cur.wait_stream(self.compute_stream)
        return out

    def forward_host(self, x: np.ndarray, cond: np.ndarray, ctx_tokens: np.ndarray | None,
                     out: np.ndarray) -> np.ndarray:
        B, N = x.shape[0], x.shape[1]
        L = ctx_tokens.shape[1] if ctx_tokens is not None else 0
        dlo_forward_host(self.ctx, x.ctypes.data, cond.ctypes.data,
                         ctx_tokens.ctypes.data if ctx_tokens is not None else None, B, N, L,
                         out.ctypes.data)
        return out

    def wait(self, timeout_ms: int = 0) -> None:
        dlo_wait(self.ctx, timeout_ms)

    def stats(self) -> dict:
        return dlo_get_stats(self.ctx)

    def log(self) -> list:
        return dlo_get_log(self.ctx)

    def reset_log(self) -> None:
        dlo_reset_log(self.ctx)

    def set_timing(self, level: int) -> None:
        dlo_set_timing(self.ctx, level)

    def set_graphs(self, on: bool) -> None:
        dlo_set_graphs(self.ctx, on)

    def verify_slot(self, slot: int, block: int = -1) -> bool:
        return dlo_verify_slot(self.ctx, slot, block) == OK

    def close(self) -> int:
        st = 0
        if self.ctx:
            st = dlo_destroy(self.ctx)
            self.ctx = 0
        if self._own_host:
            self.host.close()
        self._resident = []
        return st

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
