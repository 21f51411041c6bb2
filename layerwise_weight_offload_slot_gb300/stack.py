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
               dlo_block_bytes, dlo_block_layout, dlo_create, dlo_destroy, dlo_forward,
               dlo_forward_host, dlo_get_log, dlo_get_stats, dlo_pack_block,
               dlo_register_host_blocks, dlo_reset_log, dlo_set_resident, dlo_set_timing,
               dlo_verify_slot, dlo_wait, dlo_workspace_bytes, make_desc)

PAGE = 4096


def _round(n: int, a: int) -> int:
    return (n + a - 1) // a * a


class HostBlocks:
    """n flat blocks of `block_bytes`, each page-aligned, in one allocation.

    mode "pinned": torch pinned memory (cudaHostAlloc); "register": anonymous
    mmap (pageable) for the library to register; "pageable": anonymous mmap
    that stays pageable (the library packs it through pinned host slots).
    """

    def __init__(self, n: int, block_bytes: int, mode: str):
        self.n = n
        self.block_bytes = block_bytes
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
        return np.ctypeslib.as_array((ctypes.c_uint8 * self.block_bytes).from_address(self.ptrs[i]))

    def close(self):
        self._t = None
        if self._buf is not None:
            self._anchor = None
            self._buf.close()
            self._buf = None


class OffloadStack:
    def __init__(self, *, block_kind: int, n_blocks: int, hidden: int = 0, heads: int = 0,
                 head_dim: int = 0, ffn: int = 0, cond_dim: int = 0, text_dim: int = 0,
                 max_batch: int = 1, max_tokens: int = 1, max_text_tokens: int = 0,
                 wdtype: int = W_BF16, eps: float = 1e-6, staging: int = STAGE_MEMCPY,
                 host_mode: str = "pinned", register_budget_bytes: int = 0,
                 bytes_block: int = 0, device: int = 0, host: "HostBlocks | None" = None):
        self.desc = make_desc(block_kind=block_kind, n_blocks=n_blocks, hidden=hidden, heads=heads,
                              head_dim=head_dim, ffn=ffn, cond_dim=cond_dim, text_dim=text_dim,
                              max_batch=max_batch, max_tokens=max_tokens,
                              max_text_tokens=max_text_tokens, wdtype=wdtype, eps=eps,
                              staging=staging, register_budget_bytes=register_budget_bytes,
                              bytes_block=bytes_block)
        self.block_bytes = dlo_block_bytes(self.desc)
        if self.block_bytes == 0:
            raise ValueError("invalid stack description")
        self.layout = dlo_block_layout(self.desc)
        self.ws_bytes = dlo_workspace_bytes(self.desc)
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
        self.host = host if host is not None else HostBlocks(n_blocks, self.block_bytes, host_mode)
        self.host_mode = host_mode
        self.n_blocks = n_blocks
        self.kind = block_kind
        self._resident = []
        torch.cuda.synchronize(self.dev)
        self.ctx = dlo_create(self.desc, device, self.slot_ptrs[0], self.slot_ptrs[1], sb,
                              self.ws_ptr, self.ws_bytes, self.compute_stream.cuda_stream,
                              self.copy_stream.cuda_stream)

    # ---------------------------------------------------------------- setup
    def pack(self, i: int, params: dict) -> None:
        dlo_pack_block(self.desc, params, self.host.ptrs[i], self.block_bytes)

    def pack_all(self, blocks, threads: int = 8) -> None:
        """blocks: list of param dicts, or a callable i -> param dict."""
        get = blocks if callable(blocks) else (lambda i: blocks[i])
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda i: self.pack(i, get(i)), range(self.n_blocks)))

    def attach(self) -> None:
        flags = {"pinned": HOST_PINNED, "register": HOST_REGISTER,
                 "pageable": HOST_PAGEABLE}[self.host_mode]
        dlo_register_host_blocks(self.ctx, self.host.ptrs, self.block_bytes, flags)

    def set_resident(self, k: int) -> None:
        bufs = []
        for _ in range(k):
            t = torch.empty(self.block_bytes + 256, dtype=torch.uint8, device=self.dev)
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

    def forward(self, x: torch.Tensor, cond: torch.Tensor, ctx_tokens: torch.Tensor | None = None,
                out: torch.Tensor | None = None) -> torch.Tensor:
        B, N, _ = x.shape
        L = ctx_tokens.shape[1] if ctx_tokens is not None else 0
        if out is None:
            out = torch.empty_like(x)
        cur = torch.cuda.current_stream(self.dev)
        self.compute_stream.wait_stream(cur)
        dlo_forward(self.ctx, x.data_ptr(), cond.data_ptr(),
                    ctx_tokens.data_ptr() if ctx_tokens is not None else None, B, N, L,
                    out.data_ptr())
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
