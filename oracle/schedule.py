"""Circular two-slot prefetch order -- oracle (test infrastructure only).

Follows "CPU Offloading for Diffusion Models", section "Layerwise (Blockwise)
Offloading", Execution Flow table: before block i computes, block i+1 is
prefetched, and the last block prefetches the first block again.  Two device
slots hold the streamed blocks ("Distributed Layerwise Offload", section
"AllGather path": two shared device buffers; "Fixed double-buffer" in the
user guide's "Distributed Layerwise Offloading" key features).  Resident
leading layers ("Distributed Layerwise Offload", Feature compatibility table,
row "Resident leading layers") are never staged; the ring then runs over the
streamed blocks k..n-1, so the block after n-1 is k.

The first streamed block is staged into slot 0 before the first forward
("Distributed Layerwise Offload", Startup and runtime sequence: "prime the
first block").
"""
from __future__ import annotations


def next_block(i: int, n: int, k: int) -> int:
    """Block prefetched while streamed block i computes (k <= i < n)."""
    if not (k <= i < n):
        raise ValueError("i must be a streamed block")
    return i + 1 if i < n - 1 else k


def schedule(n: int, k: int, steps: int):
    """Ordered staging/execution events of `steps` stack forwards.

    Returns a list of tuples:
      ("stage", block, slot)   copy of `block` into device slot `slot`
      ("exec", block, slot)    execution of `block`; slot is None for a
                               resident block
    The priming stage comes first.  Streamed execution j (counted over all
    steps) reads slot j % 2; the stage issued just before it writes
    next_block(block_j) into slot (j + 1) % 2.
    """
    if not (0 <= k <= n):
        raise ValueError("need 0 <= k <= n")
    ev = []
    if k < n:
        ev.append(("stage", k, 0))
    j = 0
    for _ in range(steps):
        for i in range(k):
            ev.append(("exec", i, None))
        for i in range(k, n):
            ev.append(("stage", next_block(i, n, k), (j + 1) % 2))
            ev.append(("exec", i, j % 2))
            j += 1
    return ev
