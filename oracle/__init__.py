"""CPU oracle for the streamed DiT block stack -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct numpy code in float64.  It shares no code with
the CUDA library (`layerwise_weight_offload_slot_gb300`) and imports nothing
from it.  Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import or run anything in this package; the product path never
does and fails loudly when its CUDA library is missing.

Modules
  schedule  the circular two-slot prefetch order (CPU Offloading for Diffusion
            Models, "Layerwise (Blockwise) Offloading", Execution Flow table)
  fp8       OCP FP8 E4M3 decode and the per-tensor quantiser (amax / 448)
  dit       DiT adaLN-zero block and video-DiT block forward, stack forward

What pins each function (tests/test_oracle_*.py, run with -m "not gpu"):
  schedule  the page's Execution Flow table (tests/golden/), brute-force
            simulation of slot contents for n <= 6, k <= n, steps <= 3
  fp8       all 256 codes against the closed-form OCP definition and against
            torch.float8_e4m3fn; rounding against torch's RNE cast
  dit       primitives against torch library routines (layer_norm, gelu,
            silu, scaled_dot_product_attention); whole DiT block against a
            composition of torch.nn library modules (nn.LayerNorm,
            nn.MultiheadAttention, nn.Linear); closed forms (zero gates give
            the identity, equal keys give the mean of v); invariants (token
            permutation equivariance, batch independence)
  The block math is not printed on the pages, so the block functions are
  pinned to the standard DiT definitions above, not to page values.
"""
