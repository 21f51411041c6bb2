"""The Python quick start of the library's documentation, as a test: the same
calls, on the tiny DiT stack instead of DiT-XL to keep the test short."""
import pytest
import torch

import synth

dlo = pytest.importorskip("layerwise_weight_offload_slot_gb300")

pytestmark = pytest.mark.gpu


def quick_start(cfg):
    from layerwise_weight_offload_slot_gb300.stack import OffloadStack

    st = OffloadStack(block_kind=dlo.BLOCK_DIT, n_blocks=cfg.n_blocks, hidden=cfg.hidden,
                      heads=cfg.heads, head_dim=cfg.head_dim, ffn=cfg.ffn, cond_dim=cfg.cond_dim,
                      max_batch=cfg.batch, max_tokens=cfg.tokens)
    st.pack_all(lambda i: synth.block_params(cfg, i))
    st.attach()
    st.set_resident(0)
    st.set_graphs(True)

    x = torch.randn(cfg.batch, cfg.tokens, cfg.hidden, device="cuda").to(torch.bfloat16)
    c = torch.randn(cfg.batch, cfg.cond_dim, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(x)
    for step in range(10):
        st.forward(x, c, out=out)
        x, out = out, x
    st.wait()
    stats, log = st.stats(), st.log()
    st.close()
    return st, stats, log, x


def test_quick_start_runs():
    cfg = synth.CFG_TINY
    st, stats, log, x = quick_start(cfg)
    assert st.ctx == 0   # closed
    assert stats["forwards"] == 10
    assert stats["staged_bytes"] == stats["stagings"] * st.block_bytes
    assert log[0] == ("stage", 0, 0)   # the prime: block 0 staged into slot 0
    assert bool(torch.isfinite(x.float()).all())
