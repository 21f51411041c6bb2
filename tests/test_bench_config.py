"""Host logic of the bench line's `config`: both arms build it with one
function, the streamed-bytes note follows residency and the L2 size, and
the block sizes come from the library's layout table (CPU only)."""
import argparse

import pytest

import bench
import synth


def _args(**kw):
    a = dict(resident=0, staging="memcpy", host="pinned", no_graphs=False)
    a.update(kw)
    return argparse.Namespace(**a)


def test_config_of_the_dit_xl_workload():
    cfg = synth.CFG_DITXL
    parts = bench.parts_of(cfg)
    sizes = [47810304]
    c = bench.run_config(_args(), cfg, parts, sizes, 1)
    assert c["workload"] == cfg.name and c["blocks"] == 28 and c["parallelism"] == "single"
    assert c["containers"] == [{"kind": "dit", "blocks": 28, "heads": 16, "ffn": 4608,
                                "block_bytes": 47810304, "weights": "bf16"}]
    assert c["l2"].startswith("inputs larger than L2: 1.34 GB")
    # resident blocks are not streamed; replicas under torchrun
    c = bench.run_config(_args(resident=27), cfg, parts, sizes, 4)
    assert c["l2"].startswith("inputs smaller than L2 (47.8 MB")
    assert c["parallelism"] == "replicas" and c["resident"] == 27


def test_multi_container_config_lists_every_container():
    mc = synth.MULTI_DITXL
    parts = bench.parts_of(mc)
    sizes = [1000, 2000][:len(parts)]
    c = bench.run_config(_args(no_graphs=True), mc, parts, sizes, 1)
    assert [x["blocks"] for x in c["containers"]] == [p.n_blocks for p in parts]
    assert c["graphs"] is False
    assert sum(x["blocks"] for x in c["containers"]) == c["blocks"]


def test_block_sizes_come_from_the_layout_table():
    dlo = pytest.importorskip("layerwise_weight_offload_slot_gb300")
    parts = bench.parts_of(synth.CFG_DITXL)
    assert bench.container_bytes_of(parts) == [dlo.dlo_block_bytes(dlo.make_desc(
        block_kind=dlo.BLOCK_DIT, n_blocks=28, hidden=1152, heads=16, head_dim=72, ffn=4608,
        cond_dim=synth.CFG_DITXL.cond_dim, max_batch=2, max_tokens=1024))]
