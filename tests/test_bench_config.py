"""Host logic of the bench line's `config`: both arms build it with one
function from host arithmetic only (the reference arm loads nothing of the
library), and the streamed-bytes note follows residency and the L2 size."""
import argparse

import bench
import synth


def _args(**kw):
    a = dict(resident=0, staging="memcpy", host="pinned", no_graphs=False)
    a.update(kw)
    return argparse.Namespace(**a)


def test_config_of_the_dit_xl_workload():
    cfg = synth.CFG_DITXL
    parts = bench.parts_of(cfg)
    c = bench.run_config(_args(), cfg, parts, 1)
    assert c["workload"] == cfg.name and c["blocks"] == 28 and c["parallelism"] == "single"
    assert c["containers"] == [{"kind": "dit", "blocks": 28, "heads": 16, "ffn": 4608, "weights": "bf16"}]
    assert c["l2"].startswith("inputs larger than L2: 1.34 GB")
    # resident blocks are not streamed; replicas under torchrun
    c = bench.run_config(_args(resident=27), cfg, parts, 4)
    assert c["l2"].startswith("inputs smaller than L2 (47.8 MB")
    assert c["parallelism"] == "replicas" and c["resident"] == 27


def test_weight_bytes_count_every_parameter():
    # DiT-XL block: adaLN 6D x C + qkv 3D x D + proj D x D + fc1/fc2 2 x F x D, biases, bf16
    D, F, C = 1152, 4608, 1152
    n = 6 * D * C + 6 * D + 3 * D * D + 3 * D + D * D + D + F * D + F + D * F + D
    assert bench.weight_bytes(synth.CFG_DITXL) == 2 * n
    # E4M3 linears: one byte per weight element plus one fp32 scale per linear
    v8 = bench.weight_bytes(synth.CFG_VIDEO_FP8)
    v16 = bench.weight_bytes(synth.CFG_VIDEO)
    lin = sum(int(__import__("numpy").prod(s)) for _, s, r in synth.param_specs(synth.CFG_VIDEO)
              if r == "linear_w")
    assert v16 - v8 == lin - 4 * 10


def test_multi_container_config_lists_every_container():
    mc = synth.MULTI_DITXL
    parts = bench.parts_of(mc)
    c = bench.run_config(_args(no_graphs=True), mc, parts, 1)
    assert [x["blocks"] for x in c["containers"]] == [p.n_blocks for p in parts]
    assert c["graphs"] is False
    assert sum(x["blocks"] for x in c["containers"]) == c["blocks"]


def test_reference_arm_reports_what_it_timed(capsys):
    """--impl reference on the tiny stack: ms_per_step x steps is the time of
    the steps actually run (one block each); value extrapolates to the stack."""
    import json
    args = argparse.Namespace(resident=0, staging="memcpy", host="pinned", no_graphs=False,
                              steps=2, warmup=0)
    bench.run_reference(args, synth.CFG_TINY, 0, 1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    ex = line["extrapolation"]
    assert line["impl"] == "reference" and line["steps"] == 2
    assert ex["blocks_per_timed_step"] == 1 and ex["blocks_per_stack_step"] == 4
    assert abs(ex["stack_ms_per_step"] - 4 * line["ms_per_step"]) <= 1e-6 * ex["stack_ms_per_step"]
    assert abs(line["value"] - 1e3 / ex["stack_ms_per_step"]) <= 1e-9 * line["value"]
