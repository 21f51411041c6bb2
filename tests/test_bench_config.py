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


def test_traffic_records_follow_code_not_comments(tmp_path):
    """A committed ncu traffic record is shown only while its kernel source's
    code is unchanged: comments and whitespace may change, code may not; the
    committed records match the committed sources."""
    base = "__global__ void k(int* p) { p[0] = 1; }  // store one\n"
    a, b, c = tmp_path / "a.cu", tmp_path / "b.cu", tmp_path / "c.cu"
    a.write_text(base)
    b.write_text("/* a kernel */\n__global__  void k(int* p) {\n  p[0] = 1;  // store\n}\n")
    c.write_text(base.replace("= 1", "= 2"))
    assert bench.source_digest(str(a)) == bench.source_digest(str(b))
    assert bench.source_digest(str(a)) != bench.source_digest(str(c))
    assert bench.traffic_record("dit-xl-28x1152-b2-n1024", "gemm_bf16") is not None
    assert bench.traffic_record("video-fp8-40x5120-n8192", "gemm_e4m3") is not None
    assert bench.traffic_record("dit-xl-28x1152-b2-n1024", "attention") is None
