"""CPU checks of the host-side logic around the step: workload shapes, the
benchmark's work accounting and schedule helpers.  No GPU and no library call."""
import math

import numpy as np
import pytest

import bench
import oracle as O
import workloads as W


@pytest.mark.parametrize("name", ["c3", "c4", "c4bf16"])
def test_conv_geometry_matches_layer_shapes(name):
    """Every convolution's geometry gives its layer's d_in and row count, and the
    oracle's patch matrix has that shape."""
    cfg = W.get_config(name)
    convs = [l for l in cfg.layers if l.conv is not None]
    assert convs
    for l in convs:
        c = l.conv
        assert c.c_in * c.kh * c.kw == l.d_in
        assert c.batch * c.h_out * c.w_out == l.rows
        assert c.h_out == O.conv_out_size(c.h, c.kh, c.sh, c.ph, c.dh)
        assert c.w_out == O.conv_out_size(c.w, c.kw, c.sw, c.pw, c.dw)
    # a small batch of the first convolution, through the oracle's im2col
    li = cfg.layers.index(convs[0])
    d = W.conv_inputs(cfg, li, 1, batch=1)
    c = d["geom"]
    P = O.im2col(d["x"], (c.kh, c.kw), (c.sh, c.sw), (c.ph, c.pw), (c.dh, c.dw))
    assert P.shape == (c.h_out * c.w_out, convs[0].d_in)


def test_conv_draws_are_seeded_and_distinct():
    cfg = W.get_config("c3")
    a = W.conv_inputs(cfg, 2, 1, batch=1)["x"]
    b = W.conv_inputs(cfg, 2, 1, batch=1)["x"]
    c = W.conv_inputs(cfg, 2, 2, batch=1)["x"]
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    assert (a >= 0).all()                         # post-ReLU activations


def test_qkv_ties_map_key_and_value_to_query():
    cfg, layers = bench.bench_config("transformer4_qkv_tied")
    ties = bench.qkv_ties(layers)
    assert len(ties) == 8                          # k and v of 4 blocks
    for li, src in ties.items():
        blk, _, proj = layers[li].name.rpartition(".")
        assert proj in ("k", "v") and layers[src].name == f"{blk}.q"
        assert layers[li].n == layers[src].n and layers[li].kind == layers[src].kind == "kron"


def test_work_accounting_of_the_variants():
    """Shared A factors drop their products and inverses; an inverse-free refresh
    counts 7 n^3 per factor; NCHW inputs read the tensors, not the patches."""
    cfg, layers = bench.bench_config("transformer4_qkv_tied")
    ties = set(bench.qkv_ties(layers))
    base = bench.algorithmic(layers, 10)
    tied = bench.algorithmic(layers, 10, tied=ties)
    drop = sum(l.rows * l.n * (l.n + 1) for i, l in enumerate(layers) if i in ties)
    assert math.isclose(base["factor_flop"] - tied["factor_flop"], drop, rel_tol=1e-12)
    cfg2, layers2 = bench.bench_config("mlp4")
    a = bench.algorithmic(layers2, 10)
    b = bench.algorithmic(layers2, 10, ikfac=True)
    assert math.isclose(b["invert_flop"], 7 * a["invert_flop"], rel_tol=1e-12)
    cfg3, layers3 = bench.bench_config("resnet18_nchw")
    u = bench.algorithmic(layers3, 20)
    v = bench.algorithmic(layers3, 20, nchw=True)
    assert v["factor_bytes"] < u["factor_bytes"]
    assert v["factor_flop"] == u["factor_flop"]


def test_stale_schedule_matches_bench_refresh_cadence():
    """With no warm-up and equal cadences the stale schedule is the plain one
    (refresh at t = 1, 1 + k, ...) shifted to start after the warm-up step."""
    k = 10
    flags = [O.stale_refresh(t, 1, k, k) for t in range(1, 42)]
    plain = [(t - 1) % k == 0 for t in range(1, 42)]
    assert [f[0] for f in flags] == plain and [f[1] for f in flags] == plain


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the float64 oracle on the host) prints one JSON
    line with the contract's keys, on the GPU arm's metric and workload name."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--workload", "single_linear", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "steps/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"].startswith("single_linear_64x32_b128")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "steps/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def _run_bench(args, env_extra):
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(root, "bench.py")] + args,
                          capture_output=True, text=True, timeout=300, cwd=root, env=env)


def test_gpu_arm_refuses_more_than_one_rank():
    """The library is single-GPU: the GPU arm exits with a message (and no JSON
    line) when started as one of several ranks or with --gpus > 1, before it
    touches a GPU."""
    r = _run_bench(["--workload", "single_linear"], {"WORLD_SIZE": "2", "RANK": "0"})
    assert r.returncode == 2 and "one GPU only" in r.stderr
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]
    r = _run_bench(["--workload", "single_linear", "--gpus", "2"], {})
    assert r.returncode == 2 and "one GPU only" in r.stderr


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun the reference arm runs on rank 0 alone; other ranks exit 0."""
    r = _run_bench(["--impl", "reference", "--workload", "single_linear", "--steps", "1"],
                   {"WORLD_SIZE": "2", "RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_default_workload_is_the_transformer_set():
    """With no flags the bench times the largest single-GPU layer set: four
    transformer blocks (d_model 2048, FFN 8192, 16384 tokens, bf16 inputs)."""
    import sys
    old = sys.argv
    sys.argv = ["bench.py"]
    try:
        a = bench.parse()
    finally:
        sys.argv = old
    assert a.workload == "transformer4" and a.gpus == 1
    cfg, layers = bench.bench_config(a.workload)
    kron = [l for l in layers if l.kind == "kron"]
    assert len(kron) == 24 and max(l.n for l in kron) == 8193 and max(l.d_out for l in kron) == 8192
    assert all(l.rows == 16384 and l.in_dtype == "bf16" for l in kron)
    assert bench.path_dtype(layers) == "bf16-in/f32"
