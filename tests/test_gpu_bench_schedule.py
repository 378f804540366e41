"""The benchmark's launch configuration against the float64 oracle.

`bench.py` drives the MLP set (4 Kronecker-factored layers plus a diagonal twin
of each) as batched library calls captured into CUDA graphs, replayed on three
streams: the diagonal step always alongside, the factor update alongside the
preconditioning on steps without a refresh.  This runs that same schedule for
12 steps (refreshes at steps 1 and 11) and compares every layer's parameters
with the oracle.  Tolerances as for the per-call tests: W of the
Kronecker-factored layers 1e-4, of the diagonal layers 1e-6 (relative Frobenius).
"""
import dataclasses

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_helpers import to_dev, to_np, rel_fro

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import second_order_optimizer_gb300 as K  # noqa: E402


def test_mlp_graph_replay_on_three_streams_matches_oracle():
    cfg = W.get_config("c2")
    hp, k, steps, NB = cfg.hp, cfg.invert_every, 12, 2
    kron = list(cfg.layers)
    layers = kron + [dataclasses.replace(l, name=l.name + "_diag", kind="diag") for l in kron]
    nk = len(kron)
    h = K.Kfac([(K.KFAC_KRON if l.kind == "kron" else K.KFAC_DIAG, l.d_out, l.d_in, l.has_bias,
                 K.KFAC_F32) for l in layers], max_rows=max(l.rows for l in layers),
               ema_decay=hp.ema_decay, damping=hp.damping, lr=hp.lr, momentum=hp.momentum,
               weight_decay=hp.weight_decay)
    orc = O.KfacOracle(hp.ema_decay, hp.damping, hp.lr, hp.momentum, hp.weight_decay, k)
    # two seeded input batches, used alternately (step t reads batch t % 2)
    host = [[W.layer_inputs(cfg, li, 1 + b) for li in range(nk)] for b in range(NB)]
    dev = [[{key: (to_dev(v) if v is not None else None) for key, v in x.items()} for x in hb]
           for hb in host]
    states, params = [], []
    for li, l in enumerate(layers):
        w0, b0 = W.initial_params(cfg, li % nk)
        states.append(O.LayerState(l.kind, l.d_out, l.d_in, l.has_bias, w0, b0))
        params.append((to_dev(w0), to_dev(b0)))
    KR, DG = list(range(nk)), list(range(nk, 2 * nk))
    gnew = [torch.empty(l.d_out, device="cuda") for l in kron]
    anew = [torch.empty(l.n, device="cuda") for l in kron]

    def factor(b):
        x = dev[b]
        h.update_factors_batched(KR, [x[i]["a"] for i in KR], [x[i]["g"] for i in KR])

    def precond(b):
        x = dev[b]
        h.precondition_batched(KR, [x[i]["grad_w"] for i in KR], [x[i]["grad_b"] for i in KR],
                               None, None, [params[i][0] for i in KR], [params[i][1] for i in KR])

    def diag(b):
        x = dev[b]
        h.diag_factors_batched(DG, [x[i]["a"] for i in KR], [x[i]["g"] for i in KR], gnew, anew)
        h.diag_step_batched(DG, gnew, anew, [x[i]["grad_w"] for i in KR],
                            [x[i]["grad_b"] for i in KR], [params[i][0] for i in DG],
                            [params[i][1] for i in DG])

    def oracle_step(t):
        x = host[t % NB]
        for i in KR:
            orc.step_kron(states[i], x[i]["a"], x[i]["g"], x[i]["grad_w"], x[i]["grad_b"])
        for j, i in enumerate(DG):
            orc.step_diag(states[i], O.diag_factor(x[j]["g"]), O.diag_factor(x[j]["a"], 1),
                          x[j]["grad_w"], x[j]["grad_b"])

    # step 1 eagerly (factor, refresh, preconditioning, diagonal), as the warm-up does
    factor(1)
    h.invert(-1)
    precond(1)
    diag(1)
    oracle_step(1)
    torch.cuda.synchronize()
    # capture each phase per batch (capture records, it does not run the kernels)
    graphs = {}
    for b in range(NB):
        for name, fn in (("factor", factor), ("precond", precond), ("diag", diag)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn(b)
            graphs[(name, b)] = g
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        h.invert(-1)
    graphs[("invert", 0)] = g
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    side, dside = torch.cuda.Stream(), torch.cuda.Stream()
    e0, e_side, e_d = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
    for t in range(2, steps + 1):
        b, refresh = t % NB, (t - 1) % k == 0
        e0.record(main)
        dside.wait_event(e0)
        with torch.cuda.stream(dside):
            graphs[("diag", b)].replay()
            e_d.record(dside)
        if refresh:
            graphs[("factor", b)].replay()
            graphs[("invert", 0)].replay()
            graphs[("precond", b)].replay()
        else:
            side.wait_event(e0)
            with torch.cuda.stream(side):
                graphs[("factor", b)].replay()
                e_side.record(side)
            graphs[("precond", b)].replay()
            main.wait_event(e_side)
        main.wait_event(e_d)
        oracle_step(t)
    torch.cuda.synchronize()
    assert h.get_status()[0] == 0
    for i, l in enumerate(layers):
        Wg = O.grad_hat(to_np(params[i][0]), to_np(params[i][1]))
        tol = 1e-4 if l.kind == "kron" else 1e-6
        assert rel_fro(Wg, states[i].W) <= tol, (l.name, rel_fro(Wg, states[i].W))


def test_bench_prints_one_contract_line():
    """`bench.py` on the single-linear set prints one JSON line with every key the
    measurement contract asks for."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--workload",
                        "single_linear", "--steps", "20", "--warmup", "3", "--no-cpu-baseline"],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["value"] > 0 and d["gpu_launches"] > 0
    roof = d["roofline"]
    assert roof["bound"] in ("hbm", "tensor", "alu") and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-3, abs=1e-4)
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
