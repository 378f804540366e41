"""Benchmark of the Kronecker-factored optimizer step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mlp4|...] [--impl reference]

One step = the whole hot path over one batch of synthetic inputs:
  K1  factor update (A and G, EMA) for every KRON layer
  K2+K3 damped inverses of every factor, on the steps the refresh cadence selects
  K4  precondition + fused momentum / weight-decay update for every KRON layer
  K5+K6 diagonal factors + fused diagonal step for every DIAG layer (for layer
        sets without DIAG layers, the diagonal twins of the KRON layers)
Inputs are resident in HBM when the timed region starts; L2 is flushed between
steps outside the per-step CUDA events.  Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as Wl  # noqa: E402

METRIC = "K-FAC precond steps/s; factor-GEMM TFLOP/s & diag-step GB/s vs GB300 peak"
WORKLOADS = {"mlp4": "c2", "single_linear": "c1", "resnet18": "c3", "resnet50": "c4",
             "resnet50_bf16": "c4bf16", "transformer4": "c5",
             "resnet18_nchw": "c3", "resnet50_nchw": "c4", "resnet50_bf16_nchw": "c4bf16",
             "transformer4_qkv_tied": "c5", "mlp4_ikfac": "c2",
             "resnet18_diag_nchw": "c3", "mlp4_ikfac_bf16": "c2",
             "transformer4_ikfac_bf16": "c5", "transformer1": "c5b1",
             "transformer4_bf16_precond": "c5", "mlp4_bf16_precond": "c2"}
# workloads whose convolutions hand the library their NCHW input and output
# gradient (kfac_update_factors_conv2d_batched) instead of unfolded matrices
NCHW_WORKLOADS = {"resnet18_nchw", "resnet50_nchw", "resnet50_bf16_nchw", "resnet18_diag_nchw"}
# workloads that put every layer on the diagonal path (AdaFisher-style, as the
# CAFIN page trains ResNet-18), convolutions fed as NCHW tensors
DIAG_WORKLOADS = {"resnet18_diag_nchw"}
# workloads whose key and value projections share the query projection's A
# factor (kfac_tie_a_factor: the three read the same input)
TIED_WORKLOADS = {"transformer4_qkv_tied"}
# workloads whose refreshes after the first are inverse-free steps
# (kfac_ikfac_update, beta = 1) instead of Cholesky inversions: products in 3xTF32,
# or on bf16 tensor cores
IKFAC_WORKLOADS = {"mlp4_ikfac", "mlp4_ikfac_bf16", "transformer4_ikfac_bf16"}
IKFAC_BF16_WORKLOADS = {"mlp4_ikfac_bf16", "transformer4_ikfac_bf16"}
# workloads whose preconditioning products run in bf16 (hp.math = KFAC_MATH_BF16)
BF16_PRECOND_WORKLOADS = {"transformer4_bf16_precond", "mlp4_bf16_precond"}


def qkv_ties(layers):
    """{tied layer index: source index}: b.k and b.v use b.q's A (KRON layers only)."""
    pos = {l.name: i for i, l in enumerate(layers) if l.kind == "kron"}
    ties = {}
    for name, i in pos.items():
        blk, _, proj = name.rpartition(".")
        if proj in ("k", "v") and f"{blk}.q" in pos:
            ties[i] = pos[f"{blk}.q"]
    return ties
# fallback roofline denominators when MEASURED_PEAKS.json is absent
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TF32_PER_BF16 = 1.1 / 2.25          # nominal dense ratio
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of each phase's
# launches in one step of the transformer workload: one ncu capture per phase of
#   python bench.py --workload transformer1 --steps 2 --warmup 1 --no-e2e \
#       --no-cpu-baseline --no-graphs --nvtx
# (ncu --nvtx --nvtx-include "<phase>/", the last step's launches) on the
# one-block set, times four: the four blocks are the same layers, batched into
# the same kinds of launches (ncu does not count writes that are still in L2
# when a kernel ends).  Valid only for the kernel sources with this digest: any
# change to them reports null until the counters are taken again.
MEASURED_TRAFFIC = {
    "workload": "transformer4",
    "sources_sha256": "b1caf7e8f7732ac757d2c11dd5ac8ff7d08c12d00c66c558b8ef3ae09d12a1c0",
    "bytes": {"factor": 4 * 5.0202e9, "precond": 4 * 6.0914e9, "diag": 4 * 2.1917e9},
    "note": "one-block capture (transformer1) x 4",
}


def sources_digest() -> str:
    import hashlib
    d = os.path.join(ROOT, "second_order_optimizer_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh")):
            h.update(f.encode())
            with open(os.path.join(d, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12   # FFMA lanes x 2 flop x max SM clock


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="transformer4", choices=sorted(WORKLOADS))
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graphs", action="store_true", help="time eager calls, not CUDA graphs")
    p.add_argument("--schedule", choices=["auto", "serial", "overlap"], default="auto",
                   help="serial: the phases of a step in order on one stream; overlap: the "
                        "diagonal step, and on steps without a refresh the factor update, on "
                        "side streams alongside the preconditioning; auto (default): the "
                        "faster of the two over one refresh period each, measured untimed "
                        "before the timed steps")
    p.add_argument("--nvtx", action="store_true",
                   help="NVTX ranges factor/invert/precond/diag around the phases of eager steps "
                        "(for profiler filters; use with --no-graphs)")
    # single-kernel mode: time one phase on one layer shape (not the headline line)
    p.add_argument("--micro", choices=["factor", "precond", "invert", "diag"], default=None)
    p.add_argument("--n", type=int, default=8193, help="micro: A dimension (d_in + 1)")
    p.add_argument("--o", type=int, default=2048, help="micro: G dimension (d_out)")
    p.add_argument("--rows", type=int, default=16384, help="micro: rows M")
    p.add_argument("--dtype", choices=["f32", "bf16"], default="bf16")
    p.add_argument("--reps", type=int, default=10)
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            out = {}
            for k in FALLBACK:
                v = d.get(k)
                if isinstance(v, dict):
                    v = v.get("value")
                out[k] = float(v) if v is not None else None
            if all(v is not None for v in out.values()):
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


def bench_config(workload):
    cfg = Wl.get_config(WORKLOADS[workload])
    layers = list(cfg.layers)
    if workload in DIAG_WORKLOADS:
        import dataclasses
        return cfg, [dataclasses.replace(l, kind="diag") for l in layers]
    if not cfg.diag_layers:
        import dataclasses
        layers += [dataclasses.replace(l, name=l.name + "_diag", kind="diag") for l in cfg.layers]
    return cfg, layers


def workload_name(cfg, workload):
    """The layer set's name with the bench variant's suffixes (both arms print it)."""
    return (cfg.name + ("+diag_twins" if not cfg.diag_layers else "")
            + ("+nchw_conv_inputs" if workload in NCHW_WORKLOADS else "")
            + ("+all_layers_diagonal" if workload in DIAG_WORKLOADS else "")
            + ("+qkv_shared_A" if workload in TIED_WORKLOADS else "")
            + ("+inverse_free_refresh" if workload in IKFAC_WORKLOADS else "")
            + ("_bf16" if workload in IKFAC_BF16_WORKLOADS else "")
            + ("+bf16_preconditioning" if workload in BF16_PRECOND_WORKLOADS else ""))


def path_dtype(layers, workload=None):
    """Arithmetic of the step: fp32 state, factors and preconditioning (fp32 operands
    on the tensor cores: 3xTF32 factor products, TF32 + bf16-correction
    preconditioning products); factor products read bf16 inputs where the layer
    set has them; the bf16 inverse-free variants refresh with bf16 products."""
    d = "bf16-in/f32" if any(l.in_dtype == "bf16" for l in layers) else "f32"
    return (d + ("+bf16-refresh" if workload in IKFAC_BF16_WORKLOADS else "")
            + ("+bf16-precond" if workload in BF16_PRECOND_WORKLOADS else ""))


# ----------------------------------------------------------------------------- accounting

def algorithmic(layers, k, nchw=False, tied=(), ikfac=False, ikfac_bf16=False):
    """Per-step algorithmic flops and bytes of each phase (fp32 state, input dtype as given).
    nchw: convolutions read their NCHW input and output gradient, not unfolded matrices.
    tied: indices of layers whose A is another layer's (no A product or inverse)."""
    f = {"factor_flop": 0.0, "factor_bytes": 0.0, "invert_flop": 0.0, "precond_flop": 0.0,
         "precond_bytes": 0.0, "diag_bytes": 0.0, "diagfac_bytes": 0.0}
    for li, l in enumerate(layers):
        elt = 2 if l.in_dtype == "bf16" else 4
        n, o, M = l.n, l.d_out, l.rows
        if l.kind == "kron":
            own_a = li not in tied
            # upper triangle only: M * n(n+1) flop (2 per FMA) per factor
            f["factor_flop"] += M * n * (n + 1) * own_a + M * o * (o + 1)
            if nchw and l.conv is not None:
                c = l.conv
                f["factor_bytes"] += (c.batch * c.c_in * c.h * c.w + M * o) * elt
            else:
                f["factor_bytes"] += M * (l.d_in * own_a + o) * elt
            f["factor_bytes"] += 2 * 4 * (n * n * own_a + o * o)
            # Cholesky n^3/3 + L^-1 n^3/3 + X^T X n^3/3; inverse-free: three n^3 products
            # (2 n^3 each) and K K^T (n^3, upper triangle); with bf16 products the first
            # one reads F_d as a hi/lo pair (a reduction of 2n: 4 n^3)
            per = 9 if ikfac_bf16 else 7 if ikfac else 1
            f["invert_flop"] += per * (n ** 3 * own_a + o ** 3) / k
            f["precond_flop"] += 2 * o * n * n + 2 * o * o * n
            f["precond_bytes"] += 4 * (n * n + o * o + 2 * o * n) + 4 * 3 * o * n
        else:
            f["diag_bytes"] += 20 * o * n + 8 * (o + n)
            if nchw and l.conv is not None:
                c = l.conv
                f["diagfac_bytes"] += (c.batch * c.c_in * c.h * c.w + M * o) * elt
            elif l.act != "bn":
                f["diagfac_bytes"] += M * (l.d_in + o) * elt
    return f


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        # the raw samples (the bench line carries their summary); KFAC_CLOCKS_DIR keeps them
        import tempfile
        d = os.environ.get("KFAC_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle

def blas_threads():
    """Threads the oracle's BLAS uses (NumPy's bundled OpenBLAS), else the affinity count."""
    import ctypes
    try:
        for line in open("/proc/self/maps"):
            if "openblas" in line and ".so" in line:
                lib = ctypes.CDLL(line.split()[-1])
                for fn in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                           "openblas_get_num_threads"):
                    if hasattr(lib, fn):
                        return int(getattr(lib, fn)())
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def oracle_steps_per_s(cfg, layers, budget_s=20.0, min_s=10.0, nchw=False, tied=False,
                       ikfac=False):
    """Time the float64 oracle as it stands on a bounded sample of the workload.

    Sample: one K-FAC step of as many KRON layers as fit the budget (factor
    build, precondition, update) plus one refresh (both damped inverses) of
    each of them; the diagonal path of the same layers.  Passes over the sampled
    layers repeat until at least ``min_s`` seconds of CPU work have been timed,
    and the per-layer times are averaged over the passes.  Per-layer times are
    scaled to the whole layer set, with the refresh amortised by the cadence.
    nchw: convolutions build their factors from NCHW draws through the oracle's
    input patches, as the GPU arm's NCHW workloads do.  tied: key and value
    projections use the query projection's A (no A of their own).  ikfac: the
    refresh is the oracle's inverse-free step instead of its inversion."""
    import oracle as O
    hp = cfg.hp
    orc = O.KfacOracle(hp.ema_decay, hp.damping, hp.lr, hp.momentum, hp.weight_decay, 1)
    kron = [l for l in layers if l.kind == "kron"]
    diag = [l for l in layers if l.kind == "diag"]
    tied_names = ({layers[i].name for i in qkv_ties(layers)} if tied else set())
    own_a = lambda l: l.name not in tied_names
    cost = lambda l: (l.rows * (l.n ** 2 * own_a(l) + l.d_out ** 2) + l.n ** 3 * own_a(l)
                      + l.d_out ** 3)
    t0 = time.perf_counter()
    inputs = {}

    def kron_once(l):
        if l.name not in inputs:
            li = cfg.layers.index(l) if l in cfg.layers else 0
            inputs[l.name] = Wl.layer_inputs(cfg, li, 1, rows=l.rows)
            if nchw and l.conv is not None:
                inputs[l.name].update(Wl.conv_inputs(cfg, li, 1))
        x = inputs[l.name]
        st = O.LayerState("kron", l.d_out, l.d_in, l.has_bias,
                          np.zeros((l.d_out, l.d_in)), np.zeros(l.d_out) if l.has_bias else None)
        ts = time.perf_counter()
        if "geom" in x:
            c = x["geom"]
            An, Gn = O.conv_factors(x["x"], x["gy"], (c.kh, c.kw), (c.sh, c.sw), (c.ph, c.pw),
                                    (c.dh, c.dw), l.has_bias)
        elif own_a(l):
            An, Gn = O.factor(x["a"], l.has_bias), O.factor(x["g"], 0)
        else:
            An, Gn = None, O.factor(x["g"], 0)
        if An is not None:
            st.A = O.ema(st.A, An, orc.xi)
        st.G = O.ema(st.G, Gn, orc.xi)
        tf = time.perf_counter()
        if ikfac:
            KA, KG = np.eye(l.n), np.eye(l.d_out)
            st.Ainv = O.ikfac_inverse(O.ikfac_update(KA, st.A, orc.gamma, 1.0)) if own_a(l) else KA
            st.Ginv = O.ikfac_inverse(O.ikfac_update(KG, st.G, orc.gamma, 1.0))
        else:
            st.Ainv = O.damped_inverse(st.A, orc.gamma) if own_a(l) else np.eye(l.n)
            st.Ginv = O.damped_inverse(st.G, orc.gamma)
        ti = time.perf_counter()
        P = O.precondition(st.Ginv, O.grad_hat(x["grad_w"], x["grad_b"]), st.Ainv)
        st.W, st.m = O.momentum_update(P, st.W, st.m, orc.lr, orc.mu, orc.wd)
        tp = time.perf_counter()
        return (tf - ts) + (tp - ti) + (ti - tf) / cfg.invert_every

    def diag_once(l):
        st = O.LayerState("diag", l.d_out, l.d_in, l.has_bias, np.zeros((l.d_out, l.d_in)),
                          np.zeros(l.d_out) if l.has_bias else None)
        gw = np.zeros((l.d_out, l.d_in))
        gn, an = np.ones(l.d_out), np.ones(l.n)
        li = cfg.layers.index(dataclasses.replace(l, kind="kron")) if l.conv is not None else -1
        ts = time.perf_counter()
        if nchw and l.conv is not None:     # the new diagonal factors from the NCHW tensors
            if l.name not in inputs:
                inputs[l.name] = Wl.conv_inputs(cfg, li, 1)
            c = inputs[l.name]["geom"]
            ts = time.perf_counter()
            gn, an = O.conv_diag_factors(inputs[l.name]["x"], inputs[l.name]["gy"], (c.kh, c.kw),
                                         (c.sh, c.sw), (c.ph, c.pw), (c.dh, c.dw), l.has_bias)
        orc.step_diag(st, gn, an, gw, np.zeros(l.d_out) if l.has_bias else None)
        return time.perf_counter() - ts

    # first pass: as many KRON layers (cheapest first) as fit the budget
    sums, sampled = {}, []
    for l in sorted(kron, key=cost):
        if time.perf_counter() - t0 > budget_s and sampled:
            break
        sums[l.name] = kron_once(l)
        sampled.append(l)
    dsample = diag[:4]
    dsum = sum(diag_once(l) for l in dsample)
    passes = 1
    # further passes over the same sample until enough CPU work has been timed
    while time.perf_counter() - t0 < min_s:
        for l in sampled:
            sums[l.name] += kron_once(l)
        dsum += sum(diag_once(l) for l in dsample)
        passes += 1
    # scale the sampled layers' time to the whole set by the flop-weighted cost
    scale = sum(cost(l) for l in kron) / max(1.0, sum(cost(l) for l in sampled))
    t_total = sum(sums.values()) / passes * scale
    if diag:
        t_total += dsum / passes * len(diag) / len(dsample)
    names = [l.name for l in sampled]
    sample = (f"oracle fp64 (NumPy: matrix products through NumPy's BLAS, Cholesky and "
              f"substitutions as column loops): factor+precond+update of {len(sampled)}/"
              f"{len(kron)} KRON layers ({', '.join(names[:4])}{'...' if len(names) > 4 else ''})"
              f" with one refresh amortised by {cfg.invert_every}, diag step of "
              f"{len(dsample)}/{len(diag)} DIAG layers, {passes} pass(es) averaged; "
              f"extrapolated to the full layer set by flop-weighted cost")
    return 1.0 / t_total, sample, time.perf_counter() - t0


# ----------------------------------------------------------------------------- GPU arm

def run_gpu(args, peaks, peak_kind):
    import torch
    import second_order_optimizer_gb300 as K

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg, layers = bench_config(args.workload)
    hp = cfg.hp
    k = cfg.invert_every
    kd = lambda l: K.KFAC_BF16 if l.in_dtype == "bf16" else K.KFAC_F32
    descs = [(K.KFAC_KRON if l.kind == "kron" else K.KFAC_DIAG, l.d_out, l.d_in, l.has_bias, kd(l))
             for l in layers]
    max_rows = max(l.rows for l in layers)
    ikfac = args.workload in IKFAC_WORKLOADS
    mode = (K.KFAC_IKFAC_BF16 if args.workload in IKFAC_BF16_WORKLOADS
            else K.KFAC_IKFAC_TF32 if ikfac else K.KFAC_IKFAC_OFF)
    # The inverse-free step K <- K(I - (beta/2)(K^T F_d K - I)) contracts only while
    # K^T F_d K stays near I: with the EMA starting from zero a factor grows about
    # 8x between the first refresh (the Cholesky seed) and the next, and beta = 1
    # steps then diverge (inverse error 0.6, 30, 1e11 at steps 11, 21, 31).  Those
    # variants start the EMA from the first factor, so that K follows the batch-to-
    # batch changes only.
    h = K.Kfac(descs, ema_decay=hp.ema_decay, damping=hp.damping, lr=hp.lr, momentum=hp.momentum,
               weight_decay=hp.weight_decay, max_rows=max_rows, device=dev, ikfac=mode,
               ema_init=K.KFAC_EMA_INIT_FIRST if ikfac else K.KFAC_EMA_INIT_ZERO,
               math=(K.KFAC_MATH_BF16 if args.workload in BF16_PRECOND_WORKLOADS
                     else K.KFAC_MATH_3XTF32))
    ties = qkv_ties(layers) if args.workload in TIED_WORKLOADS else {}
    for li, src in ties.items():
        h.tie_a_factor(li, src)
    # inputs: two seeded batches per layer, resident in HBM, used alternately
    base = {l.name.replace("_diag", ""): i for i, l in enumerate(cfg.layers)}
    srcidx = [base.get(l.name.replace("_diag", ""), i) for i, l in enumerate(layers)]
    NB = 2
    data = []
    nchw = args.workload in NCHW_WORKLOADS
    is_conv = lambda l: nchw and l.conv is not None
    for b in range(NB):
        per = []
        for li, l in enumerate(layers):
            x = Wl.layer_inputs_torch(cfg, srcidx[li], 1 + b, dev)
            if is_conv(l):      # NCHW input and output gradient replace the unfolded a, g
                del x["a"], x["g"]
                c = Wl.conv_inputs_torch(cfg, srcidx[li], 1 + b, dev)
                x["x"], x["gy"] = c["x"], c["gy"]
            per.append(x)
        data.append(per)
    # all parameters live in one flat device buffer (256-byte aligned views), so the
    # end-to-end leg reads every updated parameter back with one copy
    init = [Wl.initial_params_torch(cfg, srcidx[li], dev) for li in range(len(layers))]
    al = lambda n: (n + 63) // 64 * 64
    params_flat = torch.zeros(sum(al(w.numel()) + (al(bb.numel()) if bb is not None else 0)
                                  for w, bb in init), device=dev)
    params, off = [], 0
    for w, bb in init:
        pw = params_flat[off:off + w.numel()].view(w.shape)
        pw.copy_(w)
        off += al(w.numel())
        pb = None
        if bb is not None:
            pb = params_flat[off:off + bb.numel()]
            pb.copy_(bb)
            off += al(bb.numel())
        params.append((pw, pb))
    del init
    gnew = [torch.empty(l.d_out, device=dev) if l.kind == "diag" else None for l in layers]
    anew = [torch.empty(l.n, device=dev) if l.kind == "diag" else None for l in layers]
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    kron_idx = [li for li, l in enumerate(layers) if l.kind == "kron"]
    # batches share one input dtype
    kron_groups, conv_groups, geoms = {}, {}, {}
    for li in kron_idx:
        l = layers[li]
        if is_conv(l):
            c = l.conv
            geoms[li] = K.conv2d_geom((c.batch, c.c_in, c.h, c.w), (c.kh, c.kw), (c.sh, c.sw),
                                      (c.ph, c.pw), (c.dh, c.dw))
            conv_groups.setdefault(l.in_dtype, []).append(li)
        else:
            kron_groups.setdefault(l.in_dtype, []).append(li)

    def phase_factor(x):
        for grp in kron_groups.values():
            h.update_factors_batched(grp, [None if li in ties else x[li]["a"] for li in grp],
                                     [x[li]["g"] for li in grp])
        for grp in conv_groups.values():
            h.update_factors_conv2d_batched(grp, [x[li]["x"] for li in grp],
                                            [x[li]["gy"] for li in grp], [geoms[li] for li in grp])

    def phase_invert():
        h.invert(-1)

    # the refresh the timed steps replay: the first refresh (a warm-up step) is a
    # Cholesky inversion, which also seeds the inverse factors of an ikfac handle
    def phase_refresh():
        if ikfac:
            h.ikfac_update(-1, beta=1.0)
        else:
            h.invert(-1)

    def phase_precond(x):
        if kron_idx:
            h.precondition_batched(kron_idx, [x[li]["grad_w"] for li in kron_idx],
                                   [x[li]["grad_b"] for li in kron_idx], None, None,
                                   [params[li][0] for li in kron_idx],
                                   [params[li][1] for li in kron_idx])

    diag_idx = [li for li, l in enumerate(layers) if l.kind == "diag"]
    k5_groups = {}   # layers whose diagonal factors come from a and g, by input dtype
    conv_diag = []   # convolutions on the diagonal path, fed as NCHW tensors
    for li in diag_idx:
        if is_conv(layers[li]):
            conv_diag.append(li)
        elif layers[li].act != "bn":
            k5_groups.setdefault(layers[li].in_dtype, []).append(li)

    def phase_diag(x):
        for grp in k5_groups.values():
            h.diag_factors_batched(grp, [x[li]["a"] for li in grp], [x[li]["g"] for li in grp],
                                   [gnew[li] for li in grp], [anew[li] for li in grp])
        for li in conv_diag:
            c = layers[li].conv
            h.diag_factors_conv2d(li, x[li]["x"], x[li]["gy"], gnew[li], anew[li], (c.kh, c.kw),
                                  (c.sh, c.sw), (c.ph, c.pw), (c.dh, c.dw))
        if diag_idx:
            bn = lambda li: layers[li].act == "bn"
            h.diag_step_batched(
                diag_idx, [x[li]["g_new"] if bn(li) else gnew[li] for li in diag_idx],
                [x[li]["a_new"] if bn(li) else anew[li] for li in diag_idx],
                [x[li]["grad_w"] for li in diag_idx], [x[li]["grad_b"] for li in diag_idx],
                [params[li][0] for li in diag_idx], [params[li][1] for li in diag_idx])

    import contextlib
    rng = ((lambda name: torch.cuda.nvtx.range(name)) if args.nvtx
           else (lambda name: contextlib.nullcontext()))

    def step(t, x, ev=None):
        """The eager step through the public API (used for warm-up and end-to-end)."""
        if ev: ev[0].record(stream)
        with rng("factor"):
            phase_factor(x)
        if ev: ev[1].record(stream)
        if (t - 1) % k == 0:
            with rng("invert"):
                phase_invert() if t == 1 else phase_refresh()
        if ev: ev[2].record(stream)
        with rng("precond"):
            phase_precond(x)
        if ev: ev[3].record(stream)
        with rng("diag"):
            phase_diag(x)
        if ev: ev[4].record(stream)

    t = 0
    for _ in range(args.warmup):
        t += 1
        step(t, data[t % NB])
    torch.cuda.synchronize()
    code = h.get_status()[0]
    if code:
        raise RuntimeError(f"device status {code} after warm-up")

    # Each phase of each input batch is captured once into a CUDA graph; a timed step
    # replays the four phase graphs (the inverse refresh only on refresh steps), with
    # events on the replay stream between them.  Capture runs every library call once
    # (that work is discarded by the steps that follow: the state evolves as usual).
    graphs = {}
    kernels_in = {}
    if not args.no_graphs:
        for b in range(NB):
            for name, fn in (("factor", lambda b=b: phase_factor(data[b])),
                             ("precond", lambda b=b: phase_precond(data[b])),
                             ("diag", lambda b=b: phase_diag(data[b]))):
                g = torch.cuda.CUDAGraph()
                c0 = K.launch_count()
                with torch.cuda.graph(g):
                    fn()
                graphs[(name, b)] = g
                kernels_in[(name, b)] = K.launch_count() - c0
        g = torch.cuda.CUDAGraph()
        c0 = K.launch_count()
        with torch.cuda.graph(g):
            phase_refresh()
        graphs[("invert", 0)] = g
        kernels_in[("invert", 0)] = K.launch_count() - c0
        torch.cuda.synchronize()

    # On a step without a refresh the factor update is independent of the
    # preconditioning and the diagonal step (they read the last refresh's
    # inverses), and the library keeps their scratch apart: the factor graph
    # replays on a side stream alongside them.  Refresh steps run in order.
    side = torch.cuda.Stream(dev)
    ev_side = torch.cuda.Event()
    dside = torch.cuda.Stream(dev)
    ev_dside = torch.cuda.Event()

    def step_graph(t, b, ev, overlap):
        refresh = (t - 1) % k == 0
        ev[0].record(stream)
        if overlap:
            # the diagonal step touches only the DIAG layers: always alongside
            dside.wait_event(ev[0])
            with torch.cuda.stream(dside):
                graphs[("diag", b)].replay()
                ev_dside.record(dside)
            if refresh:
                graphs[("factor", b)].replay()
                ev[1].record(stream)
                graphs[("invert", 0)].replay()
                ev[2].record(stream)
                graphs[("precond", b)].replay()
            else:
                side.wait_event(ev[0])
                with torch.cuda.stream(side):
                    graphs[("factor", b)].replay()
                    ev_side.record(side)
                graphs[("precond", b)].replay()
                stream.wait_event(ev_side)
            stream.wait_event(ev_dside)
        else:
            graphs[("factor", b)].replay()
            ev[1].record(stream)
            if refresh:
                graphs[("invert", 0)].replay()
            ev[2].record(stream)
            graphs[("precond", b)].replay()
            ev[3].record(stream)
            graphs[("diag", b)].replay()
        ev[4].record(stream)
        return (kernels_in[("factor", b)] + kernels_in[("precond", b)] + kernels_in[("diag", b)]
                + (kernels_in[("invert", 0)] if refresh else 0))

    def calibrate():
        """Untimed: one refresh period of steps in each schedule; the faster wins."""
        nonlocal t
        cost = {}
        for ov in (False, True):
            e = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(k)]
            for i in range(k):
                t += 1
                flush.zero_()
                step_graph(t, t % NB, e[i], ov)
            torch.cuda.synchronize()
            cost[ov] = sum(e[i][0].elapsed_time(e[i][4]) for i in range(k))
        return cost[True] < cost[False], cost

    calibration = None
    if not graphs or args.schedule == "serial":
        overlap = False
    elif args.schedule == "overlap":
        overlap = True
    else:
        overlap, calibration = calibrate()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    torch.cuda.synchronize()
    sampler.start()
    l0 = K.launch_count()
    graph_launches = 0
    wall0 = time.perf_counter()
    refreshed = []
    for i in range(args.steps):
        t += 1
        refreshed.append((t - 1) % k == 0)
        flush.zero_()                         # L2 flush outside the step's events
        if graphs:
            graph_launches += step_graph(t, t % NB, evs[i], overlap)
        else:
            step(t, data[t % NB], evs[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    launches = K.launch_count() - l0 + graph_launches
    clocks = sampler.stop()
    code = h.get_status()[0]
    if code:
        raise RuntimeError(f"device status {code} in the timed region")
    ms_step = float(np.mean([evs[i][0].elapsed_time(evs[i][4]) for i in range(args.steps)]))
    refresh_steps = [i for i in range(args.steps) if refreshed[i]]
    inv_ms_refresh = (float(np.mean([evs[i][1].elapsed_time(evs[i][2]) for i in refresh_steps]))
                      if refresh_steps else 0.0)
    # per-phase breakdown: the phases of overlapped steps share the GPU, so they
    # are timed on a separate pass that runs them in order (not the headline)
    seq_steps = args.steps
    if overlap:
        seq_steps = min(args.steps, 100)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(seq_steps)]
        for i in range(seq_steps):
            t += 1
            flush.zero_()
            step_graph(t, t % NB, evs[i], False)
        torch.cuda.synchronize()
    ph = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(4)]
                   for i in range(seq_steps)])  # ms: factor, invert, precond, diag

    acc = algorithmic(layers, k, nchw, set(ties), ikfac, args.workload in IKFAC_BF16_WORKLOADS)
    phase_ms = ph.mean(axis=0)
    phase_ms[1] = inv_ms_refresh / k   # invert, amortised over the refresh period
    factor_tfs = acc["factor_flop"] / (phase_ms[0] * 1e-3) / 1e12
    diag_gbs = (acc["diag_bytes"] + acc["diagfac_bytes"]) / (phase_ms[3] * 1e-3) / 1e9 if phase_ms[3] > 0 else 0.0
    precond_tfs = acc["precond_flop"] / (phase_ms[2] * 1e-3) / 1e12
    phases = {"factor_ms": round(float(phase_ms[0]), 4), "invert_ms_per_step": round(float(phase_ms[1]), 4),
              "invert_ms_per_refresh": round(inv_ms_refresh, 4),
              "precond_ms": round(float(phase_ms[2]), 4), "diag_ms": round(float(phase_ms[3]), 4),
              "factor_tflops": round(factor_tfs, 3), "precond_tflops": round(precond_tfs, 3),
              "diag_gbs": round(diag_gbs, 1),
              "timed": (f"phases in order on one stream, {seq_steps} steps (the headline "
                        "runs them on three streams, see config.phase_overlap)"
                        if overlap else "the timed steps")}
    # dominant phase -> roofline
    names = ["factor", "invert", "precond", "diag"]
    dom = names[int(np.argmax(phase_ms))]
    tf32_peak = peaks["bf16_tflops"] * TF32_PER_BF16
    if dom == "diag":
        roof = {"bound": "hbm", "achieved": round(diag_gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "kernel": "diag_factor_grouped_kernel + diag_step_grouped_kernel"}
    elif dom in ("factor", "precond"):
        flop = acc["factor_flop"] if dom == "factor" else acc["precond_flop"]
        ms = phase_ms[0] if dom == "factor" else phase_ms[2]
        ach = flop / (ms * 1e-3) / 1e12
        # the products' own arithmetic sets the peak: bf16 operands (bf16 inputs in the
        # factor phase, bf16 preconditioning) against the bf16 peak, fp32 operands
        # against the TF32 peak (factor products: three TF32 MMAs per k step;
        # preconditioning: one TF32 MMA and one bf16 correction MMA of the same time)
        bf = (all(l.in_dtype == "bf16" for l in layers if l.kind == "kron") if dom == "factor"
              else args.workload in BF16_PRECOND_WORKLOADS)
        issue = 3 if dom == "factor" else 2
        arith = "bf16" if bf else "3xTF32" if dom == "factor" else "TF32+bf16-corrections"
        peak = peaks["bf16_tflops"] if bf else tf32_peak
        kern = (f"pack_grouped + gemm_tc_pair/persistent (tcgen05) with the SYRK epilogue ({arith})"
                if dom == "factor" else
                f"gradhat_pack_grouped + gemm_tc_pair/persistent (tcgen05) with the SPLIT epilogue, "
                f"then the PRECOND epilogue ({arith})")
        roof = {"bound": "tensor", "achieved": round(ach, 3), "peak": round(peak, 1),
                "unit": "TFLOP/s", "kernel": kern, "timed": "one batched library call (the phase)",
                "arithmetic": arith}
        if not bf:
            roof["issued_frac"] = round(issue * ach / tf32_peak, 4)
        roof["note"] = ("algorithmic flops (upper triangle for factors)"
                        + ("" if bf else f"; {arith} issues {issue}x TF32 MMA time"))
    else:
        ach = acc["invert_flop"] * k / (inv_ms_refresh * 1e-3) / 1e12
        roof = {"bound": "alu", "achieved": round(ach, 3), "peak": round(FP32_ALU_TFLOPS, 1),
                "unit": "TFLOP/s", "kernel": "chol_diag/chol_panel/chol_trailing/tri_level"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = None
    if (args.workload == MEASURED_TRAFFIC["workload"] and dom in MEASURED_TRAFFIC["bytes"]
            and sources_digest() == MEASURED_TRAFFIC["sources_sha256"]):
        roof["traffic"] = MEASURED_TRAFFIC["bytes"][dom]
        roof["traffic_note"] = ("DRAM bytes per step of the phase's launches (ncu, same sources; "
                                + MEASURED_TRAFFIC["note"] + ")")
        if dom == "precond":
            roof["algorithmic_bytes"] = acc.get("precond_bytes")
    roof["phase"] = dom
    roof["peak_source"] = {
        "hbm": f"{peak_kind} HBM copy bandwidth",
        "tensor": (f"{peak_kind} bf16 dense (burst)" if roof.get("arithmetic") == "bf16" else
                   f"{peak_kind} bf16 dense (burst) x 1.1/2.25 (nominal TF32:bf16 ratio)"),
        "alu": "derived: 152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz"}[roof["bound"]]

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, layers, data[0], params_flat, srcidx, t, dev,
                      (phase_factor, phase_refresh, phase_precond, phase_diag), k, overlap,
                      graphs.get(("invert", 0)))
    return {
        "ms_per_step": ms_step, "phases": phases, "roofline": roof, "clocks": clocks,
        "gpu_launches": int(launches), "wall_s": wall, "e2e": e2e,
        "dtype": path_dtype(layers, args.workload),
        "config": {"workload": workload_name(cfg, args.workload),
                   "kron_layers": sum(l.kind == "kron" for l in layers),
                   "diag_layers": sum(l.kind == "diag" for l in layers),
                   "invert_every": k, "max_rows": max_rows,
                   "cuda_graphs": not args.no_graphs,
                   "phase_overlap": ("three streams: the diagonal step (DIAG layers) alongside "
                                     "the KRON path every step; the factor update alongside "
                                     "preconditioning on steps without a refresh"
                                     if overlap else
                                     "none: the phases of a step in order on one stream"),
                   "schedule": args.schedule + (
                       "" if calibration is None else
                       " (untimed calibration over {} steps each: serial {:.2f} ms, "
                       "overlap {:.2f} ms)".format(k, calibration[False], calibration[True])),
                   "l2": "flushed between steps (256 MiB write, outside the per-step events)"},
    }


def run_e2e(args, layers, x_dev, params_flat, srcidx, t, dev, phases, k, overlap,
            invert_graph=None):
    """Same step through the public API from pinned host memory: every step copies its
    inputs host -> device and reads its result back, inside the timed region.  The
    inputs of all layers are one packed pinned buffer (a diagonal twin shares its
    layer's tensors, so they are copied once), copied into a ring of E2E_BUFFERS
    device staging buffers on a copy stream that runs up to E2E_BUFFERS - 1 steps
    ahead of the compute (a data loader's prefetch): the copy engine keeps
    streaming through a refresh step, which computes longer than a copy takes.  A
    buffer is refilled only after the step that read it has finished.  The step's
    result is a metric of the updated parameters, the sum of all of them (every
    updated value enters it; the parameters themselves stay on the device, as in
    training), reduced on the device in fp32 and read back (D2H, 4 bytes) on a
    second copy stream.  On steps without a refresh the factor update runs on a
    side stream alongside the preconditioning and the diagonal step (as in the
    timed steps).  With CUDA graphs (the default) the library calls of each phase
    are captured once per staging buffer and replayed, as the timed steps do;
    --no-graphs makes them eagerly every step.  Two untimed steps per staging
    buffer come first, as a pass of their own (in a fresh process the first passes
    of the copy engines over the newly pinned buffer ran at about half speed); the
    timed pass starts from an idle GPU, so every copy of a timed step is inside
    the timed region."""
    phase_factor, phase_invert, phase_precond, phase_diag = phases
    import torch
    first = {}
    for li in range(len(layers)):
        first.setdefault(srcidx[li], li)
    entries, off = [], 0
    for li in sorted(first.values()):
        for key, v in x_dev[li].items():
            if v is None:
                continue
            nb = v.numel() * v.element_size()
            entries.append((li, key, off, v))
            off += (nb + 255) // 256 * 256
    total = off
    host, host_release = pinned_host_buffer(total)
    for li, key, o, v in entries:
        nb = v.numel() * v.element_size()
        host[o:o + nb].copy_(v.contiguous().view(-1).view(torch.uint8).cpu())
    nbuf = E2E_BUFFERS
    stage = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(nbuf)]

    def views(buf):
        per_src = {}
        for li, key, o, v in entries:
            nb = v.numel() * v.element_size()
            per_src.setdefault(li, {k2: None for k2 in x_dev[li]})[key] = \
                stage[buf][o:o + nb].view(v.dtype).view(v.shape)
        return [per_src[first[srcidx[li]]] for li in range(len(layers))]

    xs = [views(bb) for bb in range(nbuf)]
    if invert_graph is not None:      # capture each phase on each staging buffer
        import second_order_optimizer_gb300 as K  # noqa: F401
        torch.cuda.synchronize()
        gph = {}
        for bb in range(nbuf):
            for name, fn in (("factor", phase_factor), ("precond", phase_precond),
                             ("diag", phase_diag)):
                gg = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gg):
                    fn(xs[bb])
                gph[(name, bb)] = gg
        torch.cuda.synchronize()
        run = lambda name, bb: gph[(name, bb)].replay()
        run_invert = invert_graph.replay
    else:
        run = lambda name, bb: {"factor": phase_factor, "precond": phase_precond,
                                "diag": phase_diag}[name](xs[bb])
        run_invert = phase_invert
    steps = steps_cap(args)
    warm = 2 * E2E_BUFFERS   # untimed steps: the first DMA passes over a fresh buffer are slow
    outs = torch.empty(warm + steps, dtype=torch.float32, pin_memory=True)
    metric = torch.empty(warm + steps, dtype=torch.float32, device=dev)
    main = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    copy_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_used = [torch.cuda.Event() for _ in range(nbuf)]
    ev_done = torch.cuda.Event()
    fside = torch.cuda.Stream(dev)
    dside = torch.cuda.Stream(dev)
    ev_djoin = torch.cuda.Event()
    ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()
    tt = [t]

    def issue_copy(j):
        """Inputs of step j of a pass into buffer j % nbuf, once step j - nbuf (the
        last reader of that buffer, already issued) has finished."""
        bb = j % nbuf
        with torch.cuda.stream(copy):
            if j >= nbuf:
                copy.wait_event(ev_used[bb])
            stage[bb].copy_(host, non_blocking=True)
            ev_in[bb].record(copy)

    def one_pass(count, base):
        for j in range(min(nbuf, count)):
            issue_copy(j)
        for j in range(count):
            tt[0] += 1
            t_ = tt[0]
            b = j % nbuf
            main.wait_event(ev_in[b])
            if overlap:                             # diagonal step alongside the KRON path
                ev_fork.record(main)
                dside.wait_event(ev_fork)
                with torch.cuda.stream(dside):
                    run("diag", b)
                    ev_djoin.record(dside)
            if overlap and (t_ - 1) % k != 0:      # factor update alongside the rest
                ev_fork.record(main)
                fside.wait_event(ev_fork)
                with torch.cuda.stream(fside):
                    run("factor", b)
                    ev_join.record(fside)
            else:
                run("factor", b)
                if (t_ - 1) % k == 0:
                    run_invert()
            run("precond", b)
            if not overlap:
                run("diag", b)
            if overlap and (t_ - 1) % k != 0:
                main.wait_event(ev_join)
            if overlap:
                main.wait_event(ev_djoin)
            ev_used[b].record(main)
            if j + nbuf < count:                    # refill this buffer for step j + nbuf
                issue_copy(j + nbuf)
            i = base + j
            torch.sum(params_flat, dim=0, out=metric[i])   # the step's result
            ev_done.record(main)
            with torch.cuda.stream(copy_out):      # device -> host on its own stream
                copy_out.wait_event(ev_done)
                outs[i:i + 1].copy_(metric[i:i + 1], non_blocking=True)

    torch.cuda.synchronize()
    one_pass(warm, 0)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    one_pass(steps, warm)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    host_release()
    finite = all(math.isfinite(v) for v in outs.tolist())
    if not finite:
        print("bench.py: the end-to-end steps' parameter sums are not finite (the "
              "trajectory diverged)", file=sys.stderr, flush=True)
    return {"value": round(1.0 / dt, 3), "unit": "steps/s", "h2d_bytes_per_step": int(total),
            "d2h_bytes_per_step": 4, "steps": steps, "warmup": warm,
            "result": "sum of all updated parameters (fp32, reduced on the device)",
            "result_finite": finite,
            "pipelined": (f"H2D of each step's inputs on a copy stream into a ring of {nbuf} "
                          "device buffers, up to {} steps ahead of the compute; the result's "
                          "D2H on a second copy stream").format(nbuf - 1)}


def pinned_host_buffer(nbytes):
    """Page-locked host buffer for the end-to-end inputs and a function that
    releases it: an anonymous mapping with transparent huge pages requested,
    touched and registered with CUDA.  Host-to-device copies from a buffer of the
    CUDA host allocator fell to 77-97 GB/s on a box after a long GPU test run
    (the pages it got were small and scattered), where this one kept 209 GB/s.
    Falls back to the allocator when the registration is refused."""
    import ctypes
    import mmap
    import torch
    try:
        cudart = torch.cuda.cudart()
        buf = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        try:
            buf.madvise(mmap.MADV_HUGEPAGE)
        except (AttributeError, OSError):
            pass
        addr = ctypes.addressof(ctypes.c_char.from_buffer(buf))
        ctypes.memset(addr, 0, nbytes)           # fault every page in now
        if int(cudart.cudaHostRegister(addr, nbytes, 0)) != 0:
            raise RuntimeError("cudaHostRegister refused")
    except Exception:
        return torch.empty(nbytes, dtype=torch.uint8, pin_memory=True), lambda: None
    t = torch.frombuffer(buf, dtype=torch.uint8)

    def release():
        torch.cuda.synchronize()
        cudart.cudaHostUnregister(addr)

    release.keep = buf   # the mapping lives as long as the tensor's user holds this
    return t, release


# staging buffers of the end-to-end leg (5.64 GB each on the transformer set)
E2E_BUFFERS = 4


def steps_cap(args):
    """Steps of the end-to-end leg: the timed step count, within [3, 50]."""
    return max(3, min(args.steps, 50))


# ----------------------------------------------------------------------------- micro

def run_micro(args, peaks, peak_kind):
    """Time one phase on one layer shape with CUDA events (L2 flushed between reps)."""
    import torch
    import second_order_optimizer_gb300 as K
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n, o, M = args.n, args.o, args.rows
    d_in = n - 1
    kd = K.KFAC_BF16 if args.dtype == "bf16" else K.KFAC_F32
    tdt = torch.bfloat16 if args.dtype == "bf16" else torch.float32
    kind = K.KFAC_DIAG if args.micro == "diag" else K.KFAC_KRON
    h = K.Kfac([(kind, o, d_in, 1, kd)], max_rows=M, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1)
    a = torch.randn(M, d_in, generator=gen, device=dev).clamp_(min=0).to(tdt)
    g = (torch.randn(M, o, generator=gen, device=dev) * 1e-4).to(tdt)
    gw = torch.randn(o, d_in, generator=gen, device=dev) * 1e-6
    gb = torch.randn(o, generator=gen, device=dev) * 1e-6
    pw = torch.randn(o, d_in, generator=gen, device=dev) * 0.01
    pb = torch.zeros(o, device=dev)
    gn = torch.rand(o, generator=gen, device=dev) * 1e-8
    an = torch.rand(n, generator=gen, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    if kind == K.KFAC_KRON:
        h.update_factors(0, a, g)
        h.invert(0)

    def once():
        if args.micro == "factor":
            h.update_factors(0, a, g)
        elif args.micro == "invert":
            h.invert(0)
        elif args.micro == "precond":
            h.precondition(0, gw, gb, None, None, pw, pb)
        else:
            h.diag_step(0, gn, an, gw, gb, pw, pb)

    for _ in range(3):
        once()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        once()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    code = h.get_status()[0]
    ms = float(np.median(ts))
    elt = 2 if args.dtype == "bf16" else 4
    tf32_peak = peaks["bf16_tflops"] * TF32_PER_BF16
    if args.micro == "factor":
        flop = M * n * (n + 1) + M * o * (o + 1)
        peak = peaks["bf16_tflops"] if args.dtype == "bf16" else tf32_peak
        res = {"tflops": flop / ms / 1e9, "peak_tflops": peak, "frac": flop / ms / 1e9 / peak,
               "bytes_in": M * (d_in + o) * elt}
    elif args.micro == "precond":
        flop = 2 * o * n * n + 2 * o * o * n
        res = {"tflops": flop / ms / 1e9, "peak_tflops": tf32_peak,
               "frac": flop / ms / 1e9 / tf32_peak}
    elif args.micro == "invert":
        flop = n ** 3 + o ** 3
        res = {"tflops": flop / ms / 1e9}
    else:
        byts = 20 * o * n + 8 * (o + n)
        res = {"gbs": byts / ms / 1e6, "peak_gbs": peaks["hbm_gbs"],
               "frac": byts / ms / 1e6 / peaks["hbm_gbs"]}
    out = {"micro": args.micro, "n": n, "o": o, "rows": M, "dtype": args.dtype, "ms": round(ms, 4),
           "status": code, "peaks": peak_kind, **{k: round(v, 4) for k, v in res.items()}}
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------------------------- main

def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    peaks, peak_kind = load_peaks()
    if args.micro:
        run_micro(args, peaks, peak_kind)
        return
    cfg, layers = bench_config(args.workload)

    if args.impl == "reference":
        if rank != 0:      # under torchrun: rank 0 alone times the oracle
            return
        per_step = []
        sample = None
        for _ in range(args.warmup):
            pass  # the oracle has nothing to warm up
        t0 = time.perf_counter()
        for _ in range(max(1, args.steps)):
            v, sample, _ = oracle_steps_per_s(cfg, layers, budget_s=max(2.0, 60.0 / max(1, args.steps)),
                                              min_s=0.0, nchw=args.workload in NCHW_WORKLOADS,
                                              tied=args.workload in TIED_WORKLOADS,
                                              ikfac=args.workload in IKFAC_WORKLOADS)
            per_step.append(1.0 / v)
            if time.perf_counter() - t0 > 150:
                break
        value = 1.0 / statistics.median(per_step)
        cores = blas_threads()
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "steps/s",
                "n_gpus": args.gpus, "steps": len(per_step), "warmup": args.warmup,
                "ms_per_step": round(1e3 / value, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": workload_name(cfg, args.workload),
                           "invert_every": cfg.invert_every},
                "cpu_baseline": {"value": round(value, 6), "unit": "steps/s", "cores": cores,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": round(value, 6), "unit": "steps/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if world > 1 or args.gpus != 1:
        # The library is single-GPU: each process drives one GPU and its GEMM engine
        # may pair CTAs that share tiles by TMA multicast, which stays within one
        # process on one GPU.  There is no multi-rank mode.
        print(f"bench.py: the GPU arm runs on one GPU only (WORLD_SIZE={world}, "
              f"--gpus {args.gpus}); run it without torchrun and with --gpus 1",
              file=sys.stderr, flush=True)
        sys.exit(2)
    res = run_gpu(args, peaks, peak_kind)
    cpu = None
    if not args.no_cpu_baseline:
        v, sample, spent = oracle_steps_per_s(cfg, layers, budget_s=20.0,
                                              nchw=args.workload in NCHW_WORKLOADS,
                                              tied=args.workload in TIED_WORKLOADS,
                                              ikfac=args.workload in IKFAC_WORKLOADS)
        cpu = {"value": round(v, 6), "unit": "steps/s", "cores": blas_threads(), "kind": "oracle",
               "sample": sample, "seconds": round(spent, 1)}
    value = 1e3 / res["ms_per_step"]
    line = {"metric": METRIC, "value": round(value, 3), "unit": "steps/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(res["ms_per_step"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": res["dtype"],
            "data": "synthetic", "config": res["config"], "phases": res["phases"],
            "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": res["e2e"],
            "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
            "peaks": {"source": peak_kind, **peaks}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
