"""Seeded synthetic inputs for the Kronecker-factored optimizer step.

This module holds only layer shapes and random draws.  It contains none of the
optimizer's arithmetic, so the float64 oracle and the CUDA path can both read
the inputs it makes without sharing any of the method.

The five layer sets mirror the workloads the K-FAC / AdaFisher pages train on
(Osawa et al., "Large-Scale Distributed Second-Order Optimization Using K-FAC
...", §5.1: ResNet-50 on ImageNet, 32 images per GPU; the CAFIN briefing,
"Empirical Highlights": ResNet-18 on CIFAR-10/100).  No dataset is read: the
activations and output gradients are drawn from the distributions below, with
the shapes those networks produce.

Seeds: one NumPy PCG64 stream per (config, layer, step), seed =
1_000_000*config + 1_000*layer + step; step 0 draws the initial parameters.
Large configs draw on the GPU with a seeded ``torch.Generator`` instead (same
seed formula); that is input generation only.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class ConvGeom:
    """Geometry of a 2-D convolution over NCHW input [batch, c_in, h, w]."""
    batch: int
    c_in: int
    h: int
    w: int
    kh: int
    kw: int
    sh: int = 1
    sw: int = 1
    ph: int = 0
    pw: int = 0
    dh: int = 1
    dw: int = 1

    @property
    def h_out(self) -> int:
        return (self.h + 2 * self.ph - self.dh * (self.kh - 1) - 1) // self.sh + 1

    @property
    def w_out(self) -> int:
        return (self.w + 2 * self.pw - self.dw * (self.kw - 1) - 1) // self.sw + 1

    def with_batch(self, batch: int) -> "ConvGeom":
        return dataclasses.replace(self, batch=batch)


@dataclasses.dataclass(frozen=True)
class Layer:
    name: str
    kind: str            # "kron" (full Kronecker factors) or "diag" (diagonal Fisher)
    d_out: int           # o: G dimension / output channels
    d_in: int            # input width (conv: C_in*kh*kw)
    has_bias: int        # 1: a ones column is appended, A is (d_in+1)^2
    rows: int            # M: batch, or B*H_out*W_out for conv, or tokens
    act: str = "normal"  # "normal": a~N(0,1); "relu": max(N(0,1),0); "bn": BatchNorm layer
    in_dtype: str = "f32"  # "f32" or "bf16" for a and g
    conv: Optional[ConvGeom] = None  # set for convolutions: rows = batch*h_out*w_out

    @property
    def n(self) -> int:
        return self.d_in + self.has_bias

    @property
    def params(self) -> int:
        return self.d_out * self.n


@dataclasses.dataclass(frozen=True)
class HParams:
    ema_decay: float = 0.95
    damping: float = 1e-3
    lr: float = 1e-2
    momentum: float = 0.9
    weight_decay: float = 5e-4


@dataclasses.dataclass(frozen=True)
class Config:
    index: int           # 1..5, used in seeds
    name: str
    layers: List[Layer]
    steps: int
    invert_every: int
    g_std: float
    grad_mode: str       # "computed": dW = g^T [a 1] / M ; "iid": dW ~ N(0, sigma^2)
    hp: HParams = HParams()

    @property
    def kron_layers(self):
        return [l for l in self.layers if l.kind == "kron"]

    @property
    def diag_layers(self):
        return [l for l in self.layers if l.kind == "diag"]


def _conv(name, cin, cout, k, rows, act="relu", dt="f32", geom=None):
    if geom is not None:
        assert geom.batch * geom.h_out * geom.w_out == rows and geom.c_in == cin
    return Layer(name, "kron", cout, cin * k * k, 1, rows, act, dt, geom)


def _bn(name, c, rows):
    return Layer(name, "diag", c, 1, 1, rows, "bn")


def single_linear() -> Config:
    """One linear layer 64 -> 32 (+bias), batch 128, run on both paths."""
    kron = Layer("fc", "kron", 32, 64, 1, 128, "normal")
    diag = Layer("fc_diag", "diag", 32, 64, 1, 128, "normal")
    return Config(1, "single_linear_64x32_b128", [kron, diag], steps=10,
                  invert_every=1, g_std=1e-3, grad_mode="computed")


def mlp4() -> Config:
    """4-layer MLP 1024->1024->1024->1024->10, batch 1024."""
    L = [Layer("fc1", "kron", 1024, 1024, 1, 1024, "normal"),
         Layer("fc2", "kron", 1024, 1024, 1, 1024, "relu"),
         Layer("fc3", "kron", 1024, 1024, 1, 1024, "relu"),
         Layer("fc4", "kron", 10, 1024, 1, 1024, "relu")]
    return Config(2, "mlp4_1024_b1024", L, steps=100, invert_every=10,
                  g_std=1e-4, grad_mode="computed")


def resnet18_cifar() -> Config:
    """ResNet-18 (CIFAR stem) on 32x32 input, batch 128: 21 conv/fc layers + 20 BN."""
    B = 128
    L: List[Layer] = []
    L.append(_conv("conv1", 3, 64, 3, B * 32 * 32, geom=ConvGeom(B, 3, 32, 32, 3, 3, 1, 1, 1, 1)))
    L.append(_bn("bn1", 64, B * 32 * 32))
    cin, hw = 64, 32
    for stage, (c, stride) in enumerate([(64, 1), (128, 2), (256, 2), (512, 2)], 1):
        for blk in range(2):
            s = stride if blk == 0 else 1
            hw_out = hw // s
            rows = B * hw_out * hw_out
            L.append(_conv(f"l{stage}.{blk}.conv1", cin, c, 3, rows,
                           geom=ConvGeom(B, cin, hw, hw, 3, 3, s, s, 1, 1)))
            L.append(_bn(f"l{stage}.{blk}.bn1", c, rows))
            L.append(_conv(f"l{stage}.{blk}.conv2", c, c, 3, rows,
                           geom=ConvGeom(B, c, hw_out, hw_out, 3, 3, 1, 1, 1, 1)))
            L.append(_bn(f"l{stage}.{blk}.bn2", c, rows))
            if blk == 0 and (s != 1 or cin != c):
                L.append(_conv(f"l{stage}.{blk}.short", cin, c, 1, rows,
                               geom=ConvGeom(B, cin, hw, hw, 1, 1, s, s, 0, 0)))
                L.append(_bn(f"l{stage}.{blk}.short_bn", c, rows))
            cin, hw = c, hw_out
    L.append(Layer("fc", "kron", 100, 512, 1, B, "relu"))
    return Config(3, "resnet18_cifar_b128", L, steps=20, invert_every=20,
                  g_std=1e-4, grad_mode="iid")


def resnet50_imagenet(dtype: str = "f32") -> Config:
    """ResNet-50 (v1.5: stride in the 3x3) on 224x224 input, batch 32: 54 + 53 BN."""
    B = 32
    L: List[Layer] = []
    L.append(_conv("conv1", 3, 64, 7, B * 112 * 112, "normal", dtype,
                   ConvGeom(B, 3, 224, 224, 7, 7, 2, 2, 3, 3)))
    L.append(_bn("bn1", 64, B * 112 * 112))
    cin, hw = 64, 56
    for stage, (w, nblk, stride) in enumerate([(64, 3, 1), (128, 4, 2), (256, 6, 2), (512, 3, 2)], 1):
        out = 4 * w
        for blk in range(nblk):
            s = stride if blk == 0 else 1
            hw_out = hw // s
            r_in, r_out = B * hw * hw, B * hw_out * hw_out
            p = f"l{stage}.{blk}"
            L.append(_conv(p + ".conv1", cin, w, 1, r_in, dt=dtype,
                           geom=ConvGeom(B, cin, hw, hw, 1, 1)))
            L.append(_bn(p + ".bn1", w, r_in))
            L.append(_conv(p + ".conv2", w, w, 3, r_out, dt=dtype,
                           geom=ConvGeom(B, w, hw, hw, 3, 3, s, s, 1, 1)))
            L.append(_bn(p + ".bn2", w, r_out))
            L.append(_conv(p + ".conv3", w, out, 1, r_out, dt=dtype,
                           geom=ConvGeom(B, w, hw_out, hw_out, 1, 1)))
            L.append(_bn(p + ".bn3", out, r_out))
            if blk == 0:
                L.append(_conv(p + ".down", cin, out, 1, r_out, dt=dtype,
                               geom=ConvGeom(B, cin, hw, hw, 1, 1, s, s, 0, 0)))
                L.append(_bn(p + ".down_bn", out, r_out))
            cin, hw = out, hw_out
    L.append(Layer("fc", "kron", 1000, 2048, 1, B, "relu", dtype))
    return Config(4, f"resnet50_imagenet_b32_{dtype}", L, steps=50, invert_every=50,
                  g_std=1e-4, grad_mode="iid")


def transformer4(blocks: int = 4) -> Config:
    """4 transformer blocks, d_model 2048, FFN 8192, 16384 tokens, bf16 a and g.

    Each block: Q, K, V, O projections (2048 -> 2048), FFN up (2048 -> 8192) and
    down (8192 -> 2048); all with bias.  The diagonal-path twins cover the same
    201.4M parameters.  ``blocks`` < 4: the first blocks alone (same layers and
    draws), a small case of the same products for profiler captures.
    """
    T = 16384
    L: List[Layer] = []
    for b in range(blocks):
        for nm in ("q", "k", "v", "o"):
            L.append(Layer(f"b{b}.{nm}", "kron", 2048, 2048, 1, T, "normal", "bf16"))
        L.append(Layer(f"b{b}.up", "kron", 8192, 2048, 1, T, "normal", "bf16"))
        L.append(Layer(f"b{b}.down", "kron", 2048, 8192, 1, T, "normal", "bf16"))
    L += [dataclasses.replace(l, name=l.name + "_diag", kind="diag") for l in list(L)]
    name = "transformer4_d2048_ffn8192_t16384" if blocks == 4 else f"transformer{blocks}_block"
    return Config(5, name, L, steps=10, invert_every=10, g_std=1e-5, grad_mode="iid")


CONFIGS = {
    "c1": single_linear,
    "c2": mlp4,
    "c3": resnet18_cifar,
    "c4": resnet50_imagenet,
    "c4bf16": lambda: resnet50_imagenet("bf16"),
    "c5": transformer4,
    "c5b1": lambda: transformer4(1),
}


def get_config(name: str) -> Config:
    return CONFIGS[name]()


def seed_for(cfg_index: int, layer_index: int, step: int) -> int:
    return 1_000_000 * cfg_index + 1_000 * layer_index + step


# ----------------------------------------------------------------------------
# rounding helpers (input dtype only)

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even to bfloat16, returned as float32 holding bf16 values."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def round_input(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16(x)
    return np.asarray(x, dtype=np.float32)


# ----------------------------------------------------------------------------
# NumPy draws (small and medium sizes; shared by the oracle's tests and the GPU tests)

def _act(rng, shape, act):
    z = rng.standard_normal(shape)
    if act == "relu":
        z = np.maximum(z, 0.0)
    return z


def mean_sq_act(act: str) -> float:
    """E[a^2] of the activation distribution (1 for N(0,1), 1/2 after ReLU)."""
    return 0.5 if act == "relu" else 1.0


def initial_params(cfg: Config, li: int):
    """W0 ~ N(0, 1/d_in), b0 ~ N(0, 1/d_in) (fp32)."""
    L = cfg.layers[li]
    rng = np.random.Generator(np.random.PCG64(seed_for(cfg.index, li, 0)))
    std = 1.0 / math.sqrt(L.d_in)
    w = (rng.standard_normal((L.d_out, L.d_in)) * std).astype(np.float32)
    b = (rng.standard_normal(L.d_out) * std).astype(np.float32) if L.has_bias else None
    return w, b


def layer_inputs(cfg: Config, li: int, step: int, rows: Optional[int] = None):
    """Activations a [M, d_in], output grads g [M, o], weight grads for one step.

    Returns a dict of float32 arrays (bf16 inputs are stored as float32 holding
    bf16-representable values).  For BatchNorm layers ("bn") the diagonal
    factor inputs g_new [o] and a_new [n] are drawn directly instead of a, g.
    ``rows`` overrides M (used to make small test cases).
    """
    L = cfg.layers[li]
    M = L.rows if rows is None else rows
    rng = np.random.Generator(np.random.PCG64(seed_for(cfg.index, li, step)))
    out = {}
    if L.act == "bn":
        # per-channel mean of g^2 over M positions, g ~ N(0, g_std^2); x_hat^2 mean ~ 1
        chi = 1.0 + rng.standard_normal(L.d_out) * math.sqrt(2.0 / M)
        out["g_new"] = (np.abs(chi) * cfg.g_std ** 2).astype(np.float32)
        xh = 1.0 + rng.standard_normal(1) * math.sqrt(2.0 / M)
        out["a_new"] = np.array([abs(xh[0]), 1.0], dtype=np.float32)
        sig = cfg.g_std * math.sqrt(1.0 / M)
        out["grad_w"] = (rng.standard_normal((L.d_out, 1)) * sig).astype(np.float32)
        out["grad_b"] = (rng.standard_normal(L.d_out) * sig).astype(np.float32)
        return out
    a = round_input(_act(rng, (M, L.d_in), L.act), L.in_dtype)
    g = round_input(rng.standard_normal((M, L.d_out)) * cfg.g_std, L.in_dtype)
    out["a"], out["g"] = a, g
    if cfg.grad_mode == "computed":
        a64, g64 = a.astype(np.float64), g.astype(np.float64)
        out["grad_w"] = (g64.T @ a64 / M).astype(np.float32)
        out["grad_b"] = (g64.sum(axis=0) / M).astype(np.float32) if L.has_bias else None
    else:
        sig = cfg.g_std * math.sqrt(mean_sq_act(L.act) / M)
        out["grad_w"] = (rng.standard_normal((L.d_out, L.d_in)) * sig).astype(np.float32)
        out["grad_b"] = ((rng.standard_normal(L.d_out) * sig).astype(np.float32)
                         if L.has_bias else None)
    return out


def conv_seed(cfg_index: int, layer_index: int, step: int) -> int:
    """Seed of a convolution's NCHW draws (odd, so it never equals a seed_for value)."""
    return 2 * seed_for(cfg_index, layer_index, step) + 1


def conv_inputs(cfg: Config, li: int, step: int, batch: Optional[int] = None):
    """NCHW input x [B, C, H, W] and output gradient gy [B, o, Ho, Wo] of a
    convolution layer (float32 holding values of the layer's input dtype):
    x from the layer's activation distribution, gy ~ N(0, g_std^2).  ``batch``
    overrides B (small test cases)."""
    L = cfg.layers[li]
    cg = L.conv if batch is None else L.conv.with_batch(batch)
    rng = np.random.Generator(np.random.PCG64(conv_seed(cfg.index, li, step)))
    x = round_input(_act(rng, (cg.batch, cg.c_in, cg.h, cg.w), L.act), L.in_dtype)
    gy = round_input(rng.standard_normal((cg.batch, L.d_out, cg.h_out, cg.w_out)) * cfg.g_std,
                     L.in_dtype)
    return {"x": x, "gy": gy, "geom": cg}


# ----------------------------------------------------------------------------
# Device draws for the large configs (torch is imported lazily)

def layer_inputs_torch(cfg: Config, li: int, step: int, device, rows: Optional[int] = None):
    """Same distributions as :func:`layer_inputs`, drawn on ``device`` with a seeded
    torch.Generator.  Returns torch tensors: a, g in the layer's input dtype
    (float32 or bfloat16), grad_w/grad_b float32 (iid form), or g_new/a_new for BN."""
    import torch
    L = cfg.layers[li]
    M = L.rows if rows is None else rows
    gen = torch.Generator(device=device)
    gen.manual_seed(seed_for(cfg.index, li, step))
    tdt = torch.bfloat16 if L.in_dtype == "bf16" else torch.float32
    out = {}
    if L.act == "bn":
        chi = 1.0 + torch.randn(L.d_out, generator=gen, device=device) * math.sqrt(2.0 / M)
        out["g_new"] = (chi.abs() * cfg.g_std ** 2).float()
        xh = 1.0 + torch.randn(1, generator=gen, device=device) * math.sqrt(2.0 / M)
        out["a_new"] = torch.cat([xh.abs(), torch.ones(1, device=device)]).float()
        sig = cfg.g_std * math.sqrt(1.0 / M)
        out["grad_w"] = torch.randn(L.d_out, 1, generator=gen, device=device) * sig
        out["grad_b"] = torch.randn(L.d_out, generator=gen, device=device) * sig
        return out
    a = torch.randn(M, L.d_in, generator=gen, device=device)
    if L.act == "relu":
        a.clamp_(min=0.0)
    g = torch.randn(M, L.d_out, generator=gen, device=device) * cfg.g_std
    out["a"], out["g"] = a.to(tdt), g.to(tdt)
    sig = cfg.g_std * math.sqrt(mean_sq_act(L.act) / M)
    out["grad_w"] = torch.randn(L.d_out, L.d_in, generator=gen, device=device) * sig
    out["grad_b"] = (torch.randn(L.d_out, generator=gen, device=device) * sig
                     if L.has_bias else None)
    return out


def initial_params_torch(cfg: Config, li: int, device):
    import torch
    L = cfg.layers[li]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed_for(cfg.index, li, 0))
    std = 1.0 / math.sqrt(L.d_in)
    w = torch.randn(L.d_out, L.d_in, generator=gen, device=device) * std
    b = torch.randn(L.d_out, generator=gen, device=device) * std if L.has_bias else None
    return w, b


def conv_inputs_torch(cfg: Config, li: int, step: int, device, batch: Optional[int] = None):
    """Same distributions as :func:`conv_inputs`, drawn on ``device`` with a seeded
    torch.Generator; x and gy in the layer's input dtype."""
    import torch
    L = cfg.layers[li]
    cg = L.conv if batch is None else L.conv.with_batch(batch)
    gen = torch.Generator(device=device)
    gen.manual_seed(conv_seed(cfg.index, li, step))
    tdt = torch.bfloat16 if L.in_dtype == "bf16" else torch.float32
    x = torch.randn(cg.batch, cg.c_in, cg.h, cg.w, generator=gen, device=device)
    if L.act == "relu":
        x.clamp_(min=0.0)
    gy = torch.randn(cg.batch, L.d_out, cg.h_out, cg.w_out, generator=gen, device=device)
    return {"x": x.to(tdt), "gy": (gy * cfg.g_std).to(tdt), "geom": cg}
