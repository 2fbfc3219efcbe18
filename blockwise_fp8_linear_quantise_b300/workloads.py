"""Seeded synthetic inputs shaped like Puro-2B's linear layers.

This module only draws random numbers; it holds none of the quantisation or
GEMM arithmetic.  Both the CUDA path and the CPU oracle consume the bf16
tensors it returns, so the two sides always see identical input bytes.

Model shapes follow "Puro-2B: Poor Lab's Qwen2-1.5B Trained on RTX 5090
within $5090" (bloombook.cn tutorial, model-architecture paragraph; paper
section 3.1): hidden 2048, 28 layers, 16 query heads and 8 KV heads of dim
128, FFN 6144, sequence 4096, micro-batch 2 (section 3.1.3) -> 8192 or 16384
tokens per GEMM.

Workloads (name -> what it is):

* ``tiny``       X [256, 256] ~ N(0,1) with 0.1% of entries x50, W [256, 256] ~ N(0, 0.02^2); fprop.
* ``mlp_gateup`` X [8192, 2048] ~ N(0,1) with 0.1% x30, W [12288, 2048] (gate || up) ~ N(0, 0.02^2); fprop.
* ``mlp_down``   X [8192, 6144] = SiLU(G) * U with G, U ~ 0.5 * Student-t(nu=4),
                 W [2048, 6144] ~ N(0, (0.02/sqrt(56))^2), dY [8192, 2048] ~ N(0, 1e-3^2); fprop, dgrad, wgrad.
                 ``gu`` [8192, 12288] = [G || U] itself, the gate+up output that the SiLU-gated
                 prologue turns into the down projection's input.
* ``attn_proj``  X [16384, 2048] ~ Student-t(nu=3) shared by QKV W [4096, 2048] and O W [2048, 2048]
                 ~ N(0, 0.02^2); dY [16384, 4096] and [16384, 2048] ~ N(0, 1e-3^2); all three layouts.
* ``stack28``    28 layers x {QKV 2048->4096, O 2048->2048, gate+up 2048->12288, down 6144->2048}
                 on 16384 tokens; activations and output gradients ~ N(0,1) with 0.1% x50,
                 weights ~ N(0, 0.02^2), distinct per layer; activations per shape are shared
                 across layers (the layers are not chained).

Every tensor has its own seed derived from (workload seed, tensor tag, layer).
"""

from dataclasses import dataclass, field
import math
import zlib

import numpy as np
import torch

TOKENS_8K = 8192
TOKENS_16K = 16384


@dataclass(frozen=True)
class Dist:
    """A value distribution for one tensor."""
    kind: str                 # "normal", "student_t", "silu_gated_t"
    scale: float = 1.0        # multiplies the draw
    nu: float = 0.0           # Student-t degrees of freedom
    outlier_frac: float = 0.0 # fraction of entries multiplied by outlier_mult
    outlier_mult: float = 1.0


@dataclass(frozen=True)
class LinearSpec:
    """One linear layer instance: Y [M, N] = X [M, K] . W [N, K]^T."""
    name: str
    M: int
    N: int
    K: int
    x_tag: str       # activations with equal tags are the same tensor
    w_tag: str
    dy_tag: str      # output-gradient tensor tag ("" when fprop only)
    backward: bool


@dataclass
class Workload:
    name: str
    seed: int
    linears: list
    dists: dict = field(default_factory=dict)   # tag -> Dist
    shapes: dict = field(default_factory=dict)  # tag -> (rows, cols)

    def gemm_flops(self):
        f = 0
        for l in self.linears:
            f += 2 * l.M * l.N * l.K * (3 if l.backward else 1)
        return f


def _tensor_seed(seed, tag):
    return [seed, zlib.crc32(tag.encode())]


def draw(dist, shape, seed, tag):
    """Draw a float32 numpy array of ``shape`` from ``dist`` (CPU, numpy PCG64)."""
    rng = np.random.default_rng(_tensor_seed(seed, tag))
    n = int(np.prod(shape))
    if dist.kind == "normal":
        v = rng.standard_normal(n, dtype=np.float32) * np.float32(dist.scale)
    elif dist.kind == "student_t":
        v = (rng.standard_t(dist.nu, n) * dist.scale).astype(np.float32)
    elif dist.kind == "silu_gated_t":
        g = rng.standard_t(dist.nu, n) * dist.scale
        u = rng.standard_t(dist.nu, n) * dist.scale
        v = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
    else:
        raise ValueError(dist.kind)
    if dist.outlier_frac > 0:
        mask = rng.random(n) < dist.outlier_frac
        v[mask] *= np.float32(dist.outlier_mult)
    return v.reshape(shape)


def to_bf16(a):
    """float32 numpy -> torch.bfloat16 CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def tensor(wl, tag, layer=None):
    """The bf16 CPU tensor for ``tag`` (weights take a layer index)."""
    key = tag if layer is None else f"{tag}@{layer}"
    return to_bf16(draw(wl.dists[tag], wl.shapes[tag], wl.seed, key))


def tensor_cuda(wl, tag, layer=None, device="cuda"):
    """Same distribution as ``tensor`` drawn directly on the GPU with torch's
    generator (different values; used only where no oracle comparison is made,
    to keep start-up of the large stacked workload short)."""
    dist = wl.dists[tag]
    key = tag if layer is None else f"{tag}@{layer}"
    g = torch.Generator(device=device)
    g.manual_seed((wl.seed * 1000003 + zlib.crc32(key.encode())) & 0x7FFFFFFF)
    shape = wl.shapes[tag]
    if dist.kind == "normal":
        v = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * dist.scale
    else:
        raise ValueError("device generation supports normal draws only")
    if dist.outlier_frac > 0:
        mask = torch.rand(shape, generator=g, device=device) < dist.outlier_frac
        v = torch.where(mask, v * dist.outlier_mult, v)
    return v.to(torch.bfloat16)


def _act(outlier_mult):
    return Dist("normal", 1.0, outlier_frac=1e-3, outlier_mult=outlier_mult)


W002 = Dist("normal", 0.02)
DY = Dist("normal", 1e-3)


def make(name):
    """Build the named workload description."""
    if name == "tiny":
        wl = Workload(name, 0, [LinearSpec("tiny", 256, 256, 256, "x", "w", "", False)])
        wl.dists = {"x": _act(50.0), "w": W002}
        wl.shapes = {"x": (256, 256), "w": (256, 256)}
    elif name == "mlp_gateup":
        M, N, K = TOKENS_8K, 12288, 2048
        wl = Workload(name, 2, [LinearSpec("gate_up", M, N, K, "x", "w", "", False)])
        wl.dists = {"x": _act(30.0), "w": W002}
        wl.shapes = {"x": (M, K), "w": (N, K)}
    elif name == "mlp_down":
        M, N, K = TOKENS_8K, 2048, 6144
        wl = Workload(name, 3, [LinearSpec("down", M, N, K, "x", "w", "dy", True)])
        wl.dists = {"x": Dist("silu_gated_t", 0.5, nu=4.0),
                    "w": Dist("normal", 0.02 / math.sqrt(2 * 28)), "dy": DY,
                    "gu": Dist("student_t", 0.5, nu=4.0)}
        wl.shapes = {"x": (M, K), "w": (N, K), "dy": (M, N), "gu": (M, 2 * K)}
    elif name == "attn_proj":
        M = TOKENS_16K
        wl = Workload(name, 4, [
            LinearSpec("qkv", M, 4096, 2048, "x", "w_qkv", "dy_qkv", True),
            LinearSpec("o", M, 2048, 2048, "x", "w_o", "dy_o", True)])
        wl.dists = {"x": Dist("student_t", 1.0, nu=3.0), "w_qkv": W002, "w_o": W002,
                    "dy_qkv": DY, "dy_o": DY}
        wl.shapes = {"x": (M, 2048), "w_qkv": (4096, 2048), "w_o": (2048, 2048),
                     "dy_qkv": (M, 4096), "dy_o": (M, 2048)}
    elif name == "stack28":
        M = TOKENS_16K
        lin = []
        for layer in range(28):
            lin += [
                LinearSpec(f"L{layer}.qkv", M, 4096, 2048, "x_h", "w_qkv", "dy_qkv", True),
                LinearSpec(f"L{layer}.o", M, 2048, 2048, "x_h", "w_o", "dy_o", True),
                LinearSpec(f"L{layer}.gate_up", M, 12288, 2048, "x_h", "w_gu", "dy_gu", True),
                LinearSpec(f"L{layer}.down", M, 2048, 6144, "x_f", "w_down", "dy_down", True),
            ]
        wl = Workload(name, 5, lin)
        wl.dists = {"x_h": _act(50.0), "x_f": _act(50.0),
                    "dy_qkv": _act(50.0), "dy_o": _act(50.0), "dy_gu": _act(50.0), "dy_down": _act(50.0),
                    "w_qkv": W002, "w_o": W002, "w_gu": W002, "w_down": W002}
        wl.shapes = {"x_h": (M, 2048), "x_f": (M, 6144),
                     "dy_qkv": (M, 4096), "dy_o": (M, 2048), "dy_gu": (M, 12288), "dy_down": (M, 2048),
                     "w_qkv": (4096, 2048), "w_o": (2048, 2048), "w_gu": (12288, 2048), "w_down": (2048, 6144)}
    else:
        raise KeyError(name)
    return wl


WORKLOADS = ("tiny", "mlp_gateup", "mlp_down", "attn_proj", "stack28")


def layer_of(spec):
    """Layer index of a stacked-workload linear (None for single layers)."""
    if spec.name.startswith("L") and "." in spec.name:
        return int(spec.name[1:spec.name.index(".")])
    return None
