"""Seeded synthetic workloads for the compressed Lion step.

Holds none of the optimizer's arithmetic.  It provides

* the parameter layouts of the pages' models (GPT-2 shapes; ViT-B/16 and
  DeiT-Tiny), as (name, offset, numel, flags) tensors of one flat vector;
* the workload configurations (workers, layout, gradient distribution,
  compression mode, hyper-parameters, step count);
* a counter-based GPU generator (``synth.cu``) for gradients and initial
  parameters, so each (seed, step, worker) stream is reproducible and the
  CPU oracle can consume a host copy of exactly the bits the GPU path sees;
* a numpy generator of the same distributions (different bits) for runs
  that only time the CPU oracle.

Gradients follow the workloads' stated distributions: N(0, 1e-3^2) fp32 for
the flat 1M-element case, 1e-3 * Student-t(nu) rounded to bf16 for the GPT
and ViT layouts (nu = 3, or nu = 2.5 with 0.1% of entries scaled by 100), matching
the heavy-tailed, Laplace-like update statistics reported in "Lion Cub:
Minimizing Communication Overhead in Distributed Lion" (Fig. 3 caption).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.cu")
_LIB = os.path.join(_HERE, "libsynth.so")

SYNC_M = 1  # tensor flag: momentum averaged across workers


# ---------------------------------------------------------------------------
# layouts
# ---------------------------------------------------------------------------

def gpt2_layout(d_model: int, n_layer: int, vocab: int = 50257, n_ctx: int = 1024,
                untied_head: bool = False, sync=()):
    """Flat GPT-2 parameter layout: wte, wpe; per block ln_1 (w, b), c_attn
    (w, b), c_proj (w, b), ln_2 (w, b), c_fc (w, b), mlp c_proj (w, b); ln_f
    (w, b); then the output head when it is not tied to wte.  ``sync`` names
    the tensors whose momentum is synchronized (the head is wte when tied)."""
    D = d_model
    shapes = [("wte", vocab * D), ("wpe", n_ctx * D)]
    for b in range(n_layer):
        p = f"h{b}."
        shapes += [(p + "ln_1.w", D), (p + "ln_1.b", D),
                   (p + "attn.c_attn.w", D * 3 * D), (p + "attn.c_attn.b", 3 * D),
                   (p + "attn.c_proj.w", D * D), (p + "attn.c_proj.b", D),
                   (p + "ln_2.w", D), (p + "ln_2.b", D),
                   (p + "mlp.c_fc.w", D * 4 * D), (p + "mlp.c_fc.b", 4 * D),
                   (p + "mlp.c_proj.w", 4 * D * D), (p + "mlp.c_proj.b", D)]
    shapes += [("ln_f.w", D), ("ln_f.b", D)]
    if untied_head:
        shapes.append(("head", vocab * D))
    out, off = [], 0
    for name, n in shapes:
        flags = SYNC_M if name in sync else 0
        out.append((name, off, n, flags))
        off += n
    return out


def vit_layout(d_model: int, n_layer: int, n_classes: int, img: int = 224, patch: int = 16, in_ch: int = 3,
               mlp_ratio: int = 4, sync=()):
    """Flat ViT / DeiT parameter layout (timm order): patch projection (w, b),
    class token, position embedding ((img/patch)^2 + 1 positions); per block
    norm1 (w, b), attn.qkv (w, b), attn.proj (w, b), norm2 (w, b), mlp.fc1
    (w, b), mlp.fc2 (w, b); the final norm (w, b); the classification head
    (w, b), last, so that its bias (n_classes elements, often not a multiple
    of 32) is the ragged tail.  ``sync`` names the flagged tensors."""
    D, H = d_model, mlp_ratio * d_model
    n_pos = (img // patch) ** 2 + 1
    shapes = [("patch_embed.w", D * in_ch * patch * patch), ("patch_embed.b", D), ("cls_token", D),
              ("pos_embed", n_pos * D)]
    for b in range(n_layer):
        p = f"blocks{b}."
        shapes += [(p + "norm1.w", D), (p + "norm1.b", D), (p + "attn.qkv.w", 3 * D * D), (p + "attn.qkv.b", 3 * D),
                   (p + "attn.proj.w", D * D), (p + "attn.proj.b", D), (p + "norm2.w", D), (p + "norm2.b", D),
                   (p + "mlp.fc1.w", H * D), (p + "mlp.fc1.b", H), (p + "mlp.fc2.w", D * H), (p + "mlp.fc2.b", D)]
    shapes += [("norm.w", D), ("norm.b", D), ("head.w", n_classes * D), ("head.b", n_classes)]
    out, off = [], 0
    for name, n in shapes:
        out.append((name, off, n, SYNC_M if name in sync else 0))
        off += n
    return out


def flat_layout(d: int):
    return [("flat", 0, d, 0)]


def layout_total(layout) -> int:
    return sum(n for (_, _, n, _) in layout)


def abi_layout(layout):
    """(name, offset, numel, flags) -> (offset, numel, flags) for the C ABIs."""
    return [(o, n, f) for (_, o, n, f) in layout]


# ---------------------------------------------------------------------------
# workload configurations
# ---------------------------------------------------------------------------

@dataclass
class Workload:
    key: int
    name: str
    W: int
    layout: list
    grad: str            # "f32" or "bf16"
    dist: tuple          # ("normal", sigma) or ("t", nu, scale, outlier_frac, outlier_mult)
    mode: int            # 0 sign/majority, 1 L1/int-sum
    nbits: int
    steps: int
    sync_interval: int = 0
    beta1: float = 0.9
    beta2: float = 0.99
    lr: float = 1e-4
    wd: float = 0.1
    theta_range: float = 0.05
    seed: int = 0
    flags: int = 0       # mode flags OR'ed into the mode: 0x100 tie alternation, 0x200 D-Lion average
    notes: str = field(default="")

    @property
    def d(self) -> int:
        return layout_total(self.layout)


def workloads():
    med = dict(d_model=1024, n_layer=24)
    return {
        1: Workload(1, "flat-1M-w4-sign-f32", 4, flat_layout(1_048_576), "f32", ("normal", 1e-3),
                    0, 1, 10),
        2: Workload(2, "gpt2-small-124M-w8-sign", 8, gpt2_layout(768, 12), "bf16",
                    ("t", 3.0, 1e-3, 0.0, 1.0), 0, 1, 20),
        3: Workload(3, "gpt2-medium-350M-w8-l1n4", 8, gpt2_layout(**med), "bf16",
                    ("t", 2.5, 1e-3, 0.001, 100.0), 1, 4, 20),
        4: Workload(4, "gpt2-medium-350M-w16-sign-wte-sync", 16, gpt2_layout(**med, sync=("wte",)),
                    "bf16", ("t", 3.0, 1e-3, 0.0, 1.0), 0, 1, 20, sync_interval=1),
        5: Workload(5, "gpt2-xl-like-1.3B-w8-l1n2", 8, gpt2_layout(2048, 24, untied_head=True), "bf16",
                    ("t", 3.0, 1e-3, 0.0, 1.0), 1, 2, 10),
        # the pages' vision models, beyond the five configurations above:
        # ViT-B/16 on ImageNet with the D-Lion average aggregation, and
        # DeiT-Tiny fine-tuned on CIFAR-100 with input-embedding and head
        # momentum synchronized
        6: Workload(6, "vit-b16-86M-w8-dlion-avg", 8, vit_layout(768, 12, 1000), "bf16",
                    ("t", 3.0, 1e-3, 0.0, 1.0), 0, 1, 20, flags=0x200),
        7: Workload(7, "deit-tiny-5.5M-w8-l1n4-embed-head-sync", 8,
                    vit_layout(192, 12, 100, sync=("patch_embed.w", "patch_embed.b", "cls_token", "pos_embed",
                                                   "head.w", "head.b")),
                    "bf16", ("t", 3.0, 1e-3, 0.0, 1.0), 1, 4, 20, sync_interval=1),
    }


# ---------------------------------------------------------------------------
# GPU generator
# ---------------------------------------------------------------------------

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
           "-Xcompiler", "-fPIC", "-cudart", "static", "-o", tmp, _SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the synthetic-input generator failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB):
                raise RuntimeError(f"{_LIB} is missing: run synth.build()")
            L = ctypes.CDLL(_LIB)
            L.synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float, ctypes.c_float,
                                     ctypes.c_float, ctypes.c_float, ctypes.c_void_p]
            L.synth_fill.restype = ctypes.c_int
            _lib = L
    return _lib


def _stream_id(kind: str, step: int, worker: int) -> int:
    tag = {"grad": 1, "theta": 2, "m": 3}[kind]
    return (tag << 56) | ((step & 0xffffffff) << 16) | (worker & 0xffff)


def fill_(tensor, kind: int, seed: int, stream_id: int, p=(0.0, 0.0, 0.0, 0.0), stream=None):
    """Fill a contiguous CUDA tensor (float32 or bfloat16) in place."""
    import torch
    assert tensor.is_cuda and tensor.is_contiguous()
    if tensor.dtype == torch.bfloat16:
        bf = 1
    elif tensor.dtype == torch.float32:
        bf = 0
    else:
        raise TypeError("float32 or bfloat16 only")
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = _load().synth_fill(tensor.data_ptr(), bf, tensor.numel(), kind, seed, stream_id,
                            float(p[0]), float(p[1]), float(p[2]), float(p[3]), s or None)
    if rc != 0:
        raise RuntimeError(f"synth_fill failed with CUDA error {rc}")
    return tensor


def fill_grad_(tensor, wl: Workload, step: int, worker: int, stream=None):
    if wl.dist[0] == "normal":
        return fill_(tensor, 0, wl.seed, _stream_id("grad", step, worker), (wl.dist[1], 0, 0, 0), stream)
    _, nu, scale, frac, mult = wl.dist
    return fill_(tensor, 2, wl.seed, _stream_id("grad", step, worker), (nu, scale, frac, mult), stream)


def fill_theta_(tensor, wl: Workload, stream=None):
    r = wl.theta_range
    return fill_(tensor, 1, wl.seed, _stream_id("theta", 0, 0), (-r, r, 0, 0), stream)


def grad_dtype(wl: Workload):
    import torch
    return torch.float32 if wl.grad == "f32" else torch.bfloat16


# ---------------------------------------------------------------------------
# numpy generator (same distributions, different bits): CPU-only timing runs
# ---------------------------------------------------------------------------

def numpy_grad(wl: Workload, n: int, step: int, worker: int) -> np.ndarray:
    """Host gradients of the workload's distribution: float32, or bf16 as
    uint16 bit patterns (round to nearest even)."""
    rng = np.random.default_rng([wl.seed, step, worker])
    if wl.dist[0] == "normal":
        x = (rng.standard_normal(n) * wl.dist[1]).astype(np.float32)
    else:
        _, nu, scale, frac, mult = wl.dist
        x = (rng.standard_t(nu, n) * scale).astype(np.float32)
        if frac > 0:
            x[rng.random(n) < frac] *= np.float32(mult)
    if wl.grad == "f32":
        return x
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def numpy_theta(wl: Workload, n: int) -> np.ndarray:
    rng = np.random.default_rng([wl.seed, 1 << 20])
    r = wl.theta_range
    return rng.uniform(-r, r, n).astype(np.float32)
