"""Seeded synthetic inputs for the forward convolution workloads.

This module only draws random tensors and names shapes; it holds none of the
convolution or quantisation arithmetic.  Both the CUDA path (through the
binding) and the CPU oracle (through the tests) consume exactly the bytes it
produces, so it is the one module the two sides share.

Recipe: activations ~ N(0, 1) and weights ~ N(0, std) with
std = 1/sqrt(C*T*R*S), drawn in fp32 from a seeded torch generator and
rounded to bf16 (round to nearest even).  Seeds: x 1000+i, w 2000+i, output
sample indices 3000+i for workload i.  The shapes are those of the
convolution workloads the method is measured on: a tiny 3x3x3 case, the
ViT-style 14x14 stride-14 patch embedding, a 2048-channel video conv, the
1024-channel fp8 1x3x3 conv on an NCDHW bf16 input, and a 640-channel 3x1x1
temporal conv whose tensors exceed 2^31 elements.  Two more cover patch
embeddings with many patches per image (16x16 and 14x14 patches of 224x224
RGB images: stride == filter, output 14x14 / 16x16 per image).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    x_shape: Tuple[int, ...]      # NDHWC, or NCDHW when x_layout == "ncdhw"
    w_shape: Tuple[int, ...]      # KTRSC, or KCTRS when w_layout == "kctrs"
    stride: Tuple[int, int, int]
    pad: Tuple[int, int, int]
    dil: Tuple[int, int, int] = (1, 1, 1)
    dtype: str = "bf16"           # compute dtype of the conv: "bf16" or "fp8"
    x_layout: str = "ndhwc"
    w_layout: str = "ktrsc"

    @property
    def x_seed(self) -> int:
        return 1000 + self.index

    @property
    def w_seed(self) -> int:
        return 2000 + self.index

    @property
    def sample_seed(self) -> int:
        return 3000 + self.index

    @property
    def crs(self) -> int:
        """C*T*R*S: the reduction length, used for the weight std."""
        if self.w_layout == "ktrsc":
            K, T, R, S, C = self.w_shape
        else:
            K, C, T, R, S = self.w_shape
        return C * T * R * S

    @property
    def w_std(self) -> float:
        return 1.0 / math.sqrt(self.crs)


WORKLOADS = [
    Workload("tiny_conv3d_bf16", 0, (1, 4, 8, 8, 16), (32, 3, 3, 3, 16), (1, 1, 1), (1, 1, 1)),
    Workload("patch_embed_bf16", 1, (9500, 1, 14, 14, 3), (1280, 1, 14, 14, 3), (1, 14, 14),
             (0, 0, 0)),
    Workload("video_conv3d_bf16", 2, (1, 15, 120, 120, 2048), (2048, 3, 3, 3, 2048), (1, 1, 1),
             (1, 1, 1)),
    Workload("fp8_conv3d_1x3x3", 3, (1, 1024, 120, 160, 90), (1024, 1024, 1, 3, 3), (1, 1, 1),
             (0, 1, 1), dtype="fp8", x_layout="ncdhw", w_layout="kctrs"),
    Workload("temporal_3x1x1_bf16_big", 4, (1, 240, 160, 90, 640), (640, 3, 1, 1, 640),
             (1, 1, 1), (1, 0, 0)),
]

# Reduced-depth variants of the large workloads for multi-pass profiler
# captures: same channels, filters and padding, fewer frames; every input is
# still larger than the 129 MB L2.
PROFILE_WORKLOADS = [
    Workload("video_conv3d_bf16_small", 5, (1, 3, 120, 120, 2048), (2048, 3, 3, 3, 2048),
             (1, 1, 1), (1, 1, 1)),
    Workload("fp8_conv3d_1x3x3_small", 6, (1, 1024, 16, 160, 90), (1024, 1024, 1, 3, 3),
             (1, 1, 1), (0, 1, 1), dtype="fp8", x_layout="ncdhw", w_layout="kctrs"),
    Workload("temporal_3x1x1_bf16_small", 7, (1, 16, 160, 90, 640), (640, 3, 1, 1, 640),
             (1, 1, 1), (1, 0, 0)),
]

# Patch embeddings with many patches per image (stride == filter, output
# spatially larger than 1x1): the gathered-patch GEMM.
PATCH_WORKLOADS = [
    Workload("vit_patch16_bf16", 8, (64, 1, 224, 224, 3), (768, 1, 16, 16, 3), (1, 16, 16),
             (0, 0, 0)),
    Workload("vit_patch14_bf16", 9, (64, 1, 224, 224, 3), (1024, 1, 14, 14, 3), (1, 14, 14),
             (0, 0, 0)),
]

# Channel-major (NCDHW) activations read in place by conv_fwd_ncdhw: the
# temporal workload with its activation in torch's layout, and the pointwise
# conv FlyDSL PR #860's 1x1x1 commit measures (a 14 GB bf16 activation of 512
# channels over [240, 320, 180], 48 filters; 6.8e11 flop at 8.7 ms = 78 TF).
NCDHW_WORKLOADS = [
    Workload("temporal_3x1x1_bf16_ncdhw", 10, (1, 640, 240, 160, 90), (640, 3, 1, 1, 640),
             (1, 1, 1), (1, 0, 0), x_layout="ncdhw"),
    Workload("pointwise_1x1x1_bf16_ncdhw", 11, (1, 512, 240, 320, 180), (48, 1, 1, 1, 512),
             (1, 1, 1), (0, 0, 0), x_layout="ncdhw"),
    # profiler-capture sizes of the first: 16 frames (channel planes 0.46 MB
    # apart) and 96 frames (2.8 MB apart, past a 2 MB page per channel plane)
    Workload("temporal_3x1x1_bf16_ncdhw_small", 12, (1, 640, 16, 160, 90), (640, 3, 1, 1, 640),
             (1, 1, 1), (1, 0, 0), x_layout="ncdhw"),
    Workload("temporal_3x1x1_bf16_ncdhw_d96", 13, (1, 640, 96, 160, 90), (640, 3, 1, 1, 640),
             (1, 1, 1), (1, 0, 0), x_layout="ncdhw"),
]

BY_NAME = {w.name: w for w in WORKLOADS + PROFILE_WORKLOADS + PATCH_WORKLOADS + NCDHW_WORKLOADS}


def randn_bf16(shape, seed: int, std: float = 1.0, device="cpu",
               chunk_elems: int = 1 << 28) -> torch.Tensor:
    """bf16 tensor of N(0, std^2) draws: fp32 randn from a generator seeded
    with ``seed`` on ``device``, times ``std``, rounded to bf16.  Large
    tensors are drawn in chunks (same generator, sequential) to bound the
    fp32 temporary."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        tmp = torch.randn(e - s, generator=gen, device=dev, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        flat[s:e].copy_(tmp)
        del tmp
    return out


def make_inputs(wl: Workload, device="cpu", x_shape: Optional[Tuple[int, ...]] = None):
    """(x, w) bf16 tensors for workload ``wl`` on ``device``.  ``x_shape``
    overrides the activation shape (reduced-size parity cases keep the
    workload's filter and seeds)."""
    xs = tuple(x_shape) if x_shape is not None else wl.x_shape
    x = randn_bf16(xs, wl.x_seed, 1.0, device)
    w = randn_bf16(wl.w_shape, wl.w_seed, wl.w_std, device)
    return x, w


def sample_indices(total: int, count: int, seed: int) -> torch.Tensor:
    """``count`` uniform random flat indices in [0, total) (int64, CPU)."""
    gen = torch.Generator()
    gen.manual_seed(int(seed))
    return torch.randint(0, total, (count,), generator=gen, dtype=torch.int64)
