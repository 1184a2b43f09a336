"""Workload shapes of the joint-sequence attention path.

Each workload is a video DiT attention call: batch B, H heads of dim d, a
video latent grid (t, h, w) flattened row-major into Nv = t*h*w tokens, and Nj
joint (text or audio) tokens placed after the video tokens on both the query
and the key/value side.  The video grids follow the latent geometry rule
frames -> (F-1)//4 + 1, pixels -> (px//8)//2 ("Context Parallelism in vLLM
Omni Neuron", section "Sequence Length Constraints"):
  - Kandinsky 6 Lite, 432x256, 25 frames -> (7, 16, 27)
    (diffusers issue #15156, "Setup");
  - FLUX.1 1024x1024 image, 256 text tokens -> (1, 64, 64)
    (xDiT PR #586, "Tests", Flux run command);
  - Kandinsky 6 Pro, 864x480, 125 frames -> (32, 30, 54)
    (vLLM-Omni recipe "Kandinsky 6 TI2VA -- H100", "Measured performance");
  - HunyuanVideo 720x1280, 129 frames -> (33, 45, 80)
    (xDiT PR #586, "Tests", HunyuanVideo run command).
The joint token counts (64, 128, 256, 520) are not on the pages; they are
fixed here per workload.  No arithmetic of the method lives in this module.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    d: int
    dtype: str              # "bf16" or "f32"
    grid: tuple             # (t, h, w)
    Nj: int                 # joint tokens
    axis_dim: tuple         # head dims of the t, h, w rotary axes
    joint_rope: int         # 0: joint tokens unrotated, 1: 1-D rotary over full d
    qk_std: float           # std of the N(0, std^2) Q and K entries
    v_std: float
    chunks: tuple           # K/V chunk counts exercised
    relayout_P: tuple = ()  # seq<->head split factors exercised
    theta: float = 10000.0
    note: str = ""

    @property
    def Nv(self) -> int:
        return self.grid[0] * self.grid[1] * self.grid[2]

    @property
    def S(self) -> int:
        return self.Nv + self.Nj

    def flops(self) -> float:
        """4 * B * H * Sq * Sk * d (QK^T and PV, one multiply-add = 2 flops)."""
        return 4.0 * self.B * self.H * self.S * self.S * self.d

    def with_batch(self, B: int) -> "Workload":
        return replace(self, B=B, name=f"{self.name}_b{B}")


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 64, "f32", (4, 16, 16), 64, (16, 24, 24), 0, 1.0, 1.0, (4, 1), (1, 2, 4),
                     note="1024 video + 64 text tokens, fp32"),
    "lite": Workload("lite", 1, 24, 128, "bf16", (7, 16, 27), 128, (32, 48, 48), 1, 1.0, 1.0, (2,), (1, 8),
                     note="Kandinsky 6 Lite geometry, 3024 video + 128 audio tokens (1-D rotary on audio)"),
    "image": Workload("image", 1, 24, 128, "bf16", (1, 64, 64), 256, (0, 64, 64), 0, 1.0, 1.0, (2,), (8,),
                      note="image DiT 4096 image + 256 text tokens, 2-D rotary"),
    "pro": Workload("pro", 1, 24, 128, "bf16", (32, 30, 54), 520, (32, 48, 48), 0, 0.5, 1.0, (8,), (8,),
                    note="Kandinsky 6 Pro geometry, 51840 video + 520 audio tokens = 52360"),
    # profiling case: half the Pro video grid in time (inputs still larger than L2, a few GB on device)
    "mid": Workload("mid", 1, 24, 128, "bf16", (16, 30, 54), 520, (32, 48, 48), 0, 0.5, 1.0, (2,), (8,),
                    note="half-length Pro geometry, 25920 video + 520 audio tokens = 26440"),
    "long": Workload("long", 1, 24, 128, "bf16", (33, 45, 80), 256, (32, 48, 48), 0, 1.0, 1.0, (8, 16), (8,),
                     note="HunyuanVideo 720x1280x129 geometry, 118800 video + 256 text tokens = 119056"),
}
