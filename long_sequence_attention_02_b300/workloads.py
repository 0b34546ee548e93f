"""Named attention workloads and the video -> token-grid rule.

The token grid follows the gojay.top "Wan2.1" reading, *DiT backbone* and
*Wan-VAE*: the VAE keeps the first frame and compresses the remaining ones 4x
in time and 8x8 in space, and the DiT patchifies the latent with a (1, 2, 2)
patch, so a video of 1+T frames at H x W becomes a grid of
(1 + T/4) x H/16 x W/16 tokens. Model shapes come from the *⑥ 1.3B vs 14B*
config table of the same page (dim 1536 / 12 heads and 5120 / 40 heads, so a
head is 128 wide; text conditioning of at most 512 umT5 tokens).
"""
from __future__ import annotations

from dataclasses import dataclass


def latent_grid(frames: int, height: int, width: int):
    """(F, Hp, Wp) token grid of a video of ``frames`` = 1 + T frames."""
    if frames < 1 or (frames - 1) % 4:
        raise ValueError("frames must be 1 + 4k")
    if height % 16 or width % 16:
        raise ValueError("height and width must be multiples of 16")
    return 1 + (frames - 1) // 4, height // 16, width // 16


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "self_fwd", "self_fwd_fp8", "cross_fwd" or "self_fwd_bwd"
    B: int
    grid: tuple          # (F, Hp, Wp) of the queries
    H: int
    d: int = 128
    Lk: int = 0          # cross-attention text keys (allocated length)
    kv_len_range: tuple = (16, 512)

    @property
    def L(self) -> int:
        F, Hp, Wp = self.grid
        return F * Hp * Wp

    def flops(self) -> float:
        """4*B*H*Lq*Lk*d forward; the backward counts 2.5x that on top."""
        lk = self.Lk if self.kind == "cross_fwd" else self.L
        f = 4.0 * self.B * self.H * self.L * lk * self.d
        return f * 3.5 if self.kind == "self_fwd_bwd" else f


WORKLOADS = {
    "tiny_3x8x8_h2": Workload("tiny_3x8x8_h2", "self_fwd", 1, (3, 8, 8), 2),
    "wan1.3b_480p_self_fwd": Workload("wan1.3b_480p_self_fwd", "self_fwd", 1, latent_grid(81, 480, 832), 12),
    "wan14b_720p_cross_fwd": Workload("wan14b_720p_cross_fwd", "cross_fwd", 2, latent_grid(81, 720, 1280), 40, Lk=512),
    "wan14b_720p_self_fwd": Workload("wan14b_720p_self_fwd", "self_fwd", 1, latent_grid(81, 720, 1280), 40),
    # The same 75,600-token, 40-head forward computed in FP8 (e4m3).
    "wan14b_720p_self_fwd_fp8": Workload("wan14b_720p_self_fwd_fp8", "self_fwd_fp8", 1, latent_grid(81, 720, 1280),
                                         40),
    # The 32,760-token, 12-head forward in FP8: small enough for a full
    # profiler capture of the FP8 kernel.
    "wan1.3b_480p_self_fwd_fp8": Workload("wan1.3b_480p_self_fwd_fp8", "self_fwd_fp8", 1, latent_grid(81, 480, 832),
                                          12),
    "train_64x64x64_fwd_bwd": Workload("train_64x64x64_fwd_bwd", "self_fwd_bwd", 1, (64, 64, 64), 12),
    # Same step at 1/64 of the size (32,768 tokens): small enough for a full
    # profiler capture of the backward kernel.
    "train_32x32x32_fwd_bwd": Workload("train_32x32x32_fwd_bwd", "self_fwd_bwd", 1, (32, 32, 32), 12),
}


@dataclass(frozen=True)
class ConvWorkload:
    """One causal 3x3x3 Conv3d layer of the VAE on one chunk of frames
    (channels last, bf16), with the previous chunk's cache.

    The pages give the VAE's compression (4x in time, 8x8 in space, 16 latent
    channels) and its chunking (chunks of up to 4 frames, a 2-frame cache) but
    not its channel widths; the shapes below are decoder-scale layers of that
    plan: 384 channels at 1/8 of a 720p frame and 192 at 1/2.
    """
    name: str
    B: int
    T: int
    H: int
    W: int
    c_in: int
    c_out: int
    kind: str = "conv3d"   # or "time_down": the 3 x 1 x 1, time-stride-2 layer (T input frames)

    def t_out(self) -> int:
        return self.T // 2 if self.kind == "time_down" else self.T

    def taps(self) -> int:
        return 3 if self.kind == "time_down" else 27

    def flops(self) -> float:
        """2 FLOP per multiply-add: 2 * outputs * C_out * taps * C_in."""
        return 2.0 * self.B * self.t_out() * self.H * self.W * self.c_out * self.taps() * self.c_in


CONV_WORKLOADS = {
    # 4 frames of 90 x 160 (720p / 8), 384 -> 384: inputs fit L2; parity case
    "wan_vae_conv3d_720p_384": ConvWorkload("wan_vae_conv3d_720p_384", 1, 4, 90, 160, 384, 384),
    # 4 frames of 360 x 640 (720p / 2), 192 -> 192: 354 MB of input, > L2; the timed layer
    "wan_vae_conv3d_360x640_192": ConvWorkload("wan_vae_conv3d_360x640_192", 1, 4, 360, 640, 192, 192),
    # 4 frames of 720 x 1280 (full 720p), 96 -> 96: an outer stage, reduced in 32-channel K steps
    "wan_vae_conv3d_720x1280_96": ConvWorkload("wan_vae_conv3d_720x1280_96", 1, 4, 720, 1280, 96, 96),
    # The encoder's two time-downsampling layers for a 720p chunk of 4 frames
    # (the spatial 2x stages halve 720 x 1280 first): 4 -> 2 frames of
    # 180 x 320 at 192 channels, then 2 -> 1 frame of 90 x 160 at 384.
    "wan_vae_time_down_180x320_192": ConvWorkload("wan_vae_time_down_180x320_192", 1, 4, 180, 320, 192, 192,
                                                  kind="time_down"),
    "wan_vae_time_down_90x160_384": ConvWorkload("wan_vae_time_down_90x160_384", 1, 2, 90, 160, 384, 384,
                                                 kind="time_down"),
}
