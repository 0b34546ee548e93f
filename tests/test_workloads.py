"""Workload shapes against the shapes the pages print (tests/golden)."""
import json
import os

import pytest

from long_sequence_attention_02_b300 import workloads

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "video_token_grids.json")))


@pytest.mark.parametrize("case", GOLD["cases"])
def test_latent_grid(case):
    g = workloads.latent_grid(case["frames"], case["height"], case["width"])
    assert list(g) == case["grid"]
    assert g[0] * g[1] * g[2] == case["tokens"]


@pytest.mark.parametrize("m", GOLD["models"])
def test_head_dim(m):
    assert m["dim"] // m["heads"] == m["head_dim"] == 128


def test_named_workloads():
    w = workloads.WORKLOADS
    assert w["wan1.3b_480p_self_fwd"].L == 32760 and w["wan1.3b_480p_self_fwd"].H == 12
    assert w["wan14b_720p_self_fwd"].L == 75600 and w["wan14b_720p_self_fwd"].H == 40
    assert w["wan14b_720p_cross_fwd"].Lk == GOLD["text_tokens_max"]
    assert w["train_64x64x64_fwd_bwd"].L == 262144
    assert w["tiny_3x8x8_h2"].L == 192
    assert w["wan14b_720p_self_fwd"].flops() == pytest.approx(1.1705e14, rel=1e-4)
    # the FP8 workloads are the same problems computed in e4m3
    for name, base in [("wan14b_720p_self_fwd_fp8", "wan14b_720p_self_fwd"),
                       ("wan1.3b_480p_self_fwd_fp8", "wan1.3b_480p_self_fwd")]:
        assert w[name].kind == "self_fwd_fp8"
        assert (w[name].B, w[name].grid, w[name].H) == (w[base].B, w[base].grid, w[base].H)
        assert w[name].flops() == w[base].flops()


def test_bad_video_shapes():
    with pytest.raises(ValueError):
        workloads.latent_grid(80, 480, 832)
    with pytest.raises(ValueError):
        workloads.latent_grid(81, 480, 830)


def test_conv_workloads():
    from oracle import vae

    for w in workloads.CONV_WORKLOADS.values():
        assert w.kind in ("conv3d", "time_down") and w.c_in % 32 == 0 and w.c_out % 32 == 0
        assert w.T <= 4                      # chunks of at most four frames
        if w.kind == "conv3d":
            assert w.flops() == vae.conv3d_flops(w.B, w.T, w.H, w.W, w.c_in, w.c_out)
        else:
            assert w.T % 2 == 0 and w.t_out() == w.T // 2   # later chunks: an even frame count, halved
            assert w.flops() == vae.time_downsample_flops(w.B, w.T // 2, w.H, w.W, w.c_in, w.c_out)
    # a 4-frame 720p chunk through both downsampling layers ends as one latent frame
    d1 = workloads.CONV_WORKLOADS["wan_vae_time_down_180x320_192"]
    d2 = workloads.CONV_WORKLOADS["wan_vae_time_down_90x160_384"]
    assert d1.t_out() == d2.T and d2.t_out() == 1 and (d1.H, d1.W) == (2 * d2.H, 2 * d2.W)
    big = workloads.CONV_WORKLOADS["wan_vae_conv3d_360x640_192"]
    assert big.B * big.T * big.H * big.W * big.c_in * 2 > 126 * 2**20   # the timed layer's input exceeds L2
