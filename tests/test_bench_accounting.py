"""The roofline arithmetic bench.py reports, pinned on a toy layer by the
definitions written out by hand (no GPU): forward FLOPs (router 2 T d E,
routed experts 6 T K d F - three matrices, multiply-add = 2 - shared experts
6 T d Fs S; latent: the experts on L-wide rows plus the two projections),
forward bytes (the weights of the experts that got tokens, shared and router
weights, x read, FP32 out written), the gate/up launch's FLOPs and bytes,
the backward's FLOPs (twice the forward's products) and bytes (weights read,
FP32 gradients written), and the layer roofline max(t_FLOP, t_HBM) / time.
"""
import pytest

import bench
from mixture_experts_ffn_fp32_gb300 import workloads as W

# T=10, d=16, F=32, E=4, K=2, one shared expert of width 8, BF16
TOY = W.Workload("toy", T=10, d=16, d_ff=32, E=4, K=2, n_shared=1, shared_d_ff=8, dtype="bf16",
                 gate="softmax_topk")
# the same with a latent width of 8 between the projections
TOY_LAT = W.Workload("toy_lat", T=10, d=16, d_ff=32, E=4, K=2, n_shared=1, shared_d_ff=8,
                     dtype="bf16", gate="sigmoid", latent_dim=8)
PK = {"hbm_gbs": 1000.0, "bf16_tflops": 2.0, "fp32_tflops": 1.0, "source": "test"}


def test_forward_flops():
    # router 2*10*16*4 = 1280; routed 6*10*2*16*32 = 61440; shared 6*10*16*8 = 7680
    assert TOY.flops() == 1280 + 61440 + 7680
    # latent: routed 6*10*8*32*2 = 30720, projections 2*(2*10*16*8) = 5120
    assert TOY_LAT.flops() == 1280 + 7680 + 30720 + 5120


def test_forward_bytes_count_only_used_experts():
    # every expert used: 4 experts * 3 * 16*32 * 2 B = 12288; shared 3*16*8*2 = 768;
    # router 16*4*4 = 256; x 10*16*2 = 320; out 10*16*4 = 640
    assert bench.layer_bytes(TOY) == 12288 + 768 + 256 + 320 + 640
    # two experts without tokens: their weights are not read
    assert bench.layer_bytes(TOY, counts=[5, 0, 15, 0]) == 6144 + 768 + 256 + 320 + 640
    # latent: experts on 8-wide rows (4*3*8*32*2 = 6144) plus W_dl, W_ul (2*16*8*2 = 512)
    assert bench.layer_bytes(TOY_LAT) == 6144 + 768 + 256 + 512 + 320 + 640


def test_gate_up_launch():
    # FLOPs: 4*10*2*16*32 routed + 4*10*16*8 shared
    assert bench.gate_up_flops(TOY) == 40960 + 5120
    # bytes: gate+up weights 4*2*16*32*2 = 8192, routed rows in 20*16*2 = 640,
    # hidden rows out 20*32*2 = 1280, shared weights 2*16*8*2 = 512, token rows
    # 10*16*2 = 320, shared hidden 10*8*2 = 160
    assert bench.gate_up_bytes(TOY) == 8192 + 640 + 1280 + 512 + 320 + 160


def test_backward_flops_and_bytes():
    # twice the routed and shared products (12 = 2 x 6), the router's two (4 T d E)
    assert bench.backward_flops(TOY) == 12 * 10 * 2 * 16 * 32 + 12 * 10 * 16 * 8 + 4 * 10 * 16 * 4
    # weights read (2 B) and their FP32 gradients written (4 B): (4*3*16*32 + 3*16*8) * 6;
    # router weights read and gradient written: 16*4*8; x (2 B) and dout, dx (FP32): 10*16*10
    assert bench.backward_bytes(TOY) == (6144 + 384) * 6 + 512 + 1600
    assert bench.backward_bytes(TOY, counts=[3, 0, 0, 17]) == (3072 + 384) * 6 + 512 + 1600


def test_layer_roofline_takes_the_larger_bound():
    # t_FLOP = 70400 / 2e12 s = 3.52e-5 ms; t_HBM = 14272 / 1e12 s = 1.4272e-5 ms
    r = bench.layer_roofline(TOY, 1e-4, None, PK)
    assert r["bound"] == "tensor"
    assert r["t_flop_ms"] == pytest.approx(3.52e-5)
    assert r["t_hbm_ms"] == pytest.approx(1.4272e-5)
    assert r["frac"] == pytest.approx(0.352)
    # a slow HBM makes the same layer HBM-bound
    r = bench.layer_roofline(TOY, 1e-4, None, dict(PK, hbm_gbs=100.0))
    assert r["bound"] == "hbm"
    assert r["frac"] == pytest.approx(1.4272)
