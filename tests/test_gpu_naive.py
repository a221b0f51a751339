"""Naive patch parallelism -- the seam baseline the method is measured
against (DistriFusion notes, Introduction para. 3: every band generated on
its own): zero-halo conv (DPP_HALO_ZERO), band-local GroupNorm and band-local
self-attention, through the C ABI against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import gpu_ops as G

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16


def draw(shape, seed, dt):
    return wl.normal(shape, seed, dtype="bf16" if dt == BF16 else "f32")


@pytest.mark.parametrize("B,H,W,Ci,Co,P,dt", [
    (2, 12, 20, 32, 48, 3, BF16),   # tensor-core conv, ragged tiles
    (1, 16, 150, 64, 160, 4, BF16),  # two row segments
    (1, 12, 10, 16, 8, 3, F32),     # SIMT conv
])
def test_naive_conv(cuda_device, B, H, W, Ci, Co, P, dt):
    F = draw((B, H, W, Ci), 800, dt)
    Wt = wl.conv_weight(Co, Ci, 801, "bf16" if dt == BF16 else "f32")
    bias = wl.normal((Co,), 802)
    y = G.conv(F, None, Wt, bias, P, halo=G.dpp.DPP_HALO_ZERO)
    ref = oracle.naive_conv3x3(G.f64(F), G.f64(Wt), G.f64(bias), P)
    G.assert_rms_close(G.f64(y), ref, G.TOL[dt], "naive conv")
    # the same as the displaced conv reading an all-zero stale buffer
    y0 = G.conv(F, torch.zeros_like(F), Wt, bias, P)
    bits = torch.int16 if dt == BF16 else torch.int32
    assert torch.equal(y.view(bits), y0.view(bits))


@pytest.mark.parametrize("B,H,W,C,Gn,P,dt", [
    (2, 16, 12, 320, 32, 4, BF16),
    (1, 12, 7, 40, 8, 3, BF16),
    (1, 32, 32, 64, 32, 2, F32),
])
def test_band_local_groupnorm(cuda_device, B, H, W, C, Gn, P, dt):
    F = draw((B, H, W, C), 810, dt)
    gamma, beta = wl.gn_affine(C, 12)
    ref = oracle.naive_groupnorm(G.f64(F), Gn, 1e-5, G.f64(gamma), G.f64(beta), P)
    junk = torch.randn(P, B, Gn, 2) * 100  # stale partials must be ignored
    y, _ = G.groupnorm(F, junk, Gn, 1e-5, gamma, beta, P, band_local=True)
    G.assert_rms_close(G.f64(y), ref, G.TOL[dt], "band-local groupnorm")
    y2, _ = G.groupnorm(F, None, Gn, 1e-5, gamma, beta, P, band_local=True)
    G.assert_rms_close(G.f64(y2), ref, G.TOL[dt], "band-local groupnorm, no stale state")


def test_band_local_single_pass_groupnorm(cuda_device):
    B, H, W, Ci, Co, P, Gn = 1, 16, 40, 64, 160, 4, 32
    F = draw((B, H, W, Ci), 820, BF16)
    Wt = wl.conv_weight(Co, Ci, 821, "bf16")
    gamma, beta = wl.gn_affine(Co, 13)
    y, sums = G.conv_gn(F, None, Wt, None, P, Gn)
    d = G.gn_desc(y, Gn, 1e-5, P, band_local=True)
    g = torch.empty_like(y)
    st = torch.empty((P, B, Gn, 2), device="cuda")
    G.dpp.dpp_groupnorm_apply(d, y, None, sums, st, G.cuda(gamma), G.cuda(beta), g)
    ref = oracle.naive_groupnorm(G.f64(y), Gn, 1e-5, G.f64(gamma), G.f64(beta), P)
    G.assert_rms_close(G.f64(g), ref, G.TOL[BF16], "band-local single-pass groupnorm")


@pytest.mark.parametrize("B,H,W,heads,P,dt", [
    (2, 6, 20, 2, 3, BF16),    # 40 tokens per band: ragged against the 128-key tile
    (1, 16, 32, 4, 4, BF16),   # 128 tokens per band, 4 heads
    (1, 12, 12, 2, 3, F32),    # SIMT attention
])
def test_band_local_self_attention(cuda_device, B, H, W, heads, P, dt):
    N, C = H * W, 64 * heads
    a = wl.AttnShape(B, H, W, C, heads, 64, P)
    F = draw((B, N, C), 830, dt)
    wts = wl.attn_weights(a, 14, "bf16" if dt == BF16 else "f32")
    y, _ = G.self_attn(F, wts, None, H, W, heads, P, band_local=True)
    w64 = {k: G.f64(v) for k, v in wts.items()}
    ref = oracle.naive_self_attention(G.f64(F), w64["wq"], w64["wk"], w64["wv"], w64["wo"],
                                      heads, P)
    # Attention over a single band of few keys gives peaky outputs, and the
    # bound is relative to the output's RMS: rounding the exact output to
    # bf16 alone can use most of it (2.2 % of RMS for some 128-key draws).
    # The cases here leave room: check that before judging the kernel.
    if dt == BF16:
        floor = np.abs(G.to_storage(ref, BF16) - ref).max() / np.sqrt(np.mean(ref ** 2))
        assert floor < 0.75 * G.TOL[dt], f"bf16 rounding alone is {floor:.4f} of RMS"
    G.assert_rms_close(G.f64(y), ref, G.TOL[dt], "band-local self-attention")
    # tokens outside band 0 never reach band 0's output; kv_prev is ignored
    Np = N // P
    F2 = F.clone()
    F2[:, Np:] = draw((B, N - Np, C), 831, dt)
    kv_junk = torch.randn(B, N, 2, C, device="cuda").to(G.KV_DTYPE[dt])
    y2, _ = G.self_attn(F2, wts, kv_junk, H, W, heads, P, band_local=True)
    assert torch.equal(y2[:, :Np], y[:, :Np])
    assert G.dpp.dpp_device_status() == G.dpp.DPP_OK
