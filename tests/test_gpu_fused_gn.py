"""Conv with GroupNorm sums in its epilogue (dpp_conv3x3_gn) followed by the
single-pass GroupNorm (dpp_groupnorm_apply), against the fp64 oracle and the
unfused entry points on the same seeded inputs.

The fused conv must store exactly what dpp_conv3x3 stores; its band sums must
match the fp64 partials of that stored output; the GroupNorm built on them
must match the oracle's displaced GroupNorm within the bf16 bound and agree
with dpp_groupnorm.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import gpu_ops as G

pytestmark = pytest.mark.gpu

BF16 = torch.bfloat16

FUSED_CASES = [  # (B, H, W, Ci, Co, P, groups)
    (2, 12, 20, 32, 48, 3, 8),      # ragged tiles; 6 channels per group
    (1, 16, 24, 64, 80, 4, 16),     # 5 channels per group: groups straddle 32-channel chunks
    (1, 8, 200, 64, 160, 2, 32),    # two 128-pixel segments per row, the second ragged
    (2, 16, 16, 64, 320, 4, 32),    # two N tiles of 160 channels
]


def _inputs(B, H, W, Ci, Co, seed):
    F = wl.normal((B, H, W, Ci), seed, dtype="bf16")
    S = wl.perturbed(F, seed + 1, 0.05)
    Wt = wl.conv_weight(Co, Ci, seed + 2, "bf16")
    return F, S, Wt


@pytest.mark.parametrize("B,H,W,Ci,Co,P,Gn", FUSED_CASES)
def test_fused_conv_stores_the_same_output_and_its_band_sums(cuda_device, B, H, W, Ci, Co, P,
                                                             Gn):
    F, S, Wt = _inputs(B, H, W, Ci, Co, 700)
    bias = wl.normal((Co,), 703)
    y_ref = G.conv(F, S, Wt, bias, P)
    y, sums = G.conv_gn(F, S, Wt, bias, P, Gn)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    parts = oracle.groupnorm_partials(G.f64(y), Gn, P)  # [P, B, G, 2] of the stored output
    n = H // P * W * Co // Gn
    got = sums.cpu().numpy()
    np.testing.assert_allclose(got[..., 0], parts[..., 0], rtol=0, atol=1e-5 * n)
    np.testing.assert_allclose(got[..., 1], parts[..., 1], rtol=1e-5)


@pytest.mark.parametrize("B,H,W,Ci,Co,P,Gn", FUSED_CASES)
def test_single_pass_groupnorm_matches_oracle_and_two_pass_entry_point(cuda_device, B, H, W, Ci,
                                                                        Co, P, Gn):
    F, S, Wt = _inputs(B, H, W, Ci, Co, 710)
    gamma, beta = wl.gn_affine(Co, 11)
    # step t-1 (synchronous): the stale conv output and its published partials
    yS = G.conv(S, None, Wt, None, P)
    _, st_prev = G.groupnorm(yS, None, Gn, 1e-5, gamma, beta, P)
    # step t (displaced): fused conv + single-pass GroupNorm
    y, sums = G.conv_gn(F, S, Wt, None, P, Gn)
    g, st_next = G.groupnorm_apply(y, st_prev, sums, Gn, 1e-5, gamma, beta, P)
    g2, st2 = G.groupnorm(y, st_prev, Gn, 1e-5, gamma, beta, P)
    ref = oracle.displaced_groupnorm(G.f64(y), G.f64(yS), Gn, 1e-5, G.f64(gamma), G.f64(beta), P)
    G.assert_rms_close(G.f64(g), ref, G.TOL[BF16], "single-pass groupnorm")
    G.assert_rms_close(G.f64(g), G.f64(g2), G.TOL[BF16], "single-pass vs two-pass")
    np.testing.assert_allclose(st_next.cpu().numpy(), sums.cpu().numpy().astype(np.float32),
                               rtol=0, atol=0)
    np.testing.assert_allclose(st_next.cpu().numpy()[..., 1], st2.cpu().numpy()[..., 1],
                               rtol=1e-5)
    # synchronous step: statistics of the whole image
    g0, _ = G.groupnorm_apply(y, None, sums, Gn, 1e-5, gamma, beta, P)
    ref0 = oracle.groupnorm(G.f64(y), Gn, 1e-5, G.f64(gamma), G.f64(beta))
    G.assert_rms_close(G.f64(g0), ref0, G.TOL[BF16], "single-pass groupnorm, synchronous")
    # in place
    yc = y.clone()
    g3, _ = G.groupnorm_apply(yc, st_prev, sums, Gn, 1e-5, gamma, beta, P, y=yc)
    assert torch.equal(g3, g)
    assert G.dpp.dpp_device_status() == G.dpp.DPP_OK


def test_fused_path_on_the_3840px_latent(cuda_device):
    """The bench's conv -> GroupNorm at full size: band sums of every band
    against fp64 sums of the stored output, and the normalised output on the
    first and last row of three bands against the oracle."""
    w = wl.WORKLOADS["sdxl_3840_cfg"]
    c = w.conv
    shape = (c.B, c.H, c.W, c.C)
    F = wl.normal(shape, wl.seed_of(w.index, 0, wl.T_FRESH), dtype=w.dtype)
    S = wl.perturbed(F, wl.seed_of(w.index, 1, wl.T_STALE_NOISE), w.stale_scale)
    Wt = wl.conv_weight(c.C, c.C, wl.seed_of(w.index, 0, wl.T_CONV_W), w.dtype)
    gamma, beta = wl.gn_affine(c.C, w.index)
    yS = G.conv(S, None, Wt, None, c.P)
    _, st_prev = G.groupnorm(yS, None, w.groups, w.eps, gamma, beta, c.P)
    y, sums = G.conv_gn(F, S, Wt, None, c.P, w.groups)
    g, _ = G.groupnorm_apply(y, st_prev, sums, w.groups, w.eps, gamma, beta, c.P)
    y64 = G.f64(y)
    parts = oracle.groupnorm_partials(y64, w.groups, c.P)
    n = c.H // c.P * c.W * c.C // w.groups
    got = sums.cpu().numpy()
    np.testing.assert_allclose(got[..., 0], parts[..., 0], rtol=0, atol=1e-5 * n)
    np.testing.assert_allclose(got[..., 1], parts[..., 1], rtol=1e-5)
    Hp = c.H // c.P
    bands = [0, 3, 7]
    rows = sorted({r for p in bands for r in (p * Hp, (p + 1) * Hp - 1)})
    ref = oracle.displaced_groupnorm(y64, G.f64(yS), w.groups, w.eps, G.f64(gamma),
                                     G.f64(beta), c.P, bands=bands)
    G.assert_rms_close(G.f64(g[:, rows]), ref[:, rows], G.TOL[BF16], "3840px single-pass GN")
