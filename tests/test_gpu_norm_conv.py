"""GroupNorm -> SiLU applied by the conv as it loads its input: the band sums
(dpp_groupnorm_sums), the per-band affine (dpp_groupnorm_affine), the
normalising conv (dpp_conv3x3_norm) and the halo-row refresh
(dpp_refresh_halo), against the oracle.

The oracle side is the unfused composition the pages describe: a displaced
GroupNorm, SiLU, then a displaced conv whose stale input is the previous
step's normalised tensor.  The GPU side keeps the previous step's
un-normalised input and affine instead and normalises on load, so a match
also shows that the halo rows are normalised as the previous step's
GroupNorm normalised them.  Two steps throughout: the synchronous one (no
stale state) and a displaced one.
"""
import numpy as np
import pytest
import torch

import displaced_patch_parallelism_02_b300 as dpp
import oracle
import oracle.blocks as OB
import workloads as wl
from tests import gpu_ops as G

pytestmark = pytest.mark.gpu

BF16, F32, F64 = torch.bfloat16, torch.float32, torch.float64
SILU, NONE = dpp.DPP_ACT_SILU, dpp.DPP_ACT_NONE


def draw(shape, seed, std=1.0, mean=0.0, dt="bf16"):
    return wl.normal(shape, seed, std=std, mean=mean, dtype=dt)


def gn_sums(x, Gr, P):
    x = G.cuda(x)
    B = x.shape[0]
    sums = torch.empty((P, B, Gr, 2), dtype=F64, device="cuda")
    dpp.dpp_groupnorm_sums(G.gn_desc(x, Gr, 1e-5, P), x, sums)
    return sums


def affine(x_shape, sums, stats_prev, Gr, eps, gamma, beta, P, band_local=False,
           dt=BF16):
    B, H, W, C = x_shape
    d = dpp.dpp_gn_desc(B, H, W, C, Gr, P, eps, G.CODES[dt], int(band_local), 0)
    aff = torch.empty((P, B, C, 2), dtype=F32, device="cuda")
    st = torch.empty((P, B, Gr, 2), dtype=F32, device="cuda")
    dpp.dpp_groupnorm_affine(d, sums, stats_prev, st, G.cuda(gamma), G.cuda(beta), aff)
    return aff, st


def norm_conv(x, stale, aff, aff_prev, w, bias, P, act=SILU, halo=dpp.DPP_HALO_STALE,
              Gout=0, y_init=None):
    x = G.cuda(x)
    stale = G.cuda(stale) if stale is not None and stale.device.type == "cpu" else stale
    B, H, W, Ci = x.shape
    Co = w.shape[0]
    wd = G.cuda(w.permute(0, 2, 3, 1))
    y = (torch.empty((B, H, W, Co), dtype=BF16, device="cuda") if y_init is None
         else y_init.to("cuda", copy=True).contiguous())
    sums = torch.empty((P, B, Gout, 2), dtype=F64, device="cuda") if Gout else None
    d = dpp.dpp_conv_desc(B, H, W, Ci, Co, P, dpp.DPP_BF16, int(halo), int(y_init is not None))
    dpp.dpp_conv3x3_norm(d, x, stale, aff, aff_prev, act, wd, G.cuda(bias), y, Gout, sums)
    return y, sums


def apply_table(x64, aff, P):
    """y = x * a + s with band p's row of the affine table on band p's rows."""
    a = aff.cpu().numpy().astype(np.float64)  # [P, B, C, 2]
    B, H, W, C = x64.shape
    Hp = H // P
    y = np.empty_like(x64)
    for p in range(P):
        sl = slice(p * Hp, (p + 1) * Hp)
        y[:, sl] = x64[:, sl] * a[p, :, None, None, :, 0] + a[p, :, None, None, :, 1]
    return y


def act_of(y, act):
    return OB.silu(y) if act == SILU else y


# ---------------------------------------------------------------- band sums
@pytest.mark.parametrize("B,H,W,C,Gr,P,dt", [
    (2, 16, 20, 64, 8, 4, "bf16"),
    (1, 12, 30, 320, 32, 3, "bf16"),   # 10 channels a group: vectors straddle groups
    (2, 8, 12, 64, 4, 2, "f32"),
    (1, 6, 7, 8, 8, 1, "bf16"),        # one channel a group, one band
])
def test_groupnorm_sums_match_the_partials(cuda_device, B, H, W, C, Gr, P, dt):
    x = draw((B, H, W, C), 900 + C, std=1.5, mean=0.3, dt=dt)
    sums = gn_sums(x, Gr, P)
    ref = oracle.groupnorm_partials(G.f64(x), Gr, P)
    np.testing.assert_allclose(sums.cpu().numpy(), ref, rtol=1e-5,
                               atol=1e-5 * np.abs(ref).max())


# ---------------------------------------------------------- affine per band
@pytest.mark.parametrize("mean", [0.0, 30.0])
def test_affine_applied_per_band_is_the_displaced_groupnorm(cuda_device, mean):
    # the variance is E[x^2] - mean^2 from fp32 partial sums: a group mean of
    # 30 sigma costs ~10 of fp32's 24 bits, so that case is held to the bf16
    # parity bar, the centred case to 1e-4
    tol = 1e-4 if mean == 0.0 else G.TOL[BF16]
    B, H, W, C, Gr, P, eps = 2, 16, 12, 64, 8, 4, 1e-5
    F = draw((B, H, W, C), 910, std=1.0, mean=mean)
    S = wl.perturbed(F, 911, 0.3)
    gamma, beta = draw((C,), 912, 0.1, 1.0, "f32"), draw((C,), 913, 0.1, 0.0, "f32")
    g64, b64 = G.f64(gamma), G.f64(beta)
    aff0, st0 = affine(F.shape, gn_sums(S, Gr, P), None, Gr, eps, gamma, beta, P)
    aff1, st1 = affine(F.shape, gn_sums(F, Gr, P), st0, Gr, eps, gamma, beta, P)
    # the synchronous step: every band the statistics of the whole image
    G.assert_rms_close(apply_table(G.f64(S), aff0, P),
                       oracle.groupnorm(G.f64(S), Gr, eps, g64, b64), tol, "sync affine")
    G.assert_rms_close(apply_table(G.f64(F), aff1, P),
                       oracle.displaced_groupnorm(G.f64(F), G.f64(S), Gr, eps, g64, b64, P),
                       tol, "displaced affine")
    # the published state is the band's fresh partials
    np.testing.assert_allclose(st1.cpu().numpy(), oracle.groupnorm_partials(G.f64(F), Gr, P),
                               rtol=1e-5, atol=1e-5 * float(np.abs(G.f64(F)).max()))
    # naive patches: each band's own statistics
    aff_n, _ = affine(F.shape, gn_sums(F, Gr, P), None, Gr, eps, gamma, beta, P, band_local=True)
    G.assert_rms_close(apply_table(G.f64(F), aff_n, P),
                       oracle.naive_groupnorm(G.f64(F), Gr, eps, g64, b64, P),
                       tol, "band-local affine")


# ----------------------------------------------------------- normalising conv
def two_steps(B, H, W, Ci, Co, P, Gr, seed, act=SILU, with_bias=True, Gout=0, y_init=None,
              mean=0.0):
    """Runs the synchronous and the displaced step on the GPU; returns the
    inputs, the GPU outputs and the oracle's unfused composition."""
    eps = 1e-5
    S = draw((B, H, W, Ci), seed, std=1.3, mean=mean)
    F = wl.perturbed(S, seed + 1, 0.4)
    w = wl.conv_weight(Co, Ci, seed + 2, "bf16")
    bias = draw((Co,), seed + 3, 0.1, 0.0, "f32") if with_bias else None
    gamma, beta = draw((Ci,), seed + 4, 0.1, 1.0, "f32"), draw((Ci,), seed + 5, 0.1, 0.0, "f32")
    aff0, st0 = affine(S.shape, gn_sums(S, Gr, P), None, Gr, eps, gamma, beta, P)
    y0, _ = norm_conv(S, None, aff0, None, w, bias, P, act)
    aff1, _ = affine(F.shape, gn_sums(F, Gr, P), st0, Gr, eps, gamma, beta, P)
    y1, sums = norm_conv(F, S, aff1, aff0, w, bias, P, act, Gout=Gout, y_init=y_init)
    W64 = G.f64(w)
    b64 = None if bias is None else G.f64(bias)
    g0 = act_of(oracle.groupnorm(G.f64(S), Gr, eps, G.f64(gamma), G.f64(beta)), act)
    g1 = act_of(oracle.displaced_groupnorm(G.f64(F), G.f64(S), Gr, eps, G.f64(gamma),
                                           G.f64(beta), P), act)
    ref0 = oracle.displaced_conv3x3(g0, g0, W64, b64, P)
    ref1 = oracle.displaced_conv3x3(g1, g0, W64, b64, P)
    if y_init is not None:
        ref1 = ref1 + G.f64(y_init)
    return dict(S=S, F=F, w=w, bias=bias, gamma=gamma, beta=beta, st0=st0, aff0=aff0,
                aff1=aff1, y0=y0, y1=y1, sums=sums, ref0=ref0, ref1=ref1, eps=eps)


@pytest.mark.parametrize("B,H,W,Ci,Co,P,Gr", [
    (2, 12, 200, 96, 96, 3, 8),      # W: a 128-pixel tile + 72; C_in: 64 + 32; one ragged N tile
    (1, 16, 64, 320, 320, 4, 32),    # N tile 160 (2 tiles), 5 channel blocks
    (2, 8, 130, 64, 64, 2, 16),      # a 2-pixel last segment; N tile 64
    (1, 8, 40, 128, 640, 2, 32),     # 4 N tiles of 160
    (1, 8, 24, 64, 64, 8, 8),        # one row per band: every input row is a halo row
])
def test_norm_conv_two_steps_match_the_unfused_oracle(cuda_device, B, H, W, Ci, Co, P, Gr):
    r = two_steps(B, H, W, Ci, Co, P, Gr, 920 + Ci + Co)
    G.assert_rms_close(G.f64(r["y0"]), r["ref0"], G.TOL[BF16], "synchronous step")
    G.assert_rms_close(G.f64(r["y1"]), r["ref1"], G.TOL[BF16], "displaced step")
    assert dpp.dpp_device_status() == dpp.DPP_OK


def test_norm_conv_without_activation_and_without_bias(cuda_device):
    r = two_steps(2, 12, 40, 64, 128, 3, 16, 940, act=NONE, with_bias=False)
    G.assert_rms_close(G.f64(r["y1"]), r["ref1"], G.TOL[BF16], "affine only")


def test_norm_conv_large_group_means(cuda_device):
    # group means of ~30 sigma: the statistics stay accurate (fp64 totals)
    r = two_steps(1, 8, 64, 64, 64, 2, 8, 945, mean=30.0)
    G.assert_rms_close(G.f64(r["y1"]), r["ref1"], G.TOL[BF16], "large means")


def test_norm_conv_accumulates_and_sums_the_stored_output(cuda_device):
    B, H, W, C, P, Gr = 2, 8, 40, 128, 2, 32
    res = draw((B, H, W, C), 950)
    r = two_steps(B, H, W, C, C, P, Gr, 951, Gout=Gr, y_init=res)
    G.assert_rms_close(G.f64(r["y1"]), r["ref1"], G.TOL[BF16], "accumulate")
    ref = oracle.groupnorm_partials(G.f64(r["y1"]), Gr, P)
    np.testing.assert_allclose(r["sums"].cpu().numpy(), ref, rtol=1e-5,
                               atol=1e-3 * np.abs(ref).max())


def test_norm_conv_agrees_with_the_unfused_library_path(cuda_device):
    """The same step through dpp_groupnorm_apply (act SiLU, the normalised
    tensor stored) and dpp_conv3x3 with the previous step's normalised tensor
    as stale: the inputs of the two convs differ only in the SiLU's
    evaluation and its bf16 rounding."""
    B, H, W, C, P, Gr = 2, 16, 72, 64, 4, 16
    r = two_steps(B, H, W, C, C, P, Gr, 960)
    sums0, sums1 = gn_sums(r["S"], Gr, P), gn_sums(r["F"], Gr, P)
    g0, _ = G.groupnorm_apply(r["S"], None, sums0, Gr, r["eps"], r["gamma"], r["beta"], P,
                              act=SILU)
    g1, _ = G.groupnorm_apply(r["F"], r["st0"], sums1, Gr, r["eps"], r["gamma"], r["beta"], P,
                              act=SILU)
    y_unfused = G.conv(g1, g0, r["w"], r["bias"], P)
    got, want = G.f64(r["y1"]), G.f64(y_unfused)
    # two bf16 outputs rounded from slightly different sums: at most one ulp
    # of the largest value (+0.5 % of RMS) apart, and 0.2 % of RMS overall
    rms = float(np.sqrt(np.mean(want ** 2)))
    err = float(np.max(np.abs(got - want)))
    assert err <= 2 * G.bf16_half_ulp_max(want) + 5e-3 * rms, (err, rms)
    assert float(np.sqrt(np.mean((got - want) ** 2))) <= 2e-3 * rms


@pytest.mark.parametrize("halo", [dpp.DPP_HALO_FRESH, dpp.DPP_HALO_ZERO])
def test_norm_conv_fresh_and_zero_halo(cuda_device, halo):
    B, H, W, C, P, Gr, eps = 2, 12, 40, 64, 3, 8, 1e-5
    F = draw((B, H, W, C), 970, 1.2)
    w = wl.conv_weight(C, C, 971, "bf16")
    gamma, beta = draw((C,), 972, 0.1, 1.0, "f32"), draw((C,), 973, 0.1, 0.0, "f32")
    naive = halo == dpp.DPP_HALO_ZERO
    aff, _ = affine(F.shape, gn_sums(F, Gr, P), None, Gr, eps, gamma, beta, P, band_local=naive)
    y, _ = norm_conv(F, None, aff, None, w, None, P, SILU, halo=halo)
    if naive:  # naive patches: band-local statistics, zero-padded bands
        g = OB.silu(oracle.naive_groupnorm(G.f64(F), Gr, eps, G.f64(gamma), G.f64(beta), P))
        ref = oracle.naive_conv3x3(g, G.f64(w), None, P)
    else:
        g = OB.silu(oracle.groupnorm(G.f64(F), Gr, eps, G.f64(gamma), G.f64(beta)))
        ref = oracle.displaced_conv3x3(g, g, G.f64(w), None, P, first_layer=True)
    G.assert_rms_close(G.f64(y), ref, G.TOL[BF16], f"halo {halo}")


def test_norm_conv_single_band(cuda_device):
    r = two_steps(1, 10, 50, 64, 64, 1, 8, 980)
    G.assert_rms_close(G.f64(r["y1"]), r["ref1"], G.TOL[BF16], "P = 1")


# ------------------------------------------------------------- halo refresh
@pytest.mark.parametrize("B,H,W,C,P", [(2, 12, 20, 64, 3), (1, 16, 8, 128, 4), (3, 8, 5, 16, 8),
                                       (2, 9, 4, 8, 1)])
def test_refresh_halo_copies_exactly_the_halo_rows(cuda_device, B, H, W, C, P):
    fresh = draw((B, H, W, C), 990).to("cuda")
    stale0 = draw((B, H, W, C), 991)
    stale = stale0.to("cuda")
    dpp.dpp_refresh_halo(fresh, stale, B, H, W * C * 2, P)
    torch.cuda.synchronize()
    Hp = H // P
    rows = sorted({r for k in range(1, P) for r in (k * Hp - 1, k * Hp)})
    want = stale0.clone()
    want[:, rows] = fresh.cpu()[:, rows]
    assert torch.equal(stale.cpu(), want)


# ------------------------------------------------------ 3840px latent, sampled
def test_sdxl_3840_norm_conv_sampled_rows(cuda_device):
    """The ResNet block's GroupNorm -> SiLU -> conv at the 3840px latent
    (2 x 480 x 480 x 320, 8 bands): the oracle composes the displaced
    GroupNorm over the whole latent and evaluates the conv on the first and
    last row of every band (the rows that read the stale halo) plus one
    interior row per band."""
    w = wl.WORKLOADS["sdxl_3840_cfg"]
    c = w.conv
    shape = (c.B, c.H, c.W, c.C)
    S = wl.normal(shape, wl.seed_of(w.index, 0, wl.T_FRESH), dtype=w.dtype)
    F = wl.perturbed(S, wl.seed_of(w.index, 1, wl.T_STALE_NOISE), w.stale_scale)
    Wt = wl.conv_weight(c.C, c.C, wl.seed_of(w.index, 0, wl.T_CONV_W), w.dtype)
    gamma, beta = wl.gn_affine(c.C, w.index)
    Sd, Fd = S.to("cuda"), F.to("cuda")
    aff0, st0 = affine(shape, gn_sums(Sd, w.groups, c.P), None, w.groups, w.eps, gamma, beta,
                       c.P)
    aff1, _ = affine(shape, gn_sums(Fd, w.groups, c.P), st0, w.groups, w.eps, gamma, beta, c.P)
    y, _ = norm_conv(Fd, Sd, aff1, aff0, Wt, None, c.P, SILU)
    assert dpp.dpp_device_status() == dpp.DPP_OK
    Hp = c.H // c.P
    rng = np.random.default_rng(3840)
    rows = sorted({r for p in range(c.P)
                   for r in (p * Hp, (p + 1) * Hp - 1, int(rng.integers(p * Hp + 1,
                                                                         (p + 1) * Hp - 1)))})
    yr = G.f64(y[:, rows])
    del y, Fd, Sd
    g64, b64 = G.f64(gamma), G.f64(beta)
    S64 = G.f64(S)
    g0 = OB.silu(oracle.groupnorm(S64, w.groups, w.eps, g64, b64))
    g1 = OB.silu(oracle.displaced_groupnorm(G.f64(F), S64, w.groups, w.eps, g64, b64, c.P))
    del S64
    ref = oracle.displaced_conv3x3(g1, g0, G.f64(Wt), None, c.P, out_rows=rows)
    G.assert_rms_close(yr, ref, G.TOL[BF16], "3840px norm conv")
