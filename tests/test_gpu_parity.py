"""GPU parity at sizes the oracle finishes in seconds: every op through the C
ABI against the fp64 oracle on the same seeded inputs, spanning several tiles
with ragged tails, plus the bit-exact and invariance checks of the method.

Tolerances (max-abs error relative to the output RMS): 1e-4 for fp32, 2e-2 for
bf16 storage with fp32 accumulation.  Refresh and indexing are bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import gpu_ops as G

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16


def draw(shape, seed, dt, std=1.0):
    return wl.normal(shape, seed, std=std, dtype="bf16" if dt == BF16 else "f32")


# ------------------------------------------------------------------ refresh
@pytest.mark.parametrize("shape,P,dt", [((2, 12, 5, 16), 4, BF16), ((1, 8, 3, 4), 2, F32),
                                        ((3, 40, 2, 64), 8, BF16)])
@pytest.mark.parametrize("mask", [None, 0b0101, 0b1, 0b10])
def test_refresh_bit_exact(cuda_device, shape, P, dt, mask):
    fresh = draw(shape, 11, dt).cuda()
    stale = draw(shape, 12, dt).cuda()
    want = stale.clone()
    Hp = shape[1] // P
    for p in range(P):
        if mask is None or (mask >> p) & 1:
            want[:, p * Hp:(p + 1) * Hp] = fresh[:, p * Hp:(p + 1) * Hp]
    row_bytes = shape[2] * shape[3] * fresh.element_size()
    G.dpp.dpp_refresh_stale(fresh, stale, shape[0], shape[1], row_bytes, P,
                            (1 << 64) - 1 if mask is None else mask)
    torch.cuda.synchronize()
    assert torch.equal(stale.view(torch.int16 if dt == BF16 else torch.int32),
                       want.view(torch.int16 if dt == BF16 else torch.int32))


def test_refresh_of_gn_stats_and_kv_state(cuda_device):
    P, B, Gs = 4, 2, 32
    fresh = torch.randn(P, B, Gs, 2, device="cuda")
    stale = torch.randn(P, B, Gs, 2, device="cuda")
    want = fresh.clone()
    G.dpp.dpp_refresh_stale(fresh, stale, 1, P, B * Gs * 2 * 4, P)
    kvf = draw((2, 120, 2, 128), 3, BF16).cuda()
    kvs = draw((2, 120, 2, 128), 4, BF16).cuda()
    kv_want = kvs.clone()
    kv_want[:, 40:80] = kvf[:, 40:80]
    G.dpp.dpp_refresh_stale(kvf, kvs, 2, 120, 2 * 128 * 2, 3, 0b010)
    torch.cuda.synchronize()
    assert torch.equal(stale, want)
    assert torch.equal(kvs.view(torch.int16), kv_want.view(torch.int16))


# ---------------------------------------------------------------------- CFG
@pytest.mark.parametrize("n", [4 * 480 * 480, 1001, 3, 64 * 1024 + 5])
def test_cfg_matches_oracle(cuda_device, n):
    u, c = wl.normal((n,), 21), wl.normal((n,), 22)
    out, sums, ws = G.cfg(u, c, 7.5)
    ref_out, ref_sums = oracle.cfg_combine(G.f64(u), G.f64(c), 7.5)
    G.assert_rms_close(G.f64(out), ref_out, 1e-4, "cfg out")
    np.testing.assert_allclose(sums.cpu().numpy(), ref_sums, rtol=1e-5)
    assert int(ws[:4].view(torch.int32).item()) == 0  # completion counter left at zero


def test_cfg_bit_reproducible_and_in_place(cuda_device):
    n = 4 * 480 * 480
    u, c = wl.normal((n,), 31), wl.normal((n,), 32)
    o1, s1, ws = G.cfg(u, c, 7.5)
    o2, s2, _ = G.cfg(u, c, 7.5, ws=ws)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    ud = u.cuda()
    o3, s3, _ = G.cfg(ud, c, 7.5, out=ud)  # out aliases eps_u
    assert torch.equal(o3, o1) and torch.equal(s3, s1)


def test_cfg_closed_forms(cuda_device):
    n = 10007
    u = wl.normal((n,), 41)
    out, sums, _ = G.cfg(u, u, 7.5)
    assert torch.equal(out.cpu(), u) and sums[0].item() == 0.0
    out0, _, _ = G.cfg(u, wl.normal((n,), 42), 0.0)
    assert torch.equal(out0.cpu(), u)  # s = 0 returns eps_u exactly
    for k in (0.5, -0.25):
        _, s, _ = G.cfg(u, (1 + k) * u, 7.5)
        assert abs(s[0].item() / s[1].item() - abs(k)) < 1e-5


# --------------------------------------------------------------------- conv
CONV_CASES = [  # (B, H, W, Ci, Co, P, dtype, bias)
    (1, 32, 32, 64, 64, 2, F32, False),   # the tiny fp32 workload
    (2, 12, 20, 32, 48, 3, BF16, True),   # ragged tiles, bias
    (1, 16, 24, 64, 80, 4, BF16, False),
    (2, 8, 6, 8, 16, 8, F32, True),       # one row per band
]


@pytest.mark.parametrize("B,H,W,Ci,Co,P,dt,use_bias", CONV_CASES)
@pytest.mark.parametrize("stale_scale", [0.05, None])  # None: independent stale draw
def test_conv_matches_oracle(cuda_device, B, H, W, Ci, Co, P, dt, use_bias, stale_scale):
    F = draw((B, H, W, Ci), 100, dt)
    S = wl.perturbed(F, 101, stale_scale) if stale_scale else draw((B, H, W, Ci), 101, dt)
    Wt = wl.conv_weight(Co, Ci, 102, "bf16" if dt == BF16 else "f32")
    bias = wl.normal((Co,), 103) if use_bias else None
    y = G.conv(F, S, Wt, bias, P)
    ref = oracle.displaced_conv3x3(G.f64(F), G.f64(S), G.f64(Wt),
                                   None if bias is None else G.f64(bias), P)
    G.assert_rms_close(G.f64(y), ref, G.TOL[dt], "conv")
    # synchronous step (no stale buffer) is the full-image layer
    y0 = G.conv(F, None, Wt, bias, P)
    ref0 = oracle.conv3x3(G.f64(F), G.f64(Wt), None if bias is None else G.f64(bias))
    G.assert_rms_close(G.f64(y0), ref0, G.TOL[dt], "conv sync")


def test_conv_reads_only_halo_rows_of_stale(cuda_device):
    B, H, W, C, P = 1, 16, 24, 64, 4
    F, S = draw((B, H, W, C), 1, BF16), draw((B, H, W, C), 2, BF16)
    Wt = wl.conv_weight(C, C, 3, "bf16")
    base = G.conv(F, S, Wt, None, P)
    for p in range(P):
        S2 = S.clone()
        S2[:, p * 4:(p + 1) * 4] += 10.0
        y = G.conv(F, S2, Wt, None, P)
        assert torch.equal(y[:, p * 4:(p + 1) * 4], base[:, p * 4:(p + 1) * 4])
    # rows without a stale neighbour equal the synchronous conv bit for bit
    sync = G.conv(F, None, Wt, None, P)
    inner = [h for h in range(H) if h % 4 not in (0, 3) or h in (0, H - 1)]
    assert torch.equal(base[:, inner], sync[:, inner])
    # and every band-edge row differs from it (the halo is really stale)
    for h in range(H):
        if h % 4 in (0, 3) and h not in (0, H - 1):
            assert not torch.equal(base[:, h], sync[:, h])


def test_conv_first_layer_ignores_stale(cuda_device):
    F, S = draw((1, 8, 16, 32), 5, BF16), draw((1, 8, 16, 32), 6, BF16)
    Wt = wl.conv_weight(32, 32, 7, "bf16")
    y = G.conv(F, S, Wt, None, 4, halo=G.dpp.DPP_HALO_FRESH)
    assert torch.equal(y, G.conv(F, None, Wt, None, 4))


# ---------------------------------------------------------------- groupnorm
GN_CASES = [  # (B, H, W, C, G, P, dtype)
    (1, 32, 32, 64, 32, 2, F32),   # the tiny fp32 workload
    (2, 12, 7, 40, 8, 3, BF16),    # 5 channels per group: vectors straddle groups
    (1, 16, 16, 320, 32, 4, BF16),
    (2, 8, 5, 16, 4, 8, F32),
]


@pytest.mark.parametrize("B,H,W,C,Gn,P,dt", GN_CASES)
@pytest.mark.parametrize("stale_scale", [0.05, None])
def test_groupnorm_two_steps_match_oracle(cuda_device, B, H, W, C, Gn, P, dt, stale_scale):
    """Step t-1 runs on S (synchronous); step t on F with S's published
    partials as the stale state: output = oracle displaced GroupNorm(F, S)."""
    F = draw((B, H, W, C), 200, dt)
    S = wl.perturbed(F, 201, stale_scale) if stale_scale else draw((B, H, W, C), 201, dt, 2.0)
    gamma, beta = wl.gn_affine(C, 7)
    y_s, stats_s = G.groupnorm(S, None, Gn, 1e-5, gamma, beta, P)
    y, stats_f = G.groupnorm(F, stats_s, Gn, 1e-5, gamma, beta, P)
    ref = oracle.displaced_groupnorm(G.f64(F), G.f64(S), Gn, 1e-5, G.f64(gamma), G.f64(beta), P)
    G.assert_rms_close(G.f64(y), ref, G.TOL[dt], "gn displaced")
    ref_s = oracle.groupnorm(G.f64(S), Gn, 1e-5, G.f64(gamma), G.f64(beta))
    G.assert_rms_close(G.f64(y_s), ref_s, G.TOL[dt], "gn sync")
    n = H // P * W * C // Gn
    parts = oracle.groupnorm_partials(G.f64(F), Gn, P)
    np.testing.assert_allclose(stats_f.cpu().double().numpy()[..., 0], parts[..., 0],
                               rtol=0, atol=1e-4 * n ** 0.5 * 3)
    np.testing.assert_allclose(stats_f.cpu().double().numpy()[..., 1], parts[..., 1], rtol=1e-4)


def test_groupnorm_without_affine_unit_moments_and_in_place(cuda_device):
    F = draw((2, 16, 16, 320), 300, BF16, std=3.0) + 1.5
    F = F.to(BF16)
    y, _ = G.groupnorm(F, None, 32, 1e-5, None, None, 4)
    yg = G.f64(y).reshape(2, -1, 32, 10)
    assert np.abs(yg.mean(axis=(1, 3))).max() < 2e-2
    assert np.abs(yg.var(axis=(1, 3)) - 1).max() < 2e-2
    xd = G.cuda(F)
    y2, _ = G.groupnorm(xd, None, 32, 1e-5, None, None, 4, y=xd)  # in place
    assert torch.equal(y2, y)


def test_groupnorm_never_uses_own_band_of_stale_state(cuda_device):
    F, S = draw((1, 16, 8, 64), 1, BF16), draw((1, 16, 8, 64), 2, BF16)
    _, st = G.groupnorm(S, None, 32, 1e-5, None, None, 4)
    base, _ = G.groupnorm(F, st, 32, 1e-5, None, None, 4)
    for p in range(4):
        st2 = st.clone()
        st2[p] *= 3.0
        y, _ = G.groupnorm(F, st2, 32, 1e-5, None, None, 4)
        assert torch.equal(y[:, 4 * p:4 * p + 4], base[:, 4 * p:4 * p + 4])
        assert not torch.equal(y, base)


@pytest.mark.parametrize("dt,lo,hi", [(BF16, 30.0, 100.0), (F32, 10.0, 20.0)])
def test_groupnorm_large_group_means(cuda_device, dt, lo, hi):
    """Groups whose mean is tens of standard deviations (a conv output with
    a large bias): the variance must not cancel away.  Every group gets its
    own mean in [lo, hi] (sign alternating), unit spread; synchronous step,
    then the displaced step on its published partials, against the oracle.
    The published state is fp32 (sum x, sum x^2), whose 2^-24 relative
    precision bounds the variance to about 6e-8 (mean / sd)^2: the fp32 case
    stays at means of 10-20 sd, inside the 1e-4 RMS bar."""
    B, H, W, C, Gn, P = 2, 16, 12, 320, 32, 4
    g = torch.Generator().manual_seed(404)
    means = (lo + (hi - lo) * torch.rand(Gn, generator=g)) * torch.tensor(
        [(-1.0) ** k for k in range(Gn)])
    shift = means.repeat_interleave(C // Gn)
    F = (draw((B, H, W, C), 405, F32) + shift).to(dt)
    S = (wl.perturbed(F.float(), 406, 0.05)).to(dt)
    gamma, beta = wl.gn_affine(C, 8)
    y_s, stats_s = G.groupnorm(S, None, Gn, 1e-5, gamma, beta, P)
    y, _ = G.groupnorm(F, stats_s, Gn, 1e-5, gamma, beta, P)
    ref_s = oracle.groupnorm(G.f64(S), Gn, 1e-5, G.f64(gamma), G.f64(beta))
    G.assert_rms_close(G.f64(y_s), ref_s, G.TOL[dt], "gn sync, large means")
    ref = oracle.displaced_groupnorm(G.f64(F), G.f64(S), Gn, 1e-5, G.f64(gamma), G.f64(beta), P)
    G.assert_rms_close(G.f64(y), ref, G.TOL[dt], "gn displaced, large means")


# ---------------------------------------------------------------- attention
ATTN_CASES = [  # (B, H, W, heads, P, dtype)
    (1, 32, 32, 1, 2, F32),     # the tiny fp32 workload
    (2, 6, 20, 2, 3, BF16),     # 40 tokens per band: ragged against every tile size
    (1, 16, 16, 4, 4, BF16),
    (1, 12, 12, 2, 3, F32),
    (1, 8, 10, 5, 2, BF16),     # C 320: each QKV weight block tiled 256 + 64 columns
]


@pytest.mark.parametrize("B,H,W,heads,P,dt", ATTN_CASES)
@pytest.mark.parametrize("stale_scale", [0.05, None])
def test_self_attn_two_steps_match_oracle(cuda_device, B, H, W, heads, P, dt, stale_scale):
    N, C = H * W, 64 * heads
    a = wl.AttnShape(B, H, W, C, heads, 64, P)
    F = draw((B, N, C), 400, dt)
    S = wl.perturbed(F, 401, stale_scale) if stale_scale else draw((B, N, C), 401, dt)
    wts = wl.attn_weights(a, 4, "bf16" if dt == BF16 else "f32")
    _, kv_s = G.self_attn(S, wts, None, H, W, heads, P)          # step t-1, synchronous
    y, kv_f = G.self_attn(F, wts, kv_s, H, W, heads, P)          # step t, displaced
    w64 = {k: G.f64(v) for k, v in wts.items()}
    ref = oracle.displaced_self_attention(G.f64(F), G.f64(S), w64["wq"], w64["wk"], w64["wv"],
                                          w64["wo"], heads, P)
    G.assert_rms_close(G.f64(y), ref, G.TOL[dt], "self-attn")
    kv_ref = oracle.kv_state(G.f64(F), w64["wk"], w64["wv"])
    G.assert_rms_close(G.f64(kv_f), kv_ref, G.TOL[dt], "kv_next")
    # the synchronous call is the full-image layer
    y0, _ = G.self_attn(F, wts, None, H, W, heads, P)
    ref0 = oracle.displaced_self_attention(G.f64(F), G.f64(F), w64["wq"], w64["wk"], w64["wv"],
                                           w64["wo"], heads, 1)
    G.assert_rms_close(G.f64(y0), ref0, G.TOL[dt], "self-attn sync")


def test_self_attn_own_band_of_stale_kv_unused(cuda_device):
    B, H, W, heads, P = 1, 8, 16, 2, 4
    N, C = H * W, 128
    a = wl.AttnShape(B, H, W, C, heads, 64, P)
    F, S = draw((B, N, C), 1, BF16), draw((B, N, C), 2, BF16)
    wts = wl.attn_weights(a, 5, "bf16")
    _, kv_s = G.self_attn(S, wts, None, H, W, heads, P)
    base, _ = G.self_attn(F, wts, kv_s, H, W, heads, P)
    Np = N // P
    for p in range(P):
        kv2 = kv_s.clone()
        kv2[:, p * Np:(p + 1) * Np] = 3.0
        y, _ = G.self_attn(F, wts, kv2, H, W, heads, P)
        assert torch.equal(y[:, p * Np:(p + 1) * Np], base[:, p * Np:(p + 1) * Np])
        assert not torch.equal(y, base)


@pytest.mark.parametrize("B,H,W,heads,n_ctx,c_ctx,dt", [
    (2, 4, 8, 2, 77, 256, BF16), (1, 8, 8, 1, 5, 64, F32), (1, 4, 30, 3, 77, 128, BF16)])
def test_cross_attn_matches_oracle(cuda_device, B, H, W, heads, n_ctx, c_ctx, dt):
    N, C = H * W, 64 * heads
    a = wl.AttnShape(B, H, W, C, heads, 64, 1, n_ctx, c_ctx)
    name = "bf16" if dt == BF16 else "f32"
    X = draw((B, N, C), 500, dt)
    ctx = wl.normal((B, n_ctx, c_ctx), 501, dtype=name)
    wts = wl.cross_weights(a, 6, name)
    y = G.cross_attn(X, ctx, wts, H, W, heads)
    w64 = {k: G.f64(v) for k, v in wts.items()}
    ref = oracle.cross_attention(G.f64(X), G.f64(ctx), w64["wq"], w64["wk"], w64["wv"],
                                 w64["wo"], heads)
    G.assert_rms_close(G.f64(y), ref, G.TOL[dt], "cross-attn")


@pytest.mark.parametrize("B,H,W,heads,n_ctx", [
    (2, 10, 30, 2, 1), (2, 10, 30, 2, 16), (2, 10, 30, 2, 17), (1, 10, 30, 2, 128),
    (2, 64, 80, 3, 77)])
def test_cross_attn_short_context_edges(cuda_device, B, H, W, heads, n_ctx):
    """The persistent core for keys that fit one tile: a single key, exact
    multiples of 16, one past, a full 128-key tile, query counts with a
    ragged last tile per image (stores clipped at each image's end), and
    more (image, head, query tile) items than SMs, so that a CTA walks
    several items and changes head and image on the way.  A softmax over a
    few keys is peaky, so the largest outputs sit far above the RMS: the bar
    is 2e-2 x RMS on top of the bf16 storage floor (half an ulp of the
    largest value), as for the chain's ops.  The tile-per-band core gives the
    same errors on these inputs."""
    N, C, c_ctx = H * W, 64 * heads, 96
    a = wl.AttnShape(B, H, W, C, heads, 64, 1, n_ctx, c_ctx)
    X = draw((B, N, C), 530, BF16)
    ctx = wl.normal((B, n_ctx, c_ctx), 531, dtype="bf16")
    wts = wl.cross_weights(a, 8, "bf16")
    y = G.cross_attn(X, ctx, wts, H, W, heads)
    w64 = {k: G.f64(v) for k, v in wts.items()}
    ref = oracle.cross_attention(G.f64(X), G.f64(ctx), w64["wq"], w64["wk"], w64["wv"],
                                 w64["wo"], heads)
    G.assert_close_over_bf16_floor(G.f64(y), ref, G.TOL[BF16], "cross-attn, short context")


@pytest.mark.parametrize("dt", [BF16, F32])
def test_cross_attn_context_kv_once_per_prompt(cuda_device, dt):
    """The context's K/V projected once (dpp_cross_attn_kv) and reused by
    dpp_cross_attn_cached over several calls: bit-identical to
    dpp_cross_attn, which is the two parts back to back, and to the oracle
    within the bar."""
    B, H, W, heads, n_ctx, c_ctx = 2, 8, 12, 2, 77, 96
    N, C = H * W, 64 * heads
    a = wl.AttnShape(B, H, W, C, heads, 64, 1, n_ctx, c_ctx)
    name = "bf16" if dt == BF16 else "f32"
    ctx = G.cuda(wl.normal((B, n_ctx, c_ctx), 511, dtype=name))
    w = {k: G.cuda(v) for k, v in wl.cross_weights(a, 7, name).items()}
    d = G.dpp.dpp_attn_desc(B, H, W, C, heads, 64, 1, n_ctx, c_ctx, G.CODES[dt], 0, 0)
    kv = torch.empty((B, n_ctx, 2, C), dtype=G.KV_DTYPE[dt], device="cuda")
    G.dpp.dpp_cross_attn_kv(d, ctx, w["wk"], w["wv"], kv)
    nws = G.dpp.dpp_cross_attn_cached_workspace_bytes(d)
    assert 0 < nws < G.dpp.dpp_cross_attn_workspace_bytes(d)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    w64 = {k: G.f64(v) for k, v in w.items()}
    for step in range(3):  # one prompt, several denoising steps
        X = G.cuda(draw((B, N, C), 520 + step, dt))
        y = torch.empty_like(X)
        G.dpp.dpp_cross_attn_cached(d, X, kv, w["wq"], w["wo"], y, ws, nws)
        y_full = G.cross_attn(X, ctx, {k: v for k, v in w.items()}, H, W, heads)
        assert torch.equal(y, y_full)
        ref = oracle.cross_attention(G.f64(X), G.f64(ctx), w64["wq"], w64["wk"], w64["wv"],
                                     w64["wo"], heads)
        G.assert_rms_close(G.f64(y), ref, G.TOL[dt], "cross-attn, cached context K/V")


def test_bf16_attention_reports_fp16_range(cuda_device):
    """A bf16 attention layer holds Q, K and V in fp16.  Inputs large enough
    that a projected K exceeds 65504 are reported as DPP_ERR_RANGE in the
    device status word (the call completes; its output is not valid), and
    the status is clean again for the next, in-range call."""
    B, H, W, heads, P = 1, 8, 8, 1, 2
    a = wl.AttnShape(B, H, W, 64, heads, 64, P)
    wts = wl.attn_weights(a, 9, "bf16")
    F = draw((B, H * W, 64), 501, BF16)
    kmax = float(np.abs(G.f64(F) @ G.f64(wts["wk"]).T).max())
    assert G.dpp.dpp_device_status() == G.dpp.DPP_OK
    big = (F.float() * (1.0e5 / kmax)).to(BF16)  # largest |K| about 1e5
    G.self_attn(big, wts, None, H, W, heads, P)
    assert G.dpp.dpp_device_status() == G.dpp.DPP_ERR_RANGE
    y, _ = G.self_attn(F, wts, None, H, W, heads, P)
    assert G.dpp.dpp_device_status() == G.dpp.DPP_OK
    w64 = {k: G.f64(v) for k, v in wts.items()}
    ref = oracle.displaced_self_attention(G.f64(F), G.f64(F), w64["wq"], w64["wk"], w64["wv"],
                                          w64["wo"], heads, P)
    G.assert_rms_close(G.f64(y), ref, G.TOL[BF16], "in-range call after the range error")


def test_no_device_timeouts_recorded(cuda_device):
    assert G.dpp.dpp_device_status() == G.dpp.DPP_OK
