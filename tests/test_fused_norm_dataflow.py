"""The dataflow of GroupNorm -> SiLU applied in the conv's load, emulated in
fp64 on the host, against the oracle's unfused composition.

The pages store each layer's output and gather it: the displaced conv's stale
input is the previous step's *normalised* tensor, every band normalised with
its own composite statistics of that step (DistriFusion developer guide,
归一化层拆分 and 卷积层拆分).  The library instead keeps the previous step's
un-normalised input, the previous step's per-band affine and the band
partials, and normalises on load: a halo row of band q is normalised with
band q's affine of the previous step.  Over four steps (the synchronous one
and three displaced) the emulated dataflow must reproduce the unfused
composition to rounding; using this step's affine for the halo rows (the
plausible mistake) must not.
"""
import numpy as np

import oracle
import oracle.blocks as OB
from oracle.displaced import patch_rows

B, H, W, C, G, P, EPS = 1, 8, 6, 16, 4, 4, 1e-5
STEPS = 4


def inputs(seed=11):
    rng = np.random.default_rng(seed)
    xs = [rng.normal(0.3, 1.2, (B, H, W, C))]
    for _ in range(STEPS - 1):
        xs.append(xs[-1] + 0.4 * rng.normal(size=(B, H, W, C)))
    gamma = 1.0 + 0.1 * rng.normal(size=C)
    beta = 0.1 * rng.normal(size=C)
    w = rng.normal(size=(C, C, 3, 3)) / np.sqrt(9 * C)
    bias = 0.1 * rng.normal(size=C)
    return xs, gamma, beta, w, bias


def band_affine(partials_fresh, partials_stale, gamma, beta):
    """Per band p: (a, s) per channel from the band's fresh partials plus the
    other bands' stale partials (all fresh in the synchronous step)."""
    n = H * W * (C // G)
    aff = np.zeros((P, B, C, 2))
    for p in range(P):
        tot = partials_fresh[p].copy()
        for q in range(P):
            if q != p:
                tot = tot + (partials_fresh[q] if partials_stale is None else partials_stale[q])
        mean = tot[..., 0] / n                      # [B, G]
        var = np.maximum(tot[..., 1] / n - mean ** 2, 0.0)
        rstd = 1.0 / np.sqrt(var + EPS)
        a = np.repeat(rstd, C // G, axis=-1) * gamma     # [B, C]
        s = beta - np.repeat(mean, C // G, axis=-1) * a
        aff[p, :, :, 0], aff[p, :, :, 1] = a, s
    return aff


def apply_per_band(x, aff):
    """SiLU(x * a + s), band q's rows with band q's affine."""
    y = np.empty_like(x)
    for q in range(P):
        lo, hi = patch_rows(H, P, q)
        y[:, lo:hi] = OB.silu(x[:, lo:hi] * aff[q][:, None, None, :, 0] + aff[q][:, None, None, :, 1])
    return y


def fused_steps(xs, gamma, beta, w, bias, halo_affine="previous"):
    """The library's dataflow: state = (raw input, affine, partials) of the
    previous step; the conv's fresh rows are this step's input normalised
    with this step's affine, its halo rows the previous raw input normalised
    with the previous step's affine of their band."""
    outs, prev = [], None
    for x in xs:
        part = oracle.groupnorm_partials(x, G, P)
        aff = band_affine(part, None if prev is None else prev["part"], gamma, beta)
        z_fresh = apply_per_band(x, aff)
        if prev is None:
            z_stale = z_fresh  # synchronous step: no stale input
        else:
            halo_aff = prev["aff"] if halo_affine == "previous" else aff
            z_stale = apply_per_band(prev["x"], halo_aff)
        outs.append(oracle.displaced_conv3x3(z_fresh, z_stale, w, bias, P))
        prev = {"x": x, "aff": aff, "part": part}
    return outs


def unfused_steps(xs, gamma, beta, w, bias):
    """The pages' dataflow: each step's normalised tensor is stored, and the
    next step's conv reads it as stale."""
    outs, g_prev, x_prev = [], None, None
    for x in xs:
        if x_prev is None:
            g = OB.silu(oracle.groupnorm(x, G, EPS, gamma, beta))
        else:
            g = OB.silu(oracle.displaced_groupnorm(x, x_prev, G, EPS, gamma, beta, P))
        outs.append(oracle.displaced_conv3x3(g, g if g_prev is None else g_prev, w, bias, P))
        g_prev, x_prev = g, x
    return outs


def test_normalising_in_the_load_reproduces_the_stored_composition():
    xs, gamma, beta, w, bias = inputs()
    want = unfused_steps(xs, gamma, beta, w, bias)
    got = fused_steps(xs, gamma, beta, w, bias)
    for t, (g, u) in enumerate(zip(got, want)):
        rms = float(np.sqrt(np.mean(u ** 2)))
        assert float(np.max(np.abs(g - u))) <= 1e-12 * rms, t


def test_halo_rows_need_the_previous_steps_affine():
    # the plausible mistake -- normalising the stale halo rows with this
    # step's statistics -- changes every displaced step's halo outputs
    xs, gamma, beta, w, bias = inputs()
    want = unfused_steps(xs, gamma, beta, w, bias)
    wrong = fused_steps(xs, gamma, beta, w, bias, halo_affine="current")
    assert np.allclose(wrong[0], want[0])  # the synchronous step has no stale input
    for t in range(1, STEPS):
        rms = float(np.sqrt(np.mean(want[t] ** 2)))
        assert float(np.max(np.abs(wrong[t] - want[t]))) > 1e-3 * rms, t
