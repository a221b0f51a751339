"""Pins for the oracle: each check compares it with something other than itself.

* special cases that reduce to a library routine: the synchronous first step
  (stale == fresh) and P == 1 must equal torch's fp64 conv2d / group_norm /
  scaled_dot_product_attention on the full image;
* brute-force loops over tiny inputs, written from the per-element definition
  with the fresh/stale source chosen per input row or token;
* invariants: halo locality and linearity of the conv, own-band rows of the
  stale buffer never read, permutation invariance over remote keys,
  GroupNorm moments, the stale-partials formulation of GroupNorm and the
  stale-K/V formulation of attention;
* closed forms for the guidance combine and its discrepancy.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as TF

import oracle

RNG = np.random.default_rng(1234)


def rnd(*shape):
    return RNG.standard_normal(shape)


def t64(a):
    return torch.from_numpy(np.ascontiguousarray(a))


def torch_conv_nhwc(X, Wt, bias=None):
    y = TF.conv2d(t64(X).permute(0, 3, 1, 2), t64(Wt),
                  None if bias is None else t64(bias), padding=1)
    return y.permute(0, 2, 3, 1).numpy()


def torch_gn_nhwc(X, G, eps, gamma=None, beta=None):
    y = TF.group_norm(t64(X).permute(0, 3, 1, 2), G,
                      None if gamma is None else t64(gamma),
                      None if beta is None else t64(beta), eps)
    return y.permute(0, 2, 3, 1).numpy()


def torch_mha(Xq, Xkv, Wq, Wk, Wv, Wo, heads):
    """Projections by torch matmul, core by torch SDPA (fp64)."""
    Q, K, V = t64(Xq) @ t64(Wq).T, t64(Xkv) @ t64(Wk).T, t64(Xkv) @ t64(Wv).T
    d = Q.shape[1] // heads
    sh = lambda t: t.reshape(t.shape[0], heads, d).permute(1, 0, 2)
    O = TF.scaled_dot_product_attention(sh(Q), sh(K), sh(V))
    O = O.permute(1, 0, 2).reshape(Q.shape[0], heads * d)
    return (O @ t64(Wo).T).numpy()


# ------------------------------------------------------------------ partition

def test_patch_rows_partition_and_rejects_uneven():
    H, P = 12, 4
    rows = [oracle.patch_rows(H, P, p) for p in range(P)]
    assert rows == [(0, 3), (3, 6), (6, 9), (9, 12)]
    with pytest.raises(ValueError):
        oracle.patch_rows(10, 4, 0)


def test_composite_takes_own_band_fresh_rest_stale():
    F, S = rnd(2, 8, 3, 4), rnd(2, 8, 3, 4)
    Z = oracle.composite(F, S, 4, 2)
    assert np.array_equal(Z[:, 4:6], F[:, 4:6])
    assert np.array_equal(Z[:, :4], S[:, :4]) and np.array_equal(Z[:, 6:], S[:, 6:])


# ----------------------------------------------------------------------- conv

@pytest.mark.parametrize("B,H,W,Ci,Co", [(1, 5, 7, 3, 4), (2, 8, 6, 5, 2)])
def test_conv_full_equals_torch_conv2d(B, H, W, Ci, Co):
    X, Wt, b = rnd(B, H, W, Ci), rnd(Co, Ci, 3, 3), rnd(Co)
    np.testing.assert_allclose(oracle.conv3x3(X, Wt, b), torch_conv_nhwc(X, Wt, b),
                               rtol=0, atol=1e-12)


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_displaced_conv_synchronous_step_equals_full_layer(P):
    F, Wt, b = rnd(2, 8, 5, 3), rnd(4, 3, 3, 3), rnd(4)
    out = oracle.displaced_conv3x3(F, F, Wt, b, P)
    np.testing.assert_allclose(out, torch_conv_nhwc(F, Wt, b), rtol=0, atol=1e-12)


def test_displaced_conv_single_patch_ignores_stale():
    F, S, Wt = rnd(1, 6, 6, 4), rnd(1, 6, 6, 4), rnd(3, 4, 3, 3)
    np.testing.assert_allclose(oracle.displaced_conv3x3(F, S, Wt, None, 1),
                               torch_conv_nhwc(F, Wt), rtol=0, atol=1e-12)


def test_first_layer_conv_uses_fresh_halo():
    F, S, Wt = rnd(1, 8, 4, 2), rnd(1, 8, 4, 2), rnd(3, 2, 3, 3)
    np.testing.assert_allclose(oracle.displaced_conv3x3(F, S, Wt, None, 4, first_layer=True),
                               torch_conv_nhwc(F, Wt), rtol=0, atol=1e-12)


def test_displaced_conv_bruteforce_tiny():
    B, H, W, Ci, Co, P = 2, 6, 4, 2, 3, 3
    F, S, Wt, bias = rnd(B, H, W, Ci), rnd(B, H, W, Ci), rnd(Co, Ci, 3, 3), rnd(Co)
    Hp = H // P
    ref = np.zeros((B, H, W, Co))
    for b, h, w, o in itertools.product(range(B), range(H), range(W), range(Co)):
        acc = bias[o]
        for i, ky, kx in itertools.product(range(Ci), range(3), range(3)):
            r, c = h + ky - 1, w + kx - 1
            if 0 <= r < H and 0 <= c < W:
                src = F if r // Hp == h // Hp else S
                acc += Wt[o, i, ky, kx] * src[b, r, c, i]
        ref[b, h, w, o] = acc
    np.testing.assert_allclose(oracle.displaced_conv3x3(F, S, Wt, bias, P), ref,
                               rtol=0, atol=1e-12)


def test_displaced_conv_halo_locality_and_linearity():
    """conv(Z_p) = conv(F) + conv(Z_p - F); Z_p - F is S - F outside band p, so
    on band p the difference is the conv of that masked difference, and it
    is nonzero only on the first and last row of the band."""
    B, H, W, Ci, Co, P = 1, 12, 5, 3, 4, 3
    F, S, Wt = rnd(B, H, W, Ci), rnd(B, H, W, Ci), rnd(Co, Ci, 3, 3)
    disp = oracle.displaced_conv3x3(F, S, Wt, None, P)
    D = disp - torch_conv_nhwc(F, Wt)
    # rows with no stale neighbour are the full layer's rows, bit for bit
    D0 = disp - oracle.conv3x3(F, Wt)
    for p in range(P):
        lo, hi = oracle.patch_rows(H, P, p)
        E = S - F
        E[:, lo:hi] = 0.0
        np.testing.assert_allclose(D[:, lo:hi], torch_conv_nhwc(E, Wt)[:, lo:hi],
                                   rtol=0, atol=1e-12)
        inner = [h for h in range(lo, hi) if h not in (lo, hi - 1)]
        assert np.all(D0[:, inner] == 0.0)
        np.testing.assert_allclose(D[:, inner], 0.0, rtol=0, atol=1e-12)
        if p > 0:
            assert np.abs(D[:, lo]).max() > 1e-3
        if p < P - 1:
            assert np.abs(D[:, hi - 1]).max() > 1e-3
    # image border rows have no stale neighbour
    assert np.all(D0[:, 0] == 0.0) and np.all(D0[:, H - 1] == 0.0)


def test_displaced_conv_never_reads_own_band_of_stale():
    F, S, Wt = rnd(1, 8, 4, 3), rnd(1, 8, 4, 3), rnd(2, 3, 3, 3)
    base = oracle.displaced_conv3x3(F, S, Wt, None, 4)
    for p in range(4):
        lo, hi = oracle.patch_rows(8, 4, p)
        S2 = S.copy()
        S2[:, lo:hi] += 100.0
        out = oracle.displaced_conv3x3(F, S2, Wt, None, 4)
        assert np.array_equal(out[:, lo:hi], base[:, lo:hi])


def test_conv_single_tap_weight_is_a_shift():
    X = rnd(1, 5, 6, 2)
    for dy, dx, i in [(0, 0, 1), (2, 1, 0), (1, 2, 1)]:
        Wt = np.zeros((1, 2, 3, 3))
        Wt[0, i, dy, dx] = 1.0
        Y = oracle.conv3x3(X, Wt)[0, :, :, 0]
        for h, w in itertools.product(range(5), range(6)):
            r, c = h + dy - 1, w + dx - 1
            want = X[0, r, c, i] if 0 <= r < 5 and 0 <= c < 6 else 0.0
            assert Y[h, w] == want


def test_conv_row_subset_matches_full():
    F, S, Wt = rnd(2, 8, 3, 2), rnd(2, 8, 3, 2), rnd(2, 2, 3, 3)
    full = oracle.displaced_conv3x3(F, S, Wt, None, 4)
    rows = [7, 0, 3, 4]
    assert np.array_equal(oracle.displaced_conv3x3(F, S, Wt, None, 4, out_rows=rows),
                          full[:, rows])


# ------------------------------------------------------------------ groupnorm

@pytest.mark.parametrize("C,G", [(8, 4), (12, 3), (6, 6)])
def test_groupnorm_equals_torch_group_norm(C, G):
    X, gamma, beta = rnd(2, 5, 3, C), rnd(C), rnd(C)
    np.testing.assert_allclose(oracle.groupnorm(X, G, 1e-5, gamma, beta),
                               torch_gn_nhwc(X, G, 1e-5, gamma, beta), rtol=0, atol=1e-12)


@pytest.mark.parametrize("P", [1, 2, 4])
def test_displaced_gn_synchronous_step_equals_full_layer(P):
    F, gamma, beta = rnd(2, 8, 3, 8), rnd(8), rnd(8)
    np.testing.assert_allclose(oracle.displaced_groupnorm(F, F, 4, 1e-5, gamma, beta, P),
                               torch_gn_nhwc(F, 4, 1e-5, gamma, beta), rtol=0, atol=1e-12)


def test_displaced_gn_single_patch_ignores_stale():
    F, S = rnd(1, 4, 4, 6), rnd(1, 4, 4, 6)
    np.testing.assert_allclose(oracle.displaced_groupnorm(F, S, 3, 1e-5, None, None, 1),
                               torch_gn_nhwc(F, 3, 1e-5), rtol=0, atol=1e-12)


def test_gn_without_affine_has_unit_moments_over_the_composite():
    F, S = 3.0 + 2.0 * rnd(2, 8, 4, 8), rnd(2, 8, 4, 8)
    for p in range(4):
        Y = oracle.groupnorm(oracle.composite(F, S, 4, p), 4, 0.0)
        Yg = Y.reshape(2, -1, 4, 2)
        np.testing.assert_allclose(Yg.mean(axis=(1, 3)), 0.0, atol=1e-12)
        np.testing.assert_allclose((Yg ** 2).mean(axis=(1, 3)), 1.0, atol=1e-12)


def test_displaced_gn_bruteforce_tiny():
    B, H, W, C, G, P, eps = 1, 4, 3, 6, 3, 2, 1e-5
    F, S, gamma, beta = rnd(B, H, W, C), rnd(B, H, W, C), rnd(C), rnd(C)
    cg, Hp = C // G, H // P
    ref = np.zeros((B, H, W, C))
    for b, h, w, c in itertools.product(range(B), range(H), range(W), range(C)):
        p, g = h // Hp, c // cg
        vals = []
        for r, x, k in itertools.product(range(H), range(W), range(g * cg, (g + 1) * cg)):
            vals.append((F if r // Hp == p else S)[b, r, x, k])
        mean = math.fsum(vals) / len(vals)
        var = math.fsum((v - mean) ** 2 for v in vals) / len(vals)
        ref[b, h, w, c] = (F[b, h, w, c] - mean) / math.sqrt(var + eps) * gamma[c] + beta[c]
    np.testing.assert_allclose(oracle.displaced_groupnorm(F, S, G, eps, gamma, beta, P), ref,
                               rtol=0, atol=1e-12)


def test_gn_partials_bruteforce_and_totals():
    X = rnd(2, 6, 2, 4)
    parts = oracle.groupnorm_partials(X, 2, 3)
    for p, b, g in itertools.product(range(3), range(2), range(2)):
        vals = [X[b, r, x, k] for r in range(2 * p, 2 * p + 2) for x in range(2)
                for k in range(2 * g, 2 * g + 2)]
        assert abs(parts[p, b, g, 0] - math.fsum(vals)) < 1e-12
        assert abs(parts[p, b, g, 1] - math.fsum(v * v for v in vals)) < 1e-12
    totals = X.reshape(2, 12, 2, 2)
    np.testing.assert_allclose(parts.sum(axis=0)[..., 0], totals.sum(axis=(1, 3)), atol=1e-12)


def test_displaced_gn_equals_stale_partials_formulation():
    """Fresh own-band partials plus stale remote-band partials give the same
    statistics as the composite image: the stale state of the displaced
    GroupNorm can be the per-band (sum x, sum x^2) of the previous step."""
    B, H, W, C, G, P, eps = 2, 8, 3, 12, 4, 4, 1e-5
    F, S, gamma, beta = rnd(B, H, W, C), rnd(B, H, W, C), rnd(C), rnd(C)
    pf, ps = oracle.groupnorm_partials(F, G, P), oracle.groupnorm_partials(S, G, P)
    n = H * W * C // G
    out = np.zeros_like(F)
    for p in range(P):
        tot = pf[p] + sum(ps[q] for q in range(P) if q != p)  # [B, G, 2]
        mean = tot[..., 0] / n
        var = tot[..., 1] / n - mean ** 2
        lo, hi = oracle.patch_rows(H, P, p)
        xg = F[:, lo:hi].reshape(B, hi - lo, W, G, C // G)
        yg = (xg - mean[:, None, None, :, None]) / np.sqrt(var[:, None, None, :, None] + eps)
        out[:, lo:hi] = yg.reshape(B, hi - lo, W, C) * gamma + beta
    np.testing.assert_allclose(oracle.displaced_groupnorm(F, S, G, eps, gamma, beta, P), out,
                               rtol=0, atol=1e-10)


def test_displaced_gn_never_reads_own_band_of_stale():
    F, S = rnd(1, 8, 2, 4), rnd(1, 8, 2, 4)
    base = oracle.displaced_groupnorm(F, S, 2, 1e-5, None, None, 4)
    S2 = S.copy()
    S2[:, 2:4] -= 50.0
    assert np.array_equal(oracle.displaced_groupnorm(F, S2, 2, 1e-5, None, None, 4)[:, 2:4],
                          base[:, 2:4])


# ------------------------------------------------------------------ attention

def test_attention_heads_equals_torch_sdpa():
    Q, K, V = rnd(7, 8), rnd(11, 8), rnd(11, 8)
    np.testing.assert_allclose(oracle.attention_heads(Q, K, V, 2), _sdpa(Q, K, V, 2),
                               rtol=0, atol=1e-12)


def _sdpa(Q, K, V, heads):
    d = Q.shape[1] // heads
    sh = lambda a: t64(a).reshape(a.shape[0], heads, d).permute(1, 0, 2)
    O = TF.scaled_dot_product_attention(sh(Q), sh(K), sh(V))
    return O.permute(1, 0, 2).reshape(Q.shape[0], heads * d).numpy()


def test_attention_rows_are_convex_weights():
    Q, K = 3.0 * rnd(9, 4), 3.0 * rnd(13, 4)
    np.testing.assert_allclose(oracle.attention_heads(Q, K, np.ones((13, 4)), 2), 1.0,
                               rtol=0, atol=1e-12)
    # a value column that is constant per key picks out a weighted mean
    V = np.repeat(rnd(13, 1), 4, axis=1)
    O = oracle.attention_heads(Q, K, V, 2)
    assert O.min() >= V.min() - 1e-12 and O.max() <= V.max() + 1e-12


@pytest.mark.parametrize("P", [1, 2, 4])
def test_displaced_self_attn_synchronous_step_equals_full_layer(P):
    B, N, C, heads = 2, 8, 8, 2
    F = rnd(B, N, C)
    Ws = [rnd(C, C) / math.sqrt(C) for _ in range(4)]
    out = oracle.displaced_self_attention(F, F, *Ws, heads, P)
    for b in range(B):
        np.testing.assert_allclose(out[b], torch_mha(F[b], F[b], *Ws, heads), rtol=0, atol=1e-12)


def test_displaced_self_attn_single_patch_ignores_stale():
    F, S = rnd(1, 6, 4), rnd(1, 6, 4)
    Ws = [rnd(4, 4) for _ in range(4)]
    np.testing.assert_allclose(oracle.displaced_self_attention(F, S, *Ws, 1, 1)[0],
                               torch_mha(F[0], F[0], *Ws, 1), rtol=0, atol=1e-12)


def test_displaced_self_attn_bruteforce_tiny():
    B, N, C, heads, P = 1, 6, 4, 2, 3
    F, S = rnd(B, N, C), rnd(B, N, C)
    Wq, Wk, Wv, Wo = (rnd(C, C) for _ in range(4))
    d, Np = C // heads, N // P
    ref = np.zeros((B, N, C))
    for b, n in itertools.product(range(B), range(N)):
        p = n // Np
        o = np.zeros(C)
        for h in range(heads):
            js = range(h * d, (h + 1) * d)
            q = [sum(F[b, n, i] * Wq[j, i] for i in range(C)) for j in js]
            scores, vals = [], []
            for m in range(N):
                src = F if m // Np == p else S
                k = [sum(src[b, m, i] * Wk[j, i] for i in range(C)) for j in js]
                v = [sum(src[b, m, i] * Wv[j, i] for i in range(C)) for j in js]
                scores.append(sum(a * c for a, c in zip(q, k)) / math.sqrt(d))
                vals.append(v)
            mx = max(scores)
            ws = [math.exp(s - mx) for s in scores]
            z = math.fsum(ws)
            for t, j in enumerate(js):
                o[j] = math.fsum(w * v[t] for w, v in zip(ws, vals)) / z
        ref[b, n] = [sum(o[i] * Wo[j, i] for i in range(C)) for j in range(C)]
    np.testing.assert_allclose(oracle.displaced_self_attention(F, S, Wq, Wk, Wv, Wo, heads, P),
                               ref, rtol=0, atol=1e-10)


def test_displaced_self_attn_invariances():
    B, N, C, heads, P = 1, 12, 4, 2, 3
    F, S = rnd(B, N, C), rnd(B, N, C)
    Ws = [rnd(C, C) for _ in range(4)]
    base = oracle.displaced_self_attention(F, S, *Ws, heads, P)
    for p in range(P):
        lo, hi = oracle.patch_rows(N, P, p)
        # own-band rows of the stale tokens are never read
        S2 = S.copy()
        S2[:, lo:hi] = 7.0
        np.testing.assert_array_equal(
            oracle.displaced_self_attention(F, S2, *Ws, heads, P)[:, lo:hi], base[:, lo:hi])
        # permuting remote stale tokens leaves band p unchanged (keys are a set)
        remote = np.array([m for m in range(N) if not lo <= m < hi])
        S3 = S.copy()
        S3[:, remote] = S[:, remote[::-1]]
        np.testing.assert_allclose(
            oracle.displaced_self_attention(F, S3, *Ws, heads, P)[:, lo:hi], base[:, lo:hi],
            rtol=0, atol=1e-12)


def test_displaced_self_attn_equals_stale_kv_formulation():
    """Attending over stale K/V (projected at the previous step) is the same
    as projecting the stale activations: the stale state can be K/V."""
    B, N, C, heads, P = 2, 8, 8, 2, 4
    F, S = rnd(B, N, C), rnd(B, N, C)
    Wq, Wk, Wv, Wo = (rnd(C, C) for _ in range(4))
    kvF, kvS = oracle.kv_state(F, Wk, Wv), oracle.kv_state(S, Wk, Wv)
    np.testing.assert_allclose(kvF[..., 0, :], (t64(F) @ t64(Wk).T).numpy(), atol=1e-12)
    np.testing.assert_allclose(kvF[..., 1, :], (t64(F) @ t64(Wv).T).numpy(), atol=1e-12)
    out = np.zeros((B, N, C))
    for b, p in itertools.product(range(B), range(P)):
        lo, hi = oracle.patch_rows(N, P, p)
        kv = kvS[b].copy()
        kv[lo:hi] = kvF[b, lo:hi]
        O = _sdpa(F[b, lo:hi] @ Wq.T, kv[:, 0], kv[:, 1], heads)
        out[b, lo:hi] = O @ Wo.T
    np.testing.assert_allclose(oracle.displaced_self_attention(F, S, Wq, Wk, Wv, Wo, heads, P),
                               out, rtol=0, atol=1e-12)


def test_self_attn_query_subset_matches_full():
    F, S = rnd(2, 8, 4), rnd(2, 8, 4)
    Ws = [rnd(4, 4) for _ in range(4)]
    full = oracle.displaced_self_attention(F, S, *Ws, 2, 4)
    qs = [7, 0, 5]
    np.testing.assert_allclose(oracle.displaced_self_attention(F, S, *Ws, 2, 4, queries=qs),
                               full[:, qs], rtol=0, atol=1e-14)


def test_cross_attention_equals_torch():
    B, N, C, nc, cc, heads = 2, 5, 8, 3, 6, 2
    X, ctx = rnd(B, N, C), rnd(B, nc, cc)
    Wq, Wk, Wv, Wo = rnd(C, C), rnd(C, cc), rnd(C, cc), rnd(C, C)
    out = oracle.cross_attention(X, ctx, Wq, Wk, Wv, Wo, heads)
    for b in range(B):
        Q, K, V = X[b] @ Wq.T, ctx[b] @ Wk.T, ctx[b] @ Wv.T
        np.testing.assert_allclose(out[b], _sdpa(Q, K, V, heads) @ Wo.T, rtol=0, atol=1e-12)


# ------------------------------------------------------------------------ CFG

def test_cfg_worked_example():
    """Hand-worked closed form: eps_u + 7.5 (eps_c - eps_u)."""
    u = np.array([1.0, -2.0, 0.5, 4.0])
    c = np.array([3.0, -2.0, -0.5, 5.0])
    out, sums = oracle.cfg_combine(u, c, 7.5)
    np.testing.assert_array_equal(out, [16.0, -2.0, -7.0, 11.5])
    np.testing.assert_array_equal(sums, [4.0, 7.5, 10.5])
    assert oracle.rel_mae(sums) == 4.0 / 7.5


def test_cfg_closed_forms():
    u, c = rnd(3, 5, 7), rnd(3, 5, 7)
    np.testing.assert_array_equal(oracle.cfg_combine(u, c, 0.0)[0], u)
    np.testing.assert_allclose(oracle.cfg_combine(u, c, 1.0)[0], c, rtol=0, atol=1e-15)
    assert oracle.rel_mae(oracle.cfg_combine(u, u, 7.5)[1]) == 0.0
    for k in (0.25, -0.5, 2.0):
        assert abs(oracle.rel_mae(oracle.cfg_combine(u, (1 + k) * u, 7.5)[1]) - abs(k)) < 1e-12


# -------------------------------------------------------------------- refresh

def test_refresh_matches_slicing():
    fresh = torch.randn(2, 8, 3, 4, dtype=torch.float64)
    stale = torch.randn(2, 8, 3, 4, dtype=torch.float64)
    for mask in (0, 0b1111, 0b0101, 0b1000):
        want = stale.clone()
        for p in range(4):
            if (mask >> p) & 1:
                want[:, 2 * p:2 * p + 2] = fresh[:, 2 * p:2 * p + 2]
        got = oracle.refresh_stale(fresh.numpy(), stale.numpy(), 4, mask)
        assert np.array_equal(got, want.numpy())
    assert np.array_equal(oracle.refresh_stale(fresh.numpy(), stale.numpy(), 4), fresh.numpy())


# ------------------------------------------------- naive patch parallelism
# The seam baseline ([DF-notes] Introduction para. 3): every band on its own.

@pytest.mark.parametrize("B,H,W,Ci,Co,P", [(1, 6, 5, 3, 2, 3), (2, 4, 3, 2, 3, 2)])
def test_naive_conv_bruteforce_tiny(B, H, W, Ci, Co, P):
    """Per-element loops: the input rows outside the output row's band count
    as zero, exactly like the image border."""
    F, Wt, bias = rnd(B, H, W, Ci), rnd(Co, Ci, 3, 3), rnd(Co)
    want = np.zeros((B, H, W, Co))
    Hp = H // P
    for b, h, w, o in itertools.product(range(B), range(H), range(W), range(Co)):
        lo, hi = (h // Hp) * Hp, (h // Hp + 1) * Hp
        acc = bias[o]
        for i, dy, dx in itertools.product(range(Ci), range(3), range(3)):
            r, c = h + dy - 1, w + dx - 1
            if lo <= r < hi and 0 <= c < W:
                acc += Wt[o, i, dy, dx] * F[b, r, c, i]
        want[b, h, w, o] = acc
    np.testing.assert_allclose(oracle.naive_conv3x3(F, Wt, bias, P), want, rtol=0, atol=1e-12)


def test_naive_ops_with_one_band_are_the_full_layers():
    X, Wt = rnd(2, 6, 5, 8), rnd(4, 8, 3, 3)
    np.testing.assert_allclose(oracle.naive_conv3x3(X, Wt, None, 1), torch_conv_nhwc(X, Wt),
                               rtol=0, atol=1e-12)
    g, bt = rnd(8), rnd(8)
    np.testing.assert_allclose(oracle.naive_groupnorm(X, 4, 1e-5, g, bt, 1),
                               torch_gn_nhwc(X, 4, 1e-5, g, bt), rtol=0, atol=1e-12)
    F = rnd(2, 8, 8)
    Ws = [rnd(8, 8) / math.sqrt(8) for _ in range(4)]
    out = oracle.naive_self_attention(F, *Ws, 2, 1)
    for b in range(2):
        np.testing.assert_allclose(out[b], torch_mha(F[b], F[b], *Ws, 2), rtol=0, atol=1e-12)


def test_naive_groupnorm_is_torch_group_norm_of_each_band():
    X, g, bt = rnd(2, 8, 3, 12), rnd(12), rnd(12)
    out = oracle.naive_groupnorm(X, 3, 1e-5, g, bt, 4)
    for p in range(4):
        np.testing.assert_allclose(out[:, 2 * p:2 * p + 2],
                                   torch_gn_nhwc(X[:, 2 * p:2 * p + 2], 3, 1e-5, g, bt),
                                   rtol=0, atol=1e-12)
    # without affine every (image, band, group) has mean 0 and variance 1
    y = oracle.naive_groupnorm(X, 3, 0.0, None, None, 4).reshape(2, 4, 2 * 3, 3, 4)
    np.testing.assert_allclose(y.mean(axis=(2, 4)), 0.0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=(2, 4)), 1.0, atol=1e-9)


def test_naive_self_attention_is_band_local_attention():
    B, N, C, heads, P = 2, 12, 8, 2, 3
    F = rnd(B, N, C)
    Ws = [rnd(C, C) / math.sqrt(C) for _ in range(4)]
    out = oracle.naive_self_attention(F, *Ws, heads, P)
    Np = N // P
    for b, p in itertools.product(range(B), range(P)):
        X = F[b, p * Np:(p + 1) * Np]
        np.testing.assert_allclose(out[b, p * Np:(p + 1) * Np], torch_mha(X, X, *Ws, heads),
                                   rtol=0, atol=1e-12)
    # tokens outside a band never reach its output
    G2 = F.copy()
    G2[:, Np:] += 5.0
    np.testing.assert_allclose(oracle.naive_self_attention(G2, *Ws, heads, P)[:, :Np],
                               out[:, :Np], rtol=0, atol=1e-12)


# ------------------------------------------------------ adaptive switching
# Worked by hand (flat_tol 0.05, rise_tol 0.10, patience 2):
#   relative drops   d1 .5, d2 .5, d3 .025 (flat, run 1), d4 .23 (reset),
#                    d5 .033 (flat, run 1), d6 .0069 (flat, run 2) -> tau1 = 6;
#   parallel, min 1.44: d7 1.60 > 1.584 (run 1); d8 1.40 new min (reset);
#                    d9 1.50 < 1.54 (reset); d10 1.55 > 1.54 (run 1);
#                    d11 1.56 > 1.54 (run 2) -> tau2 = 11; d12 falls, no way back.
SWITCH_SERIES = [8.0, 4.0, 2.0, 1.95, 1.5, 1.45, 1.44, 1.60, 1.40, 1.50, 1.55, 1.56, 1.2]
SWITCH_STAGES = [0, 0, 0, 0, 0, 0, 1, 1, 1, 1, 1, 2, 2]


def test_switch_worked_example():
    assert oracle.switch_stages(SWITCH_SERIES, 0.05, 0.10, 2) == SWITCH_STAGES


@pytest.mark.parametrize("patience", [1, 2, 3, 5])
def test_switch_geometric_decline_closed_form(patience):
    # d_t = 10 r^t has the constant relative drop 1 - r: flat from the first
    # step when 1 - r < flat_tol (tau1 = patience, then it never rises),
    # never flat otherwise.
    slow = [10.0 * 0.99 ** t for t in range(30)]
    assert oracle.switch_stages(slow, 0.02, 0.01, patience) == \
        [0] * patience + [1] * (30 - patience)
    fast = [10.0 * 0.9 ** t for t in range(30)]
    assert oracle.switch_stages(fast, 0.02, 0.01, patience) == [0] * 30


@pytest.mark.parametrize("patience", [1, 2, 3])
def test_switch_linear_rise_closed_form(patience):
    # d_t = 1 + t: every drop is negative (flat), so tau1 = patience; in the
    # parallel stage the minimum stays 1 + tau1 and d_j > 1.1 (1 + tau1) holds
    # for every j > tau1 once j > 0.1 (1 + tau1), i.e. for all j here, so
    # tau2 = tau1 + patience.
    d = [1.0 + t for t in range(20)]
    tau1, tau2 = patience, 2 * patience
    want = [0] * tau1 + [1] * (tau2 - tau1) + [2] * (20 - tau2)
    assert oracle.switch_stages(d, 0.05, 0.10, patience) == want


def test_switch_constant_series_parallel_forever():
    assert oracle.switch_stages([0.3] * 12, 0.01, 0.01, 3) == [0] * 3 + [1] * 9


def test_switch_is_scale_invariant_and_monotone():
    rng = np.random.default_rng(77)
    for trial in range(50):
        t = np.arange(40)
        d = list(0.2 + (t / 40.0 - 0.5) ** 2 + 0.01 * rng.standard_normal(40))
        d = [abs(x) for x in d]
        p = 1 + trial % 3
        base = oracle.switch_stages(d, 0.03, 0.05, p)
        assert all(a <= b for a, b in zip(base, base[1:]))
        assert base[:p] == [0] * p
        for c in (2.0 ** -10, 2.0 ** 13):  # exact scalings: the rules are relative
            assert oracle.switch_stages([c * x for x in d], 0.03, 0.05, p) == base


def test_switch_patience_ignores_a_single_spike():
    d = [1.0, 0.5, 0.49, 0.485, 0.482, 0.60, 0.481, 0.480, 0.479]
    assert oracle.switch_stages(d, 0.05, 0.10, 2) == [0, 0, 0, 1, 1, 1, 1, 1, 1]
    assert oracle.switch_stages(d, 0.05, 0.10, 1) == [0, 0, 1, 1, 1, 2, 2, 2, 2]


def test_switch_skips_nan_and_negative_entries():
    bad = [float("nan"), -1.0]
    for pos in range(len(SWITCH_SERIES) + 1):
        d = SWITCH_SERIES[:pos] + bad + SWITCH_SERIES[pos:]
        want = SWITCH_STAGES[:pos] + [SWITCH_STAGES[pos - 1] if pos else 0] * 2 + \
            SWITCH_STAGES[pos:]
        assert oracle.switch_stages(d, 0.05, 0.10, 2) == want


# ------------------------------------------------------------ block chain
import oracle.blocks as OB  # noqa: E402


def block_params(C, C_ctx, rng, ff_mult=4):
    n = lambda *s: rng.standard_normal(s)
    res = {"gn1_g": 1 + 0.1 * n(C), "gn1_b": 0.1 * n(C), "conv1_w": n(C, C, 3, 3) / np.sqrt(9 * C),
           "conv1_b": 0.1 * n(C), "gn2_g": 1 + 0.1 * n(C), "gn2_b": 0.1 * n(C),
           "conv2_w": n(C, C, 3, 3) / np.sqrt(9 * C), "conv2_b": 0.1 * n(C)}
    F_ = ff_mult * C
    tf = {"gn_g": 1 + 0.1 * n(C), "gn_b": 0.1 * n(C), "pi_w": n(C, C) / np.sqrt(C),
          "pi_b": 0.1 * n(C), "po_w": n(C, C) / np.sqrt(C), "po_b": 0.1 * n(C),
          "wq": n(C, C) / np.sqrt(C), "wk": n(C, C) / np.sqrt(C), "wv": n(C, C) / np.sqrt(C),
          "wo": n(C, C) / np.sqrt(C), "xq": n(C, C) / np.sqrt(C),
          "xk": n(C, C_ctx) / np.sqrt(C_ctx), "xv": n(C, C_ctx) / np.sqrt(C_ctx),
          "xo": n(C, C) / np.sqrt(C), "ff1_w": n(2 * F_, C) / np.sqrt(C), "ff1_b": 0.1 * n(2 * F_),
          "ff2_w": n(C, F_) / np.sqrt(F_), "ff2_b": 0.1 * n(C)}
    for k in ("ln1", "ln2", "ln3"):
        tf[k + "_g"], tf[k + "_b"] = 1 + 0.1 * n(C), 0.1 * n(C)
    return res, tf


def torch_resblock(x, prm, G, eps):
    T = lambda k: t64(prm[k])
    X = t64(x).permute(0, 3, 1, 2)
    h = TF.conv2d(TF.silu(TF.group_norm(X, G, T("gn1_g"), T("gn1_b"), eps)), T("conv1_w"),
                  T("conv1_b"), padding=1)
    y = TF.conv2d(TF.silu(TF.group_norm(h, G, T("gn2_g"), T("gn2_b"), eps)), T("conv2_w"),
                  T("conv2_b"), padding=1)
    return (X + y).permute(0, 2, 3, 1).numpy()


def torch_attention(q_in, kv_in, wq, wk, wv, wo, heads):
    B, N, C = q_in.shape
    d = C // heads
    split = lambda t: t.reshape(B, t.shape[1], heads, d).transpose(1, 2)
    o = TF.scaled_dot_product_attention(split(TF.linear(q_in, wq)), split(TF.linear(kv_in, wk)),
                                        split(TF.linear(kv_in, wv)))
    return TF.linear(o.transpose(1, 2).reshape(B, N, C), wo)


def torch_transformer(x, ctx, prm, heads, G, eps_gn, eps_ln):
    T = lambda k: t64(prm[k])
    B, H, W, C = x.shape
    X = t64(x)
    g = TF.group_norm(X.permute(0, 3, 1, 2), G, T("gn_g"), T("gn_b"), eps_gn)
    h = TF.linear(g.permute(0, 2, 3, 1).reshape(B, H * W, C), T("pi_w"), T("pi_b"))
    t = TF.layer_norm(h, (C,), T("ln1_g"), T("ln1_b"), eps_ln)
    h = h + torch_attention(t, t, T("wq"), T("wk"), T("wv"), T("wo"), heads)
    t = TF.layer_norm(h, (C,), T("ln2_g"), T("ln2_b"), eps_ln)
    h = h + torch_attention(t, t64(ctx), T("xq"), T("xk"), T("xv"), T("xo"), heads)
    t = TF.layer_norm(h, (C,), T("ln3_g"), T("ln3_b"), eps_ln)
    a, gate = TF.linear(t, T("ff1_w"), T("ff1_b")).chunk(2, dim=-1)
    h = h + TF.linear(a * TF.gelu(gate), T("ff2_w"), T("ff2_b"))
    return (X + TF.linear(h, T("po_w"), T("po_b")).reshape(B, H, W, C)).numpy()


def test_layer_norm_gelu_silu_geglu_equal_torch():
    X = rnd(3, 7, 24)
    g, b = 1 + 0.1 * rnd(24), 0.1 * rnd(24)
    want = TF.layer_norm(t64(X), (24,), t64(g), t64(b), 1e-5).numpy()
    assert np.allclose(OB.layer_norm(X, 1e-5, g, b), want, rtol=0, atol=1e-12)
    assert np.allclose(OB.gelu(X), TF.gelu(t64(X)).numpy(), rtol=0, atol=1e-12)
    assert np.allclose(OB.silu(X), TF.silu(t64(X)).numpy(), rtol=0, atol=1e-12)
    W1, b1 = rnd(2 * 10, 24), rnd(2 * 10)
    a, gate = TF.linear(t64(X), t64(W1), t64(b1)).chunk(2, dim=-1)
    assert np.allclose(OB.geglu(X, W1, b1), (a * TF.gelu(gate)).numpy(), rtol=0, atol=1e-12)


def test_gelu_closed_forms():
    # GELU(0) = 0, GELU(x) - GELU(-x) = x, GELU(x) -> x for large x
    x = np.linspace(-4, 4, 33)
    assert OB.gelu(np.zeros(1))[0] == 0.0
    assert np.allclose(OB.gelu(x) - OB.gelu(-x), x, atol=1e-14)
    assert abs(OB.gelu(np.array([10.0]))[0] - 10.0) < 1e-12


@pytest.mark.parametrize("P", [1, 2, 4])
def test_resnet_block_synchronous_step_equals_torch(P):
    rng = np.random.default_rng(31 + P)
    x = rng.standard_normal((2, 8, 5, 16))
    prm, _ = block_params(16, 12, rng)
    out, st = OB.resnet_block(x, None, prm, P, 4, 1e-5)
    assert np.allclose(out, torch_resblock(x, prm, 4, 1e-5), rtol=0, atol=1e-10)
    assert set(st) == set(OB.RESNET_STATES)


@pytest.mark.parametrize("P", [1, 2, 4])
def test_transformer_block_synchronous_step_equals_torch(P):
    rng = np.random.default_rng(41 + P)
    x = rng.standard_normal((2, 8, 3, 16))
    ctx = rng.standard_normal((2, 5, 12))
    _, prm = block_params(16, 12, rng)
    out, st = OB.transformer_block(x, ctx, None, prm, 2, P, 4, 1e-6, 1e-5)
    assert np.allclose(out, torch_transformer(x, ctx, prm, 2, 4, 1e-6, 1e-5), rtol=0, atol=1e-10)
    assert set(st) == set(OB.TRANSFORMER_STATES)


def test_block_chain_states_route_to_their_layers():
    # With the same input twice, every layer's input repeats, so the second,
    # displaced step (fed the first step's states) equals the synchronous one;
    # a state handed to the wrong layer breaks this.
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, 8, 4, 16))
    ctx = rng.standard_normal((1, 5, 12))
    pr, pt = block_params(16, 12, rng)
    out0, st = OB.block_chain(x, ctx, None, pr, pt, 2, 4, 4, 1e-5, 1e-6, 1e-5)
    out1, st1 = OB.block_chain(x, ctx, st, pr, pt, 2, 4, 4, 1e-5, 1e-6, 1e-5)
    assert np.allclose(out1, out0, rtol=0, atol=1e-12)
    # and with a changed input the displaced step differs from the synchronous one
    x2 = x + 0.3 * rng.standard_normal(x.shape)
    sync, _ = OB.block_chain(x2, ctx, None, pr, pt, 2, 4, 4, 1e-5, 1e-6, 1e-5)
    disp, _ = OB.block_chain(x2, ctx, st, pr, pt, 2, 4, 4, 1e-5, 1e-6, 1e-5)
    assert np.abs(disp - sync).max() > 1e-3
