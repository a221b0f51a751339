"""Plain fp64 statement of the displaced-patch layer ops (test infrastructure).

Layouts: activations are NHWC ``[B, H, W, C]``; attention tokens are
``[B, N, C]`` with token n = h * W + w, so a band of image rows is a
contiguous token range.  Conv weights are in torch order ``[C_out, C_in, 3, 3]``,
linear weights ``[out, in]``.  Every array is float64; callers upcast the exact
fp32/bf16 input values.

No blocking, fusion or reordering: each function is the textbook definition,
evaluated on the composite image Z_p of the module docstring of ``oracle``.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# Partition and composite image
# --------------------------------------------------------------------------

def patch_rows(H: int, P: int, p: int):
    """Rows [lo, hi) owned by band p of P (equal height bands).

    [DF-guide] communication section: the gathered slices are concatenated
    along dim 2 of an NCHW tensor, i.e. the patches are bands of image rows.
    Unequal bands are not described, so H must be divisible by P.
    """
    if P < 1 or H % P != 0:
        raise ValueError(f"H={H} is not divisible by P={P}")
    if not 0 <= p < P:
        raise ValueError(f"patch {p} out of range for P={P}")
    h = H // P
    return p * h, (p + 1) * h


def patch_of_row(h: int, H: int, P: int) -> int:
    return h // (H // P)


def composite(F: np.ndarray, S: np.ndarray, P: int, p: int, axis: int = 1):
    """Z_p: band p's rows from the fresh tensor F, every other row from the
    stale tensor S ([DF-notes] Introduction para. 4: previous-step
    activations give the global context; Related Work / Parallelism)."""
    if F.shape != S.shape:
        raise ValueError("fresh and stale shapes differ")
    lo, hi = patch_rows(F.shape[axis], P, p)
    Z = np.array(S, dtype=np.float64, copy=True)
    idx = [slice(None)] * F.ndim
    idx[axis] = slice(lo, hi)
    Z[tuple(idx)] = F[tuple(idx)]
    return Z


# --------------------------------------------------------------------------
# 3x3 convolution (DistriConv2dPP, [DF-guide] 卷积层拆分)
# --------------------------------------------------------------------------

def _conv_row(rows_in, Wt, W):
    """One output row of a 3x3, pad-1 cross-correlation.

    rows_in[dy] is the input row h + dy - 1 as a ``[B, W, C_in]`` array, or None
    where that row lies outside the image (zero padding).
    Y[b, w, o] = sum_{dy, dx, i} Wt[o, i, dy, dx] * X[b, h+dy-1, w+dx-1, i].
    """
    B = next(r.shape[0] for r in rows_in if r is not None)
    C_in = Wt.shape[1]
    Y = np.zeros((B, W, Wt.shape[0]))
    for dy in range(3):
        r = rows_in[dy]
        if r is None:
            continue
        padded = np.zeros((B, W + 2, C_in))
        padded[:, 1:W + 1] = r
        for dx in range(3):
            Y += padded[:, dx:dx + W, :] @ Wt[:, :, dy, dx].T
    return Y


def conv3x3(X, Wt, bias=None, out_rows=None):
    """Full-image 3x3 conv, stride 1, zero padding 1 (torch Conv2d semantics:
    cross-correlation, no kernel flip).  Returns ``[B, len(out_rows), W, C_out]``
    (all rows when out_rows is None)."""
    B, H, W, _ = X.shape
    rows = range(H) if out_rows is None else list(out_rows)
    out = np.zeros((B, len(rows), W, Wt.shape[0]))
    for k, h in enumerate(rows):
        src = [X[:, r] if 0 <= r < H else None for r in (h - 1, h, h + 1)]
        out[:, k] = _conv_row(src, Wt, W)
        if bias is not None:
            out[:, k] += bias
    return out


def displaced_conv3x3(F, S, Wt, bias, P, out_rows=None, first_layer=False):
    """Displaced conv: output row h (band p = h // (H/P)) is the conv of Z_p.

    Input row r of Z_p is F[:, r] when r is in R_p, else S[:, r]; only the two
    halo rows next to the band come from S.  With ``first_layer`` (the
    ``is_first_layer`` flag the conv wrapper takes for conv_in, [DF-guide]
    卷积层拆分) the input latent is the same on every device, so every row is
    fresh.  Returns ``[B, len(out_rows), W, C_out]``.
    """
    B, H, W, _ = F.shape
    rows = range(H) if out_rows is None else list(out_rows)
    out = np.zeros((B, len(rows), W, Wt.shape[0]))
    for k, h in enumerate(rows):
        lo, hi = patch_rows(H, P, patch_of_row(h, H, P))
        src = []
        for r in (h - 1, h, h + 1):
            if not 0 <= r < H:
                src.append(None)
            elif first_layer or lo <= r < hi:
                src.append(F[:, r])
            else:
                src.append(S[:, r])
        out[:, k] = _conv_row(src, Wt, W)
        if bias is not None:
            out[:, k] += bias
    return out


def naive_conv3x3(F, Wt, bias, P, out_rows=None):
    """Naive patch parallelism ([DF-notes] Introduction para. 3): band p is
    convolved as an image of its own, so the rows just outside the band read
    as zero (zero padding at every band edge) -- no stale buffer, and the
    seams the method exists to remove.  Returns ``[B, len(out_rows), W, C_out]``."""
    B, H, W, _ = F.shape
    rows = range(H) if out_rows is None else list(out_rows)
    out = np.zeros((B, len(rows), W, Wt.shape[0]))
    for k, h in enumerate(rows):
        lo, hi = patch_rows(H, P, patch_of_row(h, H, P))
        src = [F[:, r] if lo <= r < hi else None for r in (h - 1, h, h + 1)]
        out[:, k] = _conv_row(src, Wt, W)
        if bias is not None:
            out[:, k] += bias
    return out


# --------------------------------------------------------------------------
# GroupNorm (DistriGroupNorm, [DF-guide] 归一化层拆分)
# --------------------------------------------------------------------------

def groupnorm(X, G, eps, gamma=None, beta=None):
    """Textbook GroupNorm over ``[B, H, W, C]``: per (b, g) the mean and the
    biased variance over all H*W pixels and the C/G channels of group g
    (two passes), y = (x - mean) / sqrt(var + eps), then the per-channel
    affine when gamma/beta are given."""
    B, H, W, C = X.shape
    if C % G:
        raise ValueError("C not divisible by G")
    Xg = X.reshape(B, H * W, G, C // G)
    mean = Xg.mean(axis=(1, 3), keepdims=True)
    var = ((Xg - mean) ** 2).mean(axis=(1, 3), keepdims=True)
    Y = ((Xg - mean) / np.sqrt(var + eps)).reshape(B, H, W, C)
    if gamma is not None:
        Y = Y * gamma + (0.0 if beta is None else beta)
    return Y


def groupnorm_partials(X, G, P):
    """Per-band partial sums ``[P, B, G, 2]``: (sum x, sum x^2) over the rows
    of band p and the channels of group g.  This is the state a band
    contributes to the others' statistics (the displaced GroupNorm combines
    fresh own partials with stale remote ones)."""
    B, H, W, C = X.shape
    out = np.zeros((P, B, G, 2))
    for p in range(P):
        lo, hi = patch_rows(H, P, p)
        Xg = X[:, lo:hi].reshape(B, (hi - lo) * W, G, C // G)
        out[p, :, :, 0] = Xg.sum(axis=(1, 3))
        out[p, :, :, 1] = (Xg ** 2).sum(axis=(1, 3))
    return out


def displaced_groupnorm(F, S, G, eps, gamma, beta, P, bands=None):
    """Displaced GroupNorm: band p's rows of groupnorm(Z_p).  Returns the full
    ``[B, H, W, C]`` output (band p filled from its own composite); with
    ``bands`` only those bands are evaluated and the other rows are NaN."""
    B, H, W, C = F.shape
    out = np.full((B, H, W, C), np.nan)
    for p in (range(P) if bands is None else bands):
        lo, hi = patch_rows(H, P, p)
        out[:, lo:hi] = groupnorm(composite(F, S, P, p), G, eps, gamma, beta)[:, lo:hi]
    return out


def naive_groupnorm(F, G, eps, gamma, beta, P):
    """Naive patch parallelism ([DF-notes] Introduction para. 3: every band
    generated on its own, no interaction): band p normalised with the
    statistics of its own rows only, i.e. groupnorm of the band alone."""
    B, H, W, C = F.shape
    out = np.zeros((B, H, W, C))
    for p in range(P):
        lo, hi = patch_rows(H, P, p)
        out[:, lo:hi] = groupnorm(F[:, lo:hi], G, eps, gamma, beta)
    return out


# --------------------------------------------------------------------------
# Attention (DistriSelfAttentionPP / DistriCrossAttentionPP, [DF-guide] 注意力机制拆分)
# --------------------------------------------------------------------------

def linear(X, Wt):
    """x W^T with W in torch Linear order [out, in]; no bias."""
    return X @ Wt.T


def attention_heads(Q, K, V, heads):
    """Multi-head softmax attention of ``[Nq, C]`` queries over ``[Nk, C]``
    keys/values; head h uses channels [h*d, (h+1)*d), d = C / heads, scale
    1/sqrt(d).  Softmax with max subtraction, in fp64."""
    C = Q.shape[1]
    d = C // heads
    O = np.zeros((Q.shape[0], V.shape[1]))
    for h in range(heads):
        cs = slice(h * d, (h + 1) * d)
        s = Q[:, cs] @ K[:, cs].T / np.sqrt(d)
        s = s - s.max(axis=1, keepdims=True)
        e = np.exp(s)
        O[:, cs] = (e / e.sum(axis=1, keepdims=True)) @ V[:, cs]
    return O


def kv_state(X, Wk, Wv):
    """Per-token (K, V) = (x Wk^T, x Wv^T) as ``[B, N, 2, C]``: what a band
    publishes for the others to attend over at the next step."""
    return np.stack([linear(X, Wk), linear(X, Wv)], axis=2)


def displaced_self_attention(F, S, Wq, Wk, Wv, Wo, heads, P, queries=None):
    """Displaced self-attention on ``[B, N, C]`` tokens (N = H*W, bands of
    N/P consecutive tokens).

    Band p: queries are its own fresh tokens, Q = F_{R_p} Wq^T; keys and values
    are projected from the composite tokens Z_p (fresh own band, stale rest);
    O = softmax(Q K^T / sqrt(d)) V per head; Y = O Wo^T.  ``queries`` (token
    indices, optional) restricts the returned rows; returns ``[B, nq, C]``.
    """
    B, N, C = F.shape
    qs = np.arange(N) if queries is None else np.asarray(queries)
    out = np.zeros((B, len(qs), Wo.shape[0]))
    for p in range(P):
        sel = np.nonzero((qs // (N // P)) == p)[0]
        if len(sel) == 0:
            continue
        patch_rows(N, P, p)  # validates N % P
        for b in range(B):
            Z = composite(F[b:b + 1], S[b:b + 1], P, p)[0]
            Q = linear(F[b, qs[sel]], Wq)
            O = attention_heads(Q, linear(Z, Wk), linear(Z, Wv), heads)
            out[b, sel] = linear(O, Wo)
    return out


def naive_self_attention(F, Wq, Wk, Wv, Wo, heads, P):
    """Naive patch parallelism ([DF-notes] Introduction para. 3): band p's
    queries attend over the band's own tokens only -- self-attention of each
    band as a sequence of its own.  Returns ``[B, N, C]``."""
    B, N, C = F.shape
    out = np.zeros((B, N, Wo.shape[0]))
    for p in range(P):
        lo, hi = patch_rows(N, P, p)
        for b in range(B):
            X = F[b, lo:hi]
            O = attention_heads(linear(X, Wq), linear(X, Wk), linear(X, Wv), heads)
            out[b, lo:hi] = linear(O, Wo)
    return out


def cross_attention(X, ctx, Wq, Wk, Wv, Wo, heads, queries=None):
    """Cross-attention of image tokens ``[B, N, C]`` over a text context
    ``[B, n_ctx, c_ctx]``: Q = X Wq^T, K = ctx Wk^T, V = ctx Wv^T,
    Y = softmax(Q K^T / sqrt(d)) V Wo^T.  The context is the same on every
    device, so no stale state enters."""
    B, N, C = X.shape
    qs = np.arange(N) if queries is None else np.asarray(queries)
    out = np.zeros((B, len(qs), Wo.shape[0]))
    for b in range(B):
        Q = linear(X[b, qs], Wq)
        O = attention_heads(Q, linear(ctx[b], Wk), linear(ctx[b], Wv), heads)
        out[b] = linear(O, Wo)
    return out


# --------------------------------------------------------------------------
# Classifier-free guidance and the denoising discrepancy
# --------------------------------------------------------------------------

def cfg_combine(eps_u, eps_c, scale):
    """Guided estimate eps_u + s * (eps_c - eps_u) from the unconditional and
    conditional predictions ([Hydiff-zh] condition-based partitioning: the two
    branches are the units of work), and the three sums
    (sum|eps_c - eps_u|, sum|eps_u|, sum|eps_c|) of the discrepancy reduction."""
    u = np.asarray(eps_u, dtype=np.float64)
    c = np.asarray(eps_c, dtype=np.float64)
    out = u + scale * (c - u)
    sums = np.array([np.abs(c - u).sum(), np.abs(u).sum(), np.abs(c).sum()])
    return out, sums


def rel_mae(sums):
    """Relative mean absolute error between eps_c and eps_u ([Hydiff-zh]
    adaptive switching: the denoising discrepancy is the rel-MAE of the two
    predictions; [Hydiff-ru]: the difference of conditional and unconditional
    estimates).  Read as sum|eps_c - eps_u| / sum|eps_u| over the whole map."""
    return float(sums[0] / sums[1])


# --------------------------------------------------------------------------
# Stale-buffer refresh (the AllGather, [DF-guide] 分布式通信与同步机制)
# --------------------------------------------------------------------------

def refresh_stale(fresh, stale, P, patch_mask=None, axis=1):
    """New stale buffer after the gather: band p's rows (along ``axis``) are
    replaced by the fresh ones for every p whose bit is set in patch_mask
    (all bands when None); the other rows keep the old stale values."""
    out = np.array(stale, copy=True)
    n = fresh.shape[axis]
    for p in range(P):
        if patch_mask is not None and not (patch_mask >> p) & 1:
            continue
        lo, hi = patch_rows(n, P, p)
        idx = [slice(None)] * fresh.ndim
        idx[axis] = slice(lo, hi)
        out[tuple(idx)] = fresh[tuple(idx)]
    return out


# --------------------------------------------------------------------------
# Adaptive parallelism switching ([Hydiff-zh] 自适应并行切换; [Hydiff-ru]
# Адаптивное переключение)
# --------------------------------------------------------------------------

WARMUP, PARALLEL, FULLY_CONNECTING = 0, 1, 2


def switch_stages(ds, flat_tol, rise_tol, patience):
    """Stage each denoising step runs in, read off the discrepancy series.

    [Hydiff-zh] splits the sampling run T -> 0 into a warm-up stage (T -> tau1,
    branches run serially), a parallel stage (tau1 -> tau2) and a fully
    connecting stage (tau2 -> 0, serial again); tau1 is where the decline of
    the discrepancy flattens and tau2 where it starts rising, both found from
    the live curve.  The pages give no numbers, so:

      tau1 = the first observation t >= patience at which each of the last
             ``patience`` relative drops (d[j-1] - d[j]) / d[j-1] is below
             flat_tol (a zero d[j-1] counts as drop 0);
      tau2 = the first observation t >= tau1 + patience at which each of the
             last ``patience`` values d[j] (j > tau1) is above
             (1 + rise_tol) * min(d[tau1..j]).

    Returns, for every entry of ``ds``, the stage after seeing it (the stage
    the next step runs in).  An entry that is NaN or negative carries no
    information: it is skipped and repeats the stage before it.
    """
    patience = max(1, int(patience))
    valid = [i for i, d in enumerate(ds) if d >= 0.0]  # False for NaN too
    v = [float(ds[i]) for i in valid]

    def drop(j):
        return (v[j - 1] - v[j]) / v[j - 1] if v[j - 1] > 0.0 else 0.0

    tau1 = None
    for t in range(patience, len(v)):
        if all(drop(j) < flat_tol for j in range(t - patience + 1, t + 1)):
            tau1 = t
            break
    tau2 = None
    if tau1 is not None:
        for t in range(tau1 + patience, len(v)):
            if all(v[j] > min(v[tau1:j + 1]) * (1.0 + rise_tol)
                   for j in range(t - patience + 1, t + 1)):
                tau2 = t
                break

    def stage_at(t):
        if tau2 is not None and t >= tau2:
            return FULLY_CONNECTING
        if tau1 is not None and t >= tau1:
            return PARALLEL
        return WARMUP

    out, last, k = [], WARMUP, 0
    for i in range(len(ds)):
        if k < len(valid) and valid[k] == i:
            last = stage_at(k)
            k += 1
        out.append(last)
    return out
