"""Oracle for an SDXL-shaped block chain run with displaced patch parallelism.

TEST INFRASTRUCTURE ONLY (see the package docstring): plain fp64 numpy, no
blocking or fusion, shared with nothing in the CUDA library.

[DF-guide] (sections 卷积层拆分, 注意力机制拆分, 归一化层拆分) lists the U-Net
submodules DistriFusion replaces: every Conv2d, the self-attention (attn1),
the cross-attention (attn2) and every GroupNorm.  Everything else in the
U-Net -- SiLU, LayerNorm, the feed-forward, the projections in and out of a
transformer, residual additions -- acts on one pixel or token at a time and
is left as it is.  [DF-notes] Background: the network predicting the noise
is a U-Net; its blocks below follow the SDXL layout:

  ResNet block     h = conv1(SiLU(GN1(x))) + b1;  out = x + conv2(SiLU(GN2(h))) + b2
                   (the time embedding is the same for the conditional and the
                   unconditional image of a guidance pair, so it is part of b1);
  transformer      g = GN(x);  h = g Wpi^T + bpi;
  block            h += attn1(LN1(h));  h += attn2(LN2(h), ctx);
                   h += GEGLU(LN3(h)) W2^T + b2;  out = x + h Wpo^T + bpo.

Each displaced layer reads the previous step's copy of its own input (its
stale state); the functions take and return those states.
"""
from __future__ import annotations

import numpy as np
from scipy.special import erf

from . import displaced as D


def silu(x):
    """x * sigmoid(x)."""
    return x / (1.0 + np.exp(-x))


def gelu(x):
    """The exact (erf) GELU: x * Phi(x)."""
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def layer_norm(X, eps, gamma=None, beta=None):
    """LayerNorm over the last axis (one token's channels), biased variance."""
    mean = X.mean(axis=-1, keepdims=True)
    var = ((X - mean) ** 2).mean(axis=-1, keepdims=True)
    Y = (X - mean) / np.sqrt(var + eps)
    return Y * gamma + beta if gamma is not None else Y


def linear(X, Wt, b=None):
    """X W^T (+ b); W is torch Linear [out, in]."""
    Y = X @ Wt.T
    return Y + b if b is not None else Y


def geglu(X, W1, b1):
    """The gated-GELU feed-forward input: project to 2 n features, split into
    the value half (first n) and the gate half (last n), value * GELU(gate)."""
    Hd = linear(X, W1, b1)
    n = Hd.shape[-1] // 2
    return Hd[..., :n] * gelu(Hd[..., n:])


RESNET_STATES = ("gn1", "conv1", "gn2", "conv2")


def resnet_block(x, states, prm, P, G, eps):
    """Displaced ResNet block on NHWC x.  ``states`` maps each displaced layer
    to its input at the previous step (None: the synchronous step).  Returns
    (out, new_states)."""
    st = states or {}
    g1 = silu(D.displaced_groupnorm(x, st.get("gn1", x), G, eps, prm["gn1_g"], prm["gn1_b"], P))
    h = D.displaced_conv3x3(g1, st.get("conv1", g1), prm["conv1_w"], prm["conv1_b"], P)
    g2 = silu(D.displaced_groupnorm(h, st.get("gn2", h), G, eps, prm["gn2_g"], prm["gn2_b"], P))
    y = D.displaced_conv3x3(g2, st.get("conv2", g2), prm["conv2_w"], prm["conv2_b"], P)
    return x + y, {"gn1": x, "conv1": g1, "gn2": h, "conv2": g2}


TRANSFORMER_STATES = ("gn", "attn1")


def transformer_block(x, ctx, states, prm, heads, P, G, eps_gn, eps_ln):
    """Displaced transformer block on NHWC x (tokens n = h * W + w).
    Returns (out, new_states)."""
    st = states or {}
    B, H, W, C = x.shape
    g = D.displaced_groupnorm(x, st.get("gn", x), G, eps_gn, prm["gn_g"], prm["gn_b"], P)
    h = linear(g.reshape(B, H * W, C), prm["pi_w"], prm["pi_b"])
    t1 = layer_norm(h, eps_ln, prm["ln1_g"], prm["ln1_b"])
    s1 = st.get("attn1", t1)
    h = h + D.displaced_self_attention(t1, s1, prm["wq"], prm["wk"], prm["wv"], prm["wo"],
                                       heads, P)
    t2 = layer_norm(h, eps_ln, prm["ln2_g"], prm["ln2_b"])
    h = h + D.cross_attention(t2, ctx, prm["xq"], prm["xk"], prm["xv"], prm["xo"], heads)
    t3 = layer_norm(h, eps_ln, prm["ln3_g"], prm["ln3_b"])
    h = h + linear(geglu(t3, prm["ff1_w"], prm["ff1_b"]), prm["ff2_w"], prm["ff2_b"])
    out = x + linear(h, prm["po_w"], prm["po_b"]).reshape(B, H, W, C)
    return out, {"gn": x, "attn1": t1}


def block_chain(x, ctx, states, prm_res, prm_tf, heads, P, G, eps_gn_res, eps_gn_tf, eps_ln):
    """ResNet block followed by a transformer block (one level of the U-Net's
    down path).  ``states`` = {"res": ..., "tf": ...} or None."""
    st = states or {}
    y, s_res = resnet_block(x, st.get("res"), prm_res, P, G, eps_gn_res)
    z, s_tf = transformer_block(y, ctx, st.get("tf"), prm_tf, heads, P, G, eps_gn_tf, eps_ln)
    return z, {"res": s_res, "tf": s_tf}
