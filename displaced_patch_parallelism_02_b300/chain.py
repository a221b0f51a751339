"""SDXL-shaped block chain stepped with displaced patch parallelism.

One level of the U-Net's down path: a ResNet block followed by a transformer
block, on an NHWC latent of B x H x W x C cut into P bands of rows.  Every
layer is a call into libdpp (this module only sequences the calls and owns the
buffers); the layers DistriFusion replaces (convolutions, GroupNorms, self-
attention) read the previous step's state of the other bands, the per-token
layers (LayerNorm, projections, the gated feed-forward) need none:

  ResNet block   g1 = SiLU(GN1(x))              dpp_groupnorm (act SiLU)
                 h1 = conv1(g1) + b1            dpp_conv3x3_gn (sums for GN2)
                 g2 = SiLU(GN2(h1))             dpp_groupnorm_apply (act SiLU)
                 x += conv2(g2) + b2            dpp_conv3x3_gn (accumulate; sums for GN)
  transformer    g = GN(x)                      dpp_groupnorm_apply
                 h = g Wpi^T + bpi              dpp_linear
                 h += attn1(LN1(h))             dpp_layernorm, dpp_self_attn (accumulate)
                 h += attn2(LN2(h), ctx)        dpp_layernorm, dpp_cross_attn (accumulate)
                 h += GEGLU(LN3(h)) W2^T + b2   dpp_layernorm, dpp_linear (GEGLU), dpp_linear
                 x += h Wpo^T + bpo             dpp_linear (accumulate)

With fuse_norm=True the ResNet block's GroupNorms are instead reduced to a
scale and shift per band, image and channel (dpp_groupnorm_sums,
dpp_groupnorm_affine) that the following conv applies with the SiLU as it
loads its input (dpp_conv3x3_norm), so the normalised tensors are never
stored; the results are the same up to rounding.  On B300 the stored path is
the faster one at the SDXL shapes (the convs are bound by shared-memory
bandwidth, which the on-load transform adds to), so it is the default.

The chain runs in place on x (the residual stream).  On one GPU every band's
fresh activations of step t are all in HBM, so the stale state of step t+1 is
simply step t's fresh buffer: the conv inputs, GroupNorm partials and affines
and the K/V state are double-buffered and swapped each step (the refresh costs
nothing).  x itself is overwritten later in the step, so for conv1 only the
rows the next step reads as halo are kept (dpp_refresh_halo).
The time embedding is the same for both images of a guidance pair, so it is
part of conv1's bias.
"""
from __future__ import annotations

import torch

from . import (DPP_ACT_SILU, DPP_BF16, DPP_EPI_GEGLU, DPP_EPI_NONE, dpp_attn_desc,
               dpp_conv3x3_gn, dpp_conv3x3_norm, dpp_conv_desc, dpp_cross_attn,
               dpp_cross_attn_workspace_bytes, dpp_gn_desc, dpp_groupnorm, dpp_groupnorm_affine,
               dpp_groupnorm_apply, dpp_groupnorm_sums, dpp_groupnorm_workspace_bytes,
               dpp_layernorm, dpp_linear, dpp_linear_desc, dpp_ln_desc, dpp_refresh_halo,
               dpp_self_attn, dpp_self_attn_workspace_bytes)

# weight names (torch layouts: conv [C, C, 3, 3] is passed channels-last,
# i.e. [C, 3, 3, C]; Linear [out, in]; biases and affines fp32)
RESNET_WEIGHTS = ("gn1_g", "gn1_b", "conv1_w", "conv1_b", "gn2_g", "gn2_b", "conv2_w", "conv2_b")
TRANSFORMER_WEIGHTS = ("gn_g", "gn_b", "pi_w", "pi_b", "ln1_g", "ln1_b", "wq", "wk", "wv", "wo",
                       "ln2_g", "ln2_b", "xq", "xk", "xv", "xo", "ln3_g", "ln3_b", "ff1_w",
                       "ff1_b", "ff2_w", "ff2_b", "po_w", "po_b")
OPS = ("gn1", "conv1", "gn2", "conv2", "gn", "proj_in", "ln1", "attn1", "ln2", "attn2", "ln3",
       "ff1", "ff2", "proj_out")


def weight_shapes(C, F, c_ctx):
    """Expected shape of every weight (conv weights channels-last)."""
    shapes = {"conv1_w": (C, 3, 3, C), "conv2_w": (C, 3, 3, C), "pi_w": (C, C), "po_w": (C, C),
              "wq": (C, C), "wk": (C, C), "wv": (C, C), "wo": (C, C), "xq": (C, C),
              "xk": (C, c_ctx), "xv": (C, c_ctx), "xo": (C, C), "ff1_w": (2 * F, C),
              "ff1_b": (2 * F,), "ff2_w": (C, F)}
    for k in RESNET_WEIGHTS + TRANSFORMER_WEIGHTS:
        shapes.setdefault(k, (C,))
    return shapes


def full_device(device):
    """torch.device with its index filled in ("cuda" -> "cuda:<current>"),
    so that it compares equal to a tensor's device."""
    dev = torch.device(device)
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    return dev


def check_weights(weights, C, F, c_ctx, dev):
    """The library reads weights through raw pointers, so their shapes,
    types, device and layout are checked here once, on the host."""
    dev = full_device(dev)
    shapes = weight_shapes(C, F, c_ctx)
    missing = [k for k in shapes if k not in weights]
    if missing:
        raise ValueError(f"missing weights: {missing}")
    for k, shape in shapes.items():
        t = weights[k]
        want = torch.float32 if len(shape) == 1 else torch.bfloat16
        if tuple(t.shape) != shape or t.dtype != want or t.device != dev or \
                not t.is_contiguous():
            raise ValueError(f"weight {k}: want {shape} {want} contiguous on {dev}, got "
                             f"{tuple(t.shape)} {t.dtype} on {t.device}")
    return weights


class BlockChain:
    """Buffers, states and the call sequence of one displaced step of the
    chain.  ``weights`` maps the names in RESNET_WEIGHTS and
    TRANSFORMER_WEIGHTS to device tensors (bf16 weights, fp32 biases and
    affines); ff1_w is [2 F, C] (value rows, then gate rows), ff2_w [C, F]."""

    def __init__(self, B, H, W, C, heads, P, G, n_ctx, c_ctx, weights, device,
                 ff_mult=4, eps_gn_res=1e-5, eps_gn_tf=1e-6, eps_ln=1e-5, fuse_norm=False):
        self.B, self.H, self.W, self.C, self.P, self.G = B, H, W, C, P, G
        self.fuse_norm = bool(fuse_norm)
        self.heads, self.n_ctx, self.c_ctx, self.F = heads, n_ctx, c_ctx, ff_mult * C
        dev = full_device(device)
        self.dev = dev
        self.w = check_weights(weights, C, self.F, c_ctx, dev)
        bf = torch.bfloat16
        N, M = H * W, B * H * W
        self.M = M
        act = lambda *s: torch.empty(s, dtype=bf, device=dev)
        img = (B, H, W, C)
        if self.fuse_norm:
            # conv1 reads x; of the previous step's x only the halo rows
            self.xh = [torch.zeros(img, dtype=bf, device=dev) for _ in range(2)]
            self.h1 = [act(*img), act(*img)]  # conv1 output = conv2 input, raw
            aff = lambda: [torch.empty((P, B, C, 2), dtype=torch.float32, device=dev)
                           for _ in range(2)]
            self.aff1, self.aff2 = aff(), aff()
            Hp = H // P
            self.halo_rows = sorted({r for k in range(1, P) for r in (k * Hp - 1, k * Hp)})
        else:
            self.g1 = [act(*img), act(*img)]   # conv1 input: fresh / previous step's
            self.g2 = [act(*img), act(*img)]   # conv2 input
            self.h1 = act(*img)
        self.gt = act(B, N, C)             # transformer GroupNorm output
        self.h = act(B, N, C)              # transformer residual stream
        self.t = act(B, N, C)              # LayerNorm output
        self.u = act(M, self.F)            # gated feed-forward hidden
        stats = lambda: [torch.empty((P, B, G, 2), dtype=torch.float32, device=dev)
                         for _ in range(2)]
        self.st1, self.st2, self.stt = stats(), stats(), stats()
        self.sums = [torch.empty((P, B, G, 2), dtype=torch.float64, device=dev)
                     for _ in range(3)]
        self.kv = [torch.empty((B, N, 2, C), dtype=torch.float16, device=dev) for _ in range(2)]
        self.gn1 = dpp_gn_desc(B, H, W, C, G, P, eps_gn_res, DPP_BF16, 0, DPP_ACT_SILU)
        self.gn2 = dpp_gn_desc(B, H, W, C, G, P, eps_gn_res, DPP_BF16, 0, DPP_ACT_SILU)
        self.gnt = dpp_gn_desc(B, H, W, C, G, P, eps_gn_tf, DPP_BF16, 0, 0)
        self.conv1 = dpp_conv_desc(B, H, W, C, C, P, DPP_BF16, 0, 0)
        self.conv2 = dpp_conv_desc(B, H, W, C, C, P, DPP_BF16, 0, 1)
        self.ln = dpp_ln_desc(M, C, eps_ln, DPP_BF16)
        self.lin = dpp_linear_desc(M, C, C, DPP_BF16, DPP_EPI_NONE, 0)
        self.lin_acc = dpp_linear_desc(M, C, C, DPP_BF16, DPP_EPI_NONE, 1)
        self.ff1 = dpp_linear_desc(M, C, self.F, DPP_BF16, DPP_EPI_GEGLU, 0)
        self.ff2 = dpp_linear_desc(M, self.F, C, DPP_BF16, DPP_EPI_NONE, 1)
        self.sa = dpp_attn_desc(B, H, W, C, heads, C // heads, P, 0, 0, DPP_BF16, 0, 1)
        self.xa = dpp_attn_desc(B, H, W, C, heads, C // heads, 1, n_ctx, c_ctx, DPP_BF16, 0, 1)
        ws = lambda n: torch.empty(max(int(n), 16), dtype=torch.uint8, device=dev)
        self.gn_ws_n = dpp_groupnorm_workspace_bytes(self.gn1)
        self.sa_ws_n = dpp_self_attn_workspace_bytes(self.sa)
        self.xa_ws_n = dpp_cross_attn_workspace_bytes(self.xa)
        self.gn_ws, self.sa_ws, self.xa_ws = ws(self.gn_ws_n), ws(self.sa_ws_n), ws(self.xa_ws_n)
        self.k = 0  # steps taken; step 0 is the synchronous one

    def flops(self):
        """Tensor FLOPs of one step (convolutions, projections, attention
        cores, feed-forward); the normalisations are not counted."""
        M, C, F, n = self.M, self.C, self.F, self.n_ctx
        conv = 2 * (2.0 * M * C * 9 * C)
        lin = 2 * (2.0 * M * C * C) + 2.0 * M * C * 2 * F + 2.0 * M * F * C
        self_attn = 2.0 * M * C * 3 * C + 4.0 * M * self.H * self.W * C + 2.0 * M * C * C
        cross = (2.0 * M * C * C + 2.0 * self.B * n * self.c_ctx * 2 * C + 4.0 * M * n * C
                 + 2.0 * M * C * C)
        return conv + lin + self_attn + cross

    # the displaced states a step publishes for the next one to read
    STATES_FUSED = ("xh", "h1", "aff1", "aff2", "st1", "st2", "stt", "kv")
    STATES_UNFUSED = ("g1", "g2", "st1", "st2", "stt", "kv")

    @property
    def STATES(self):
        return self.STATES_FUSED if self.fuse_norm else self.STATES_UNFUSED

    def _state(self, name, i):
        """The part of state buffer i the next step reads (of x's copy: the
        halo rows)."""
        t = getattr(self, name)[i]
        return t[:, self.halo_rows] if name == "xh" else t

    def state_dict(self):
        """A checkpoint: the step count and the states the next step reads as
        the previous step's (the conv inputs, the GroupNorm partials and the
        K/V state the last step published), copied to host memory after the
        device has finished writing them.  Before the first step there are
        none: the next step is the synchronous one."""
        sd = {"k": self.k}
        if self.k == 0:
            return sd
        i = (self.k - 1) % 2  # the buffers the last step wrote
        torch.cuda.synchronize(self.dev)
        for name in self.STATES:
            sd[name] = self._state(name, i).cpu()
        return sd

    def load_state_dict(self, sd):
        """Resumes from a checkpoint taken by state_dict on a chain of the same
        shapes: the next step reads those states as the previous step's, so
        it computes exactly what the checkpointed chain's next step would."""
        k = int(sd["k"])
        if k > 0:
            i = (k - 1) % 2
            for name in self.STATES:
                if name not in sd:
                    raise ValueError(f"{name}: not in the checkpoint (a chain with "
                                     f"fuse_norm={not self.fuse_norm}?)")
                dst, src = self._state(name, i), sd[name]
                if tuple(src.shape) != tuple(dst.shape) or src.dtype != dst.dtype:
                    raise ValueError(f"{name}: checkpoint {tuple(src.shape)} {src.dtype}, "
                                     f"chain {tuple(dst.shape)} {dst.dtype}")
                if name == "xh":
                    getattr(self, name)[i][:, self.halo_rows] = src.to(self.dev)
                else:
                    dst.copy_(src)
        self.k = k

    def step(self, x, ctx, stream=None, hook=None):
        """One displaced step on x ([B, H, W, C] bf16, updated in place) with
        the text context ctx ([B, n_ctx, c_ctx] bf16).  hook(op, when, tensors),
        when given, is called before ("pre") and after ("post") every op with
        the op's input and output tensors (for tests that check op by op)."""
        for name, t, shape in (("x", x, (self.B, self.H, self.W, self.C)),
                               ("ctx", ctx, (self.B, self.n_ctx, self.c_ctx))):
            if tuple(t.shape) != shape or t.dtype != torch.bfloat16 or \
                    not t.is_contiguous() or t.device != self.dev:
                raise ValueError(f"{name}: want {shape} bf16 contiguous on {self.dev}, got "
                                 f"{tuple(t.shape)} {t.dtype} on {t.device}")
        w, s = self.w, stream
        self._s = stream
        i, j = self.k % 2, 1 - self.k % 2
        first = self.k == 0
        prev = (lambda a: None) if first else (lambda a: a[j])
        B, N, C = self.B, self.H * self.W, self.C
        tok = x.view(B, N, C)
        call = hook or (lambda *a: None)

        def op(name, fn, ins, out):
            call(name, "pre", dict(ins, out=out))
            fn()
            call(name, "post", dict(ins, out=out))

        # ---------------------------------------------------------- ResNet block
        if self.fuse_norm:
            self._resnet_fused(x, i, prev, op)
        else:
            self._resnet_unfused(x, i, prev, op)
        # ------------------------------------------------------ transformer block
        op("gn", lambda: dpp_groupnorm_apply(self.gnt, x, prev(self.stt), self.sums[1],
                                             self.stt[i], w["gn_g"], w["gn_b"], self.gt,
                                             stream=s),
           {"x": x}, self.gt)
        self._transformer(x, tok, ctx, i, prev, op)
        self.k += 1

    def _resnet_fused(self, x, i, prev, op):
        """GroupNorm -> SiLU folded into the convs' loads.  gn1: the band sums
        of x, its affine, and x's halo rows kept for the next step's conv1
        (before conv2 overwrites x); gn2: the affine of conv1's epilogue
        sums."""
        w, s, B, H, W, C, P = self.w, self._s, self.B, self.H, self.W, self.C, self.P

        def gn1():
            dpp_groupnorm_sums(self.gn1, x, self.sums[2], stream=s)
            dpp_groupnorm_affine(self.gn1, self.sums[2], prev(self.st1), self.st1[i],
                                 w["gn1_g"], w["gn1_b"], self.aff1[i], stream=s)
            dpp_refresh_halo(x, self.xh[i], B, H, W * C * 2, P, stream=s)

        op("gn1", gn1, {"x": x}, self.aff1[i])
        op("conv1", lambda: dpp_conv3x3_norm(self.conv1, x, prev(self.xh), self.aff1[i],
                                             prev(self.aff1), DPP_ACT_SILU, w["conv1_w"],
                                             w["conv1_b"], self.h1[i], self.G, self.sums[0],
                                             stream=s),
           {"x": x}, self.h1[i])
        op("gn2", lambda: dpp_groupnorm_affine(self.gn2, self.sums[0], prev(self.st2),
                                               self.st2[i], w["gn2_g"], w["gn2_b"],
                                               self.aff2[i], stream=s),
           {"x": self.h1[i]}, self.aff2[i])
        op("conv2", lambda: dpp_conv3x3_norm(self.conv2, self.h1[i], prev(self.h1),
                                             self.aff2[i], prev(self.aff2), DPP_ACT_SILU,
                                             w["conv2_w"], w["conv2_b"], x, self.G, self.sums[1],
                                             stream=s),
           {"x": self.h1[i]}, x)

    def _resnet_unfused(self, x, i, prev, op):
        """GroupNorm -> SiLU stored, then read by the conv."""
        w, s = self.w, self._s
        op("gn1", lambda: dpp_groupnorm(self.gn1, x, prev(self.st1), self.st1[i], w["gn1_g"],
                                        w["gn1_b"], self.g1[i], self.gn_ws, self.gn_ws_n,
                                        stream=s),
           {"x": x}, self.g1[i])
        op("conv1", lambda: dpp_conv3x3_gn(self.conv1, self.g1[i], prev(self.g1), w["conv1_w"],
                                           w["conv1_b"], self.h1, self.G, self.sums[0],
                                           stream=s),
           {"x": self.g1[i]}, self.h1)
        op("gn2", lambda: dpp_groupnorm_apply(self.gn2, self.h1, prev(self.st2), self.sums[0],
                                              self.st2[i], w["gn2_g"], w["gn2_b"], self.g2[i],
                                              stream=s),
           {"x": self.h1}, self.g2[i])
        op("conv2", lambda: dpp_conv3x3_gn(self.conv2, self.g2[i], prev(self.g2), w["conv2_w"],
                                           w["conv2_b"], x, self.G, self.sums[1], stream=s),
           {"x": self.g2[i]}, x)

    def _transformer(self, x, tok, ctx, i, prev, op):
        w, s = self.w, self._s
        op("proj_in", lambda: dpp_linear(self.lin, self.gt, w["pi_w"], w["pi_b"], self.h,
                                         stream=s),
           {"x": self.gt}, self.h)
        op("ln1", lambda: dpp_layernorm(self.ln, self.h, w["ln1_g"], w["ln1_b"], self.t,
                                        stream=s),
           {"x": self.h}, self.t)
        op("attn1", lambda: dpp_self_attn(self.sa, self.t, w["wq"], w["wk"], w["wv"], w["wo"],
                                          prev(self.kv), self.kv[i], self.h, self.sa_ws,
                                          self.sa_ws_n, stream=s),
           {"x": self.t}, self.h)
        op("ln2", lambda: dpp_layernorm(self.ln, self.h, w["ln2_g"], w["ln2_b"], self.t,
                                        stream=s),
           {"x": self.h}, self.t)
        op("attn2", lambda: dpp_cross_attn(self.xa, self.t, ctx, w["xq"], w["xk"], w["xv"],
                                           w["xo"], self.h, self.xa_ws, self.xa_ws_n, stream=s),
           {"x": self.t, "ctx": ctx}, self.h)
        op("ln3", lambda: dpp_layernorm(self.ln, self.h, w["ln3_g"], w["ln3_b"], self.t,
                                        stream=s),
           {"x": self.h}, self.t)
        op("ff1", lambda: dpp_linear(self.ff1, self.t, w["ff1_w"], w["ff1_b"], self.u,
                                     stream=s),
           {"x": self.t}, self.u)
        op("ff2", lambda: dpp_linear(self.ff2, self.u, w["ff2_w"], w["ff2_b"], self.h,
                                     stream=s),
           {"x": self.u}, self.h)
        op("proj_out", lambda: dpp_linear(self.lin_acc, self.h, w["po_w"], w["po_b"], tok,
                                          stream=s),
           {"x": self.h}, tok)


class BranchPair:
    """Hydiff's condition-based partition of a guided step on one GPU (the
    gist.science summary of Hybridiff, section 基于条件的数据划分): the
    conditional and the unconditional branch as two chains of batch 1, each
    with displaced states of its own.  In the serial stages (warm-up and fully
    connecting, section 自适应并行切换) the branches run one after the other on
    the caller's stream; in the parallel stage each runs on a stream of its
    own, joined by an event, as two devices would run them.  The arithmetic
    of a branch does not depend on the schedule."""

    def __init__(self, H, W, C, heads, P, G, n_ctx, c_ctx, weights, device, **kw):
        dev = full_device(device)
        self.branches = [BlockChain(1, H, W, C, heads, P, G, n_ctx, c_ctx, weights, dev, **kw)
                         for _ in range(2)]
        self.side = torch.cuda.Stream(dev)
        self.forked, self.joined = torch.cuda.Event(), torch.cuda.Event()

    def flops(self):
        return sum(b.flops() for b in self.branches)

    def step(self, xs, ctxs, parallel, stream=None):
        """xs, ctxs: per branch ([1, H, W, C] and [1, n_ctx, c_ctx] bf16; x is
        updated in place); parallel: the stage the switching controller chose
        (DPP_STAGE_PARALLEL) runs the branches on two streams."""
        main = stream if stream is not None else torch.cuda.current_stream()
        if not parallel:
            for b in range(2):
                self.branches[b].step(xs[b], ctxs[b], stream=main)
            return
        self.forked.record(main)
        self.side.wait_event(self.forked)
        self.branches[0].step(xs[0], ctxs[0], stream=main)
        self.branches[1].step(xs[1], ctxs[1], stream=self.side)
        self.joined.record(self.side)
        main.wait_event(self.joined)
