"""The SDXL-shaped block chain on the GPU against the oracle.

Op level first: the kernel features the chain adds (LayerNorm, the linear map
with bias / residual / gated-GELU epilogues, SiLU after GroupNorm, residual
accumulation in the conv and attention outputs), each against the oracle on
the same seeded inputs, over ragged sizes and both tile paths.  Then the
chain itself (ResNet block + transformer block, DistriFusion's wrapped layers
displaced, the rest per token): two steps, the synchronous one and a
displaced one, judged op by op on each op's own GPU inputs (see check()),
and end to end
against the oracle's fp64 chain within
the bound derived from rounding every stored intermediate to bf16 (simulated
on the CPU: 1.7 % max-abs, 0.38 % RMS of the output), taken with margin as
4e-2 max-abs and 1e-2 RMS.
"""
import numpy as np
import pytest
import torch

import displaced_patch_parallelism_02_b300 as dpp
import oracle
import oracle.blocks as OB
import workloads as wl
from displaced_patch_parallelism_02_b300.chain import OPS, BlockChain
from tests import gpu_ops as G

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16


def draw(shape, seed, dt=BF16, std=1.0):
    return wl.normal(shape, seed, std=std, dtype="bf16" if dt == BF16 else "f32")


def check(got, want, dt, what):
    """The parity bar: 1e-4 x RMS for fp32; for bf16 outputs 2e-2 x RMS on
    top of the bf16 storage floor (half an ulp of the largest value: SiLU
    and gated-GELU outputs reach 7x and 17x their RMS, where storing the exact
    value in bf16 already costs 2.6 % and 4.7 % of RMS)."""
    if dt == F32:
        return G.assert_rms_close(got, want, G.TOL[F32], what)
    return G.assert_close_over_bf16_floor(got, want, G.TOL[BF16], what)


def affine(C, seed):
    return (wl.normal((C,), seed, std=0.1, mean=1.0), wl.normal((C,), seed + 1, std=0.1))


# ------------------------------------------------------------ LayerNorm
@pytest.mark.parametrize("T,C,dt", [(1, 320, BF16), (7, 640, BF16), (1000, 640, BF16),
                                    (333, 1280, BF16), (65, 2048, BF16), (50, 64, F32),
                                    (129, 1024, F32), (40, 8, BF16)])
def test_layernorm_matches_oracle(cuda_device, T, C, dt):
    x = draw((T, C), 700 + C, dt, std=2.0)
    g, b = affine(C, 710)
    y = G.layernorm(x, g, b, 1e-5)
    want = OB.layer_norm(G.f64(x), 1e-5, G.f64(g), G.f64(b))
    check(G.f64(y), want, dt, f"layernorm {T}x{C}")


def test_layernorm_in_place_and_without_affine(cuda_device):
    x = draw((257, 640), 720, BF16) + 3.0  # a large mean: the variance is taken about it
    y = G.layernorm(x, None, None, 1e-5, in_place=True)
    want = OB.layer_norm(G.f64(x), 1e-5)
    check(G.f64(y), want, BF16, "layernorm in place")


# ----------------------------------------------------------- linear maps
@pytest.mark.parametrize("M,K,N", [(1, 320, 64), (300, 640, 640), (1000, 72, 192),
                                   (129, 1280, 320)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_linear_matches_oracle(cuda_device, M, K, N, with_bias):
    x = draw((M, K), 730 + M, BF16)
    w = wl.linear_weight(N, K, 731, "bf16")
    bias = wl.normal((N,), 732, std=0.1) if with_bias else None
    y = G.linear(x, w, bias)
    want = OB.linear(G.f64(x), G.f64(w), None if bias is None else G.f64(bias))
    check(G.f64(y), want, BF16, f"linear {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N", [(300, 640, 640), (77, 320, 64)])
def test_linear_accumulates_into_y(cuda_device, M, K, N):
    x = draw((M, K), 740, BF16)
    w = wl.linear_weight(N, K, 741, "bf16")
    bias = wl.normal((N,), 742, std=0.1)
    r = draw((M, N), 743, BF16)
    y = G.linear(x, w, bias, y_init=r)
    want = G.f64(r) + OB.linear(G.f64(x), G.f64(w), G.f64(bias))
    check(G.f64(y), want, BF16, "linear accumulate")


@pytest.mark.parametrize("M,K,N", [(300, 640, 2560), (129, 320, 64), (1, 320, 1280),
                                   (260, 64, 192)])
@pytest.mark.parametrize("accumulate", [False, True])
def test_geglu_matches_oracle(cuda_device, M, K, N, accumulate):
    x = draw((M, K), 750 + N, BF16)
    w = wl.linear_weight(2 * N, K, 751, "bf16")
    bias = wl.normal((2 * N,), 752, std=0.1)
    r = draw((M, N), 753, BF16) if accumulate else None
    y = G.linear(x, w, bias, geglu=True, y_init=r)
    want = OB.geglu(G.f64(x), G.f64(w), G.f64(bias))
    if accumulate:
        want = want + G.f64(r)
    check(G.f64(y), want, BF16, f"geglu {M}x{K}x{N}")


# ----------------------------------------------------- GroupNorm -> SiLU
@pytest.mark.parametrize("dt", [BF16, F32])
def test_groupnorm_silu_displaced(cuda_device, dt):
    B, H, W, C, Gr, P = 2, 16, 12, 64, 8, 4
    F = draw((B, H, W, C), 760, dt, std=1.5)
    S = wl.perturbed(F, 761, 0.3)
    g, b = affine(C, 762)
    _, st0 = G.groupnorm(S, None, Gr, 1e-5, g, b, P)
    y, _ = G.groupnorm(F, st0, Gr, 1e-5, g, b, P, act=dpp.DPP_ACT_SILU)
    want = OB.silu(oracle.displaced_groupnorm(G.f64(F), G.f64(S), Gr, 1e-5, G.f64(g),
                                              G.f64(b), P))
    check(G.f64(y), want, dt, "groupnorm + SiLU")


def test_groupnorm_apply_silu_on_conv_sums(cuda_device):
    B, H, W, C, Gr, P = 2, 16, 20, 64, 8, 4
    x = draw((B, H, W, C), 770, BF16)
    w = wl.conv_weight(C, C, 771, "bf16")
    g, b = affine(C, 772)
    y1, sums = G.conv_gn(x, None, w, None, P, Gr)
    y, _ = G.groupnorm_apply(y1, None, sums, Gr, 1e-6, g, b, P, act=dpp.DPP_ACT_SILU)
    want = OB.silu(oracle.groupnorm(G.f64(y1), Gr, 1e-6, G.f64(g), G.f64(b)))
    check(G.f64(y), want, BF16, "groupnorm_apply + SiLU")


# ------------------------------------------------- residual accumulation
@pytest.mark.parametrize("dt", [BF16, F32])
def test_conv_accumulates_into_y(cuda_device, dt):
    B, H, W, C, P = 1, 16, 136, 64, 4  # two 128-pixel segments per row, ragged
    F = draw((B, H, W, C), 780, dt)
    S = wl.perturbed(F, 781, 0.05)
    w = wl.conv_weight(C, C, 782, "bf16" if dt == BF16 else "f32")
    bias = wl.normal((C,), 783, std=0.1)
    r = draw((B, H, W, C), 784, dt)
    y = G.conv(F, S, w, bias, P, y_init=r)
    want = G.f64(r) + oracle.displaced_conv3x3(G.f64(F), G.f64(S), G.f64(w), G.f64(bias), P)
    check(G.f64(y), want, dt, "conv accumulate")


def test_conv_gn_accumulates_and_sums_the_stored_output(cuda_device):
    B, H, W, C, Gr, P = 2, 8, 40, 128, 32, 2
    F = draw((B, H, W, C), 790, BF16)
    S = wl.perturbed(F, 791, 0.05)
    w = wl.conv_weight(C, C, 792, "bf16")
    r = draw((B, H, W, C), 793, BF16)
    y, sums = G.conv_gn(F, S, w, None, P, Gr, y_init=r)
    want = G.f64(r) + oracle.displaced_conv3x3(G.f64(F), G.f64(S), G.f64(w), None, P)
    check(G.f64(y), want, BF16, "conv_gn accumulate")
    # the sums are those of y as stored (residual included)
    ref = oracle.groupnorm_partials(G.f64(y), Gr, P)
    got = sums.cpu().numpy()
    assert np.allclose(got, ref, rtol=1e-5, atol=1e-3 * np.abs(ref).max())


@pytest.mark.parametrize("dt", [BF16, F32])
def test_self_attention_accumulates_into_y(cuda_device, dt):
    B, Hh, Ww, C, heads, P = 1, 16, 20, 128, 2, 4
    X = draw((B, Hh * Ww, C), 800, dt)
    Xs = wl.perturbed(X, 801, 0.05)
    wts = {k: wl.linear_weight(C, C, 802 + i, "bf16" if dt == BF16 else "f32")
           for i, k in enumerate(("wq", "wk", "wv", "wo"))}
    _, kv0 = G.self_attn(Xs, wts, None, Hh, Ww, heads, P)
    r = draw((B, Hh * Ww, C), 806, dt)
    y, _ = G.self_attn(X, wts, kv0, Hh, Ww, heads, P, y_init=r)
    ww = {k: G.f64(v) for k, v in wts.items()}
    want = G.f64(r) + oracle.displaced_self_attention(G.f64(X), G.f64(Xs), ww["wq"], ww["wk"],
                                                      ww["wv"], ww["wo"], heads, P)
    check(G.f64(y), want, dt, "self-attention accumulate")


def test_cross_attention_accumulates_into_y(cuda_device):
    B, Hh, Ww, C, heads, n_ctx, c_ctx = 2, 8, 24, 128, 2, 77, 256
    X = draw((B, Hh * Ww, C), 810, BF16)
    ctx = draw((B, n_ctx, c_ctx), 811, BF16)
    wts = {"wq": wl.linear_weight(C, C, 812, "bf16"), "wk": wl.linear_weight(C, c_ctx, 813, "bf16"),
           "wv": wl.linear_weight(C, c_ctx, 814, "bf16"), "wo": wl.linear_weight(C, C, 815, "bf16")}
    r = draw((B, Hh * Ww, C), 816, BF16)
    y = G.cross_attn(X, ctx, wts, Hh, Ww, heads, y_init=r)
    ww = {k: G.f64(v) for k, v in wts.items()}
    want = G.f64(r) + oracle.cross_attention(G.f64(X), G.f64(ctx), ww["wq"], ww["wk"], ww["wv"],
                                             ww["wo"], heads)
    check(G.f64(y), want, BF16, "cross-attention accumulate")


# ------------------------------------------------------------ the chain
CH = wl.CHAINS["chain_small"]
EPS_GN_RES, EPS_GN_TF, EPS_LN = 1e-5, 1e-6, 1e-5


def chain_device_weights(wts):
    dev = {}
    for k, v in wts.items():
        if k.startswith("conv") and k.endswith("_w"):
            v = v.permute(0, 2, 3, 1)  # [C, 3, 3, C]: channels-last
        dev[k] = v.contiguous().to("cuda")
    return dev


GN_KEYS = {"gn1": ("gn1_g", "gn1_b", EPS_GN_RES), "gn2": ("gn2_g", "gn2_b", EPS_GN_RES),
           "gn": ("gn_g", "gn_b", EPS_GN_TF)}


def apply_affine(x64, aff, P):
    """y = x * a + s with band p's row of the affine table [P, B, C, 2] on band
    p's rows."""
    a = G.f64(aff)
    H = x64.shape[1]
    Hp = H // P
    y = np.empty_like(x64)
    for p in range(P):
        sl = slice(p * Hp, (p + 1) * Hp)
        y[:, sl] = x64[:, sl] * a[p, :, None, None, :, 0] + a[p, :, None, None, :, 1]
    return y


def oracle_op_fused(name, pre, prev, norm_prev, W, ch):
    """The fused ResNet ops: gn1/gn2 publish an affine table, so they are
    judged by the displaced GroupNorm it applies; conv1/conv2 read the raw
    tensor and normalise it on load, so the oracle composes SiLU(displaced
    GroupNorm) of the op's GPU input (stale statistics from the previous
    step's input) with the displaced conv, whose stale input is the
    normalised tensor the oracle formed at the previous step.  Returns
    (value to compare, normalised input for the next step or None)."""
    P, Gr = ch.P, ch.G
    f = lambda k: G.f64(pre[k])
    S = lambda k: f(k) if prev is None else G.f64(prev[k])
    g = {"gn1": "gn1", "gn2": "gn2", "conv1": "gn1", "conv2": "gn2"}[name]
    kg, kb, eps = GN_KEYS[g]
    gn = oracle.displaced_groupnorm(f("x"), S("x"), Gr, eps, W[kg], W[kb], P)
    if name in ("gn1", "gn2"):
        return gn, None
    z = OB.silu(gn)
    z_prev = z if norm_prev is None else norm_prev
    y = oracle.displaced_conv3x3(z, z_prev, W[name + "_w"], W[name + "_b"], P)
    return (y + f("out") if name == "conv2" else y), z


def oracle_op(name, pre, post, prev, W, ch):
    """The oracle's value of one op of the chain on the GPU's own inputs
    (upcast); prev: the same op's inputs at the previous step (its stale
    state), or None for the synchronous step."""
    f = lambda k: G.f64(pre[k])
    S = lambda k: f(k) if prev is None else G.f64(prev[k])
    P, Gr, heads = ch.P, ch.G, ch.heads
    B, H, Wd, C = ch.B, ch.H, ch.W, ch.C
    img = lambda a: a.reshape(B, H, Wd, -1)
    tok = lambda a: a.reshape(B, H * Wd, -1)
    if name in ("gn1", "gn2", "gn"):
        keys = {"gn1": ("gn1_g", "gn1_b", EPS_GN_RES), "gn2": ("gn2_g", "gn2_b", EPS_GN_RES),
                "gn": ("gn_g", "gn_b", EPS_GN_TF)}[name]
        y = oracle.displaced_groupnorm(img(f("x")), img(S("x")), Gr, keys[2], W[keys[0]],
                                       W[keys[1]], P)
        return OB.silu(y) if name != "gn" else y
    if name in ("conv1", "conv2"):
        y = oracle.displaced_conv3x3(f("x"), S("x"), W[name + "_w"], W[name + "_b"], P)
        return y + f("out") if name == "conv2" else y
    if name == "proj_in":
        return OB.linear(f("x"), W["pi_w"], W["pi_b"])
    if name in ("ln1", "ln2", "ln3"):
        return OB.layer_norm(f("x"), EPS_LN, W[name + "_g"], W[name + "_b"])
    if name == "attn1":
        return f("out") + oracle.displaced_self_attention(tok(f("x")), tok(S("x")), W["wq"],
                                                          W["wk"], W["wv"], W["wo"], heads, P)
    if name == "attn2":
        return f("out") + oracle.cross_attention(f("x"), f("ctx"), W["xq"], W["xk"], W["xv"],
                                                 W["xo"], heads)
    if name == "ff1":
        return OB.geglu(f("x"), W["ff1_w"], W["ff1_b"])
    if name == "ff2":
        return f("out") + OB.linear(f("x"), W["ff2_w"], W["ff2_b"]).reshape(f("out").shape)
    if name == "proj_out":
        return f("out") + OB.linear(f("x"), W["po_w"], W["po_b"])
    raise KeyError(name)


@pytest.mark.parametrize("fuse_norm", [True, False])
def test_chain_two_steps_op_by_op_and_end_to_end(cuda_device, fuse_norm):
    ch = CH
    wts = wl.chain_weights(ch)
    W = {k: G.f64(v) for k, v in wts.items()}
    xs, ctx = wl.chain_inputs(ch, 1)
    chain = BlockChain(ch.B, ch.H, ch.W, ch.C, ch.heads, ch.P, ch.G, ch.n_ctx, ch.c_ctx,
                       chain_device_weights(wts), "cuda", ff_mult=ch.ff_mult,
                       fuse_norm=fuse_norm)
    fused_ops = ("gn1", "conv1", "gn2", "conv2") if fuse_norm else ()
    norm_prev = {}
    ctx_d = ctx.to("cuda")
    seen = {}

    def hook(name, when, tensors):
        torch.cuda.synchronize()
        seen[(name, when)] = {k: v.detach().to("cpu", copy=True) for k, v in tensors.items()}

    prev_inputs = None
    outs = []
    for step in range(2):
        seen.clear()
        x = xs[step].to("cuda", copy=True)
        chain.step(x, ctx_d, hook=hook)
        torch.cuda.synchronize()
        assert dpp.dpp_device_status() == dpp.DPP_OK
        inputs = {}
        for name in OPS:
            pre, post = seen[(name, "pre")], seen[(name, "post")]
            inputs[name] = pre
            prev = None if prev_inputs is None else prev_inputs[name]
            if name in ("gn1", "gn2") and fuse_norm:
                want, _ = oracle_op_fused(name, pre, prev, None, W, ch)
                got = apply_affine(G.f64(pre["x"]), post["out"], ch.P)
                G.assert_rms_close(got, want, 1e-4, f"step {step} op {name} (affine)")
                continue
            if name in fused_ops:
                want, norm_prev[name] = oracle_op_fused(name, pre, prev, norm_prev.get(name),
                                                        W, ch)
            else:
                want = oracle_op(name, pre, post, prev, W, ch)
            got = G.f64(post["out"]).reshape(want.shape)
            check(got, want, BF16, f"step {step} op {name}")
        prev_inputs = inputs
        outs.append(G.f64(x))
    # end to end against the fp64 chain on the same inputs
    res = {k: W[k] for k in ("gn1_g", "gn1_b", "conv1_w", "conv1_b", "gn2_g", "gn2_b",
                             "conv2_w", "conv2_b")}
    tf = {k: v for k, v in W.items() if k not in res}
    st = None
    for step in range(2):
        want, st = OB.block_chain(G.f64(xs[step]), G.f64(ctx), st, res, tf, ch.heads, ch.P,
                                  ch.G, EPS_GN_RES, EPS_GN_TF, EPS_LN)
        rms = float(np.sqrt(np.mean(want ** 2)))
        err = outs[step] - want
        assert np.abs(err).max() <= 4e-2 * rms, (step, np.abs(err).max() / rms)
        assert float(np.sqrt(np.mean(err ** 2))) <= 1e-2 * rms, step


@pytest.mark.parametrize("fuse_norm,launches", [(True, 24), (False, 22)])
def test_chain_launches_only_library_kernels_and_repeats(cuda_device, fuse_norm, launches):
    # the same input twice: the displaced second step reads states equal to
    # its own fresh inputs, so it reproduces the synchronous output
    ch = CH
    wts = wl.chain_weights(ch)
    xs, ctx = wl.chain_inputs(ch, 0)
    chain = BlockChain(ch.B, ch.H, ch.W, ch.C, ch.heads, ch.P, ch.G, ch.n_ctx, ch.c_ctx,
                       chain_device_weights(wts), "cuda", ff_mult=ch.ff_mult,
                       fuse_norm=fuse_norm)
    ctx_d = ctx.to("cuda")
    outs = []
    for step in range(2):
        x = xs[0].to("cuda", copy=True)
        n0 = dpp.dpp_launch_count()
        chain.step(x, ctx_d)
        torch.cuda.synchronize()
        assert dpp.dpp_launch_count() - n0 == launches
        outs.append(G.f64(x))
    check(outs[1], outs[0], BF16, "repeated input, displaced vs synchronous step")


@pytest.mark.parametrize("fuse_norm", [True, False])
def test_chain_resumes_bit_identical_from_a_checkpoint(cuda_device, fuse_norm):
    """Checkpoint / resume of the displaced states: a chain stepped four times
    without a break, against one stepped twice, checkpointed to host memory,
    dropped, and a fresh chain (new device buffers, garbage before the load)
    resumed from the checkpoint for the last two steps.  The latent and every
    state the last step publishes are bit-identical."""
    ch = CH
    wts = chain_device_weights(wl.chain_weights(ch))
    xs, ctx = wl.chain_inputs(ch, 3)
    ctx_d = ctx.to("cuda")
    args = (ch.B, ch.H, ch.W, ch.C, ch.heads, ch.P, ch.G, ch.n_ctx, ch.c_ctx, wts, "cuda")
    kw = dict(ff_mult=ch.ff_mult, fuse_norm=fuse_norm)

    def run(chain, steps, x):
        for s in steps:
            x.copy_(x + 0.0 if s == 0 else xs[s].to("cuda") * 0.5 + x * 0.5)
            chain.step(x, ctx_d)
        torch.cuda.synchronize()
        return x

    full = BlockChain(*args, **kw)
    x_full = run(full, range(4), xs[0].to("cuda", copy=True))
    first = BlockChain(*args, **kw)
    x_part = run(first, range(2), xs[0].to("cuda", copy=True))
    sd = first.state_dict()
    assert sd["k"] == 2 and all(name in sd for name in first.STATES)
    x_host = x_part.cpu()
    del first, x_part
    torch.cuda.empty_cache()
    resumed = BlockChain(*args, **kw)
    for name in resumed.STATES:  # the fresh chain's buffers hold garbage
        for t in getattr(resumed, name):
            t.view(torch.uint8).fill_(0x7f)
    resumed.load_state_dict(sd)
    x_res = run(resumed, range(2, 4), x_host.to("cuda"))
    assert dpp.dpp_device_status() == dpp.DPP_OK
    assert torch.equal(x_res, x_full)
    got, want = resumed.state_dict(), full.state_dict()
    assert got["k"] == want["k"] == 4
    for name in resumed.STATES:
        assert torch.equal(got[name], want[name]), name


def test_branch_schedules_agree(cuda_device):
    """Hydiff's condition-based partition on one GPU: the two branches as
    chains of batch 1, serially or on two streams, three steps each (the
    synchronous one and two displaced).  Serial and two-stream results are
    bit-identical; both match the batched chain at the parity bar."""
    from displaced_patch_parallelism_02_b300.chain import BranchPair
    ch = CH
    wts = chain_device_weights(wl.chain_weights(ch))
    xs, ctx = wl.chain_inputs(ch, 2)
    ctx_d = ctx.to("cuda")
    args = (ch.H, ch.W, ch.C, ch.heads, ch.P, ch.G, ch.n_ctx, ch.c_ctx, wts, "cuda")
    batched = BlockChain(ch.B, *args)
    ref = []
    for s in range(3):
        x = xs[s].to("cuda", copy=True)
        batched.step(x, ctx_d)
        ref.append(x.cpu())
    ctxs = [ctx_d[b:b + 1].contiguous() for b in range(2)]
    runs = {}
    for name, pattern in (("serial", (False, False, False)), ("two_stream", (False, True, True))):
        pair = BranchPair(*args)
        outs = []
        for s, par in enumerate(pattern):
            xb = [xs[s][b:b + 1].to("cuda", copy=True) for b in range(2)]
            pair.step(xb, ctxs, par)
            torch.cuda.synchronize()
            outs.append(torch.cat(xb).cpu())
        runs[name] = outs
    assert dpp.dpp_device_status() == dpp.DPP_OK
    for s in range(3):
        assert torch.equal(runs["serial"][s], runs["two_stream"][s]), s
        check(G.f64(runs["two_stream"][s]), G.f64(ref[s]), BF16, f"branches vs batched, step {s}")
