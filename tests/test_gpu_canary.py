"""Guard bands around every buffer an entry point writes.

compute-sanitizer is closed on this machine, so out-of-bounds writes are looked
for directly: each output, state and workspace buffer sits between two 4 KB
bands of seeded random bytes, the call runs on ragged shapes (tiles cut by
the image width, the channel count, the token count and the band size), and
afterwards both bands must hold exactly the bytes they started with.  Every
tensor-core and TMA path of the library is covered: conv (plain and with the
GroupNorm sums), GroupNorm (two reads, and one pass on the conv's sums),
self-attention (with its K/V state), cross-attention (one call, and the
per-prompt K/V with the cached step), the guidance combine, the refresh, the
linear map (plain, bias, gated GELU), LayerNorm, and the GroupNorm -> SiLU
-> conv path (band sums, per-band affine, the normalising conv, the halo
refresh).
"""
import pytest
import torch

import displaced_patch_parallelism_02_b300 as dpp

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side of a buffer
BF16, F16, F32, F64 = torch.bfloat16, torch.float16, torch.float32, torch.float64


class Guarded:
    """A device tensor of `shape` and `dtype` between two guard bands; the
    whole allocation starts as seeded random bytes."""

    def __init__(self, shape, dtype, seed):
        n = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
        g = torch.Generator(device="cpu").manual_seed(seed)
        self.pattern = torch.randint(0, 256, (n + 2 * GUARD,), dtype=torch.uint8, generator=g)
        self.buf = self.pattern.to("cuda")
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(shape)

    def intact(self):
        b = self.buf.cpu()
        return torch.equal(b[:GUARD], self.pattern[:GUARD]) and \
            torch.equal(b[-GUARD:], self.pattern[-GUARD:])


def rnd(shape, seed, dtype=BF16, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(dtype).to("cuda")


def check(*guarded):
    torch.cuda.synchronize()
    assert dpp.dpp_device_status() == dpp.DPP_OK
    for k, gb in enumerate(guarded):
        assert gb.intact(), f"guard band of buffer {k} overwritten"


def ws(n, seed):
    return Guarded((max(n, 16),), torch.uint8, seed)


def test_conv_and_conv_gn_write_inside_their_buffers(cuda_device):
    # W 200 = one 128-pixel tile + 72; C_out 96 inside a wider column tile;
    # 3 bands of 4 rows
    B, H, W, Ci, Co, P, G = 2, 12, 200, 64, 96, 3, 32
    x, stale = rnd((B, H, W, Ci), 1), rnd((B, H, W, Ci), 2)
    w, bias = rnd((Co, 3, 3, Ci), 3, scale=0.05), rnd((Co,), 4, F32)
    d = dpp.dpp_conv_desc(B, H, W, Ci, Co, P, dpp.DPP_BF16, dpp.DPP_HALO_STALE, 0)
    y = Guarded((B, H, W, Co), BF16, 10)
    dpp.dpp_conv3x3(d, x, stale, w, bias, y.t)
    check(y)
    y2, sums = Guarded((B, H, W, Co), BF16, 11), Guarded((P, B, G, 2), F64, 12)
    dpp.dpp_conv3x3_gn(d, x, stale, w, bias, y2.t, G, sums.t)
    check(y2, sums)


def test_groupnorm_writes_inside_its_buffers(cuda_device):
    B, H, W, C, G, P = 2, 12, 20, 96, 32, 3
    x = rnd((B, H, W, C), 20)
    gamma, beta = rnd((C,), 21, F32), rnd((C,), 22, F32)
    d = dpp.dpp_gn_desc(B, H, W, C, G, P, 1e-5, dpp.DPP_BF16, 0, 0)
    st_prev = torch.rand((P, B, G, 2), device="cuda") + 1.0
    st_next, y = Guarded((P, B, G, 2), F32, 23), Guarded((B, H, W, C), BF16, 24)
    n = dpp.dpp_groupnorm_workspace_bytes(d)
    w = ws(n, 25)
    dpp.dpp_groupnorm(d, x, st_prev, st_next.t, gamma, beta, y.t, w.t, n)
    check(st_next, y, w)
    # one pass on band sums (as dpp_conv3x3_gn writes them)
    sums = torch.rand((P, B, G, 2), dtype=F64, device="cuda") * 100 + 200
    st2, y2 = Guarded((P, B, G, 2), F32, 26), Guarded((B, H, W, C), BF16, 27)
    dpp.dpp_groupnorm_apply(d, x, st_prev, sums, st2.t, gamma, beta, y2.t)
    check(st2, y2)


def test_norm_conv_path_writes_inside_its_buffers(cuda_device):
    # the GroupNorm -> SiLU -> conv path: band sums, per-band affine, the
    # normalising conv (W 200 = 128 + 72, C_in 96 = 64 + 32, C_out 96 inside
    # a 128-column tile, with its epilogue sums) and the halo refresh
    B, H, W, Ci, Co, P, G = 2, 12, 200, 96, 96, 3, 8
    x, stale = rnd((B, H, W, Ci), 90), rnd((B, H, W, Ci), 91)
    gamma, beta = rnd((Ci,), 92, F32), rnd((Ci,), 93, F32)
    gd = dpp.dpp_gn_desc(B, H, W, Ci, G, P, 1e-5, dpp.DPP_BF16, 0, 0)
    sums = Guarded((P, B, G, 2), F64, 94)
    dpp.dpp_groupnorm_sums(gd, x, sums.t)
    check(sums)
    aff, st = Guarded((P, B, Ci, 2), F32, 95), Guarded((P, B, G, 2), F32, 96)
    dpp.dpp_groupnorm_affine(gd, sums.t, None, st.t, gamma, beta, aff.t)
    check(aff, st, sums)
    w = rnd((Co, 3, 3, Ci), 97, scale=0.05)
    d = dpp.dpp_conv_desc(B, H, W, Ci, Co, P, dpp.DPP_BF16, dpp.DPP_HALO_STALE, 0)
    y, ys = Guarded((B, H, W, Co), BF16, 98), Guarded((P, B, 32, 2), F64, 99)
    dpp.dpp_conv3x3_norm(d, x, stale, aff.t, aff.t, dpp.DPP_ACT_SILU, w, None, y.t, 32, ys.t)
    check(y, ys, aff)
    halo = Guarded((B, H, W, Ci), BF16, 100)
    dpp.dpp_refresh_halo(x, halo.t, B, H, W * Ci * 2, P)
    check(halo)


def test_self_attention_writes_inside_its_buffers(cuda_device):
    # 40 tokens per band: ragged against every tile; two heads
    B, H, W, heads, P = 2, 6, 20, 2, 3
    C, N = 64 * heads, H * W
    x = rnd((B, N, C), 30)
    wq, wk, wv, wo = (rnd((C, C), 31 + k, scale=C ** -0.5) for k in range(4))
    kv_prev = rnd((B, N, 2, C), 35, F16, 0.5)
    d = dpp.dpp_attn_desc(B, H, W, C, heads, 64, P, 0, 0, dpp.DPP_BF16, 0, 0)
    kv_next, y = Guarded((B, N, 2, C), F16, 36), Guarded((B, N, C), BF16, 37)
    n = dpp.dpp_self_attn_workspace_bytes(d)
    w = ws(n, 38)
    dpp.dpp_self_attn(d, x, wq, wk, wv, wo, kv_prev, kv_next.t, y.t, w.t, n)
    check(kv_next, y, w)


@pytest.mark.parametrize("n_ctx", [77, 128])
def test_cross_attention_writes_inside_its_buffers(cuda_device, n_ctx):
    # 300 queries per image: two full query tiles and a ragged one
    B, H, W, heads, c_ctx = 2, 10, 30, 2, 96
    C, N = 64 * heads, H * W
    x, ctx = rnd((B, N, C), 40), rnd((B, n_ctx, c_ctx), 41)
    wq, wo = rnd((C, C), 42, scale=C ** -0.5), rnd((C, C), 43, scale=C ** -0.5)
    wk, wv = rnd((C, c_ctx), 44, scale=c_ctx ** -0.5), rnd((C, c_ctx), 45, scale=c_ctx ** -0.5)
    d = dpp.dpp_attn_desc(B, H, W, C, heads, 64, 1, n_ctx, c_ctx, dpp.DPP_BF16, 0, 0)
    y = Guarded((B, N, C), BF16, 46)
    n = dpp.dpp_cross_attn_workspace_bytes(d)
    w = ws(n, 47)
    dpp.dpp_cross_attn(d, x, ctx, wq, wk, wv, wo, y.t, w.t, n)
    check(y, w)
    kv = Guarded((B, n_ctx, 2, C), F16, 48)
    dpp.dpp_cross_attn_kv(d, ctx, wk, wv, kv.t)
    check(kv)
    y2 = Guarded((B, N, C), BF16, 49)
    n2 = dpp.dpp_cross_attn_cached_workspace_bytes(d)
    w2 = ws(n2, 50)
    dpp.dpp_cross_attn_cached(d, x, kv.t, wq, wo, y2.t, w2.t, n2)
    check(y2, w2, kv)
    assert torch.equal(y.t, y2.t)  # the one call is the two parts back to back


def test_cfg_and_refresh_write_inside_their_buffers(cuda_device):
    n = 1003  # not a multiple of the 16-byte vector or of any block size
    u, c = rnd((n,), 60, F32), rnd((n,), 61, F32)
    out, sums = Guarded((n,), F32, 62), Guarded((3,), F64, 63)
    nws = dpp.dpp_cfg_workspace_bytes(n)
    w = ws(nws, 64)
    w.t[:16].zero_()  # the workspace's completion counter starts at zero
    dpp.dpp_cfg_combine(u, c, 7.5, n, out.t, sums.t, w.t, nws)
    check(out, sums, w)
    B, H, W, C, P = 2, 12, 20, 96, 3
    fresh = rnd((B, H, W, C), 65)
    stale = Guarded((B, H, W, C), BF16, 66)
    dpp.dpp_refresh_stale(fresh, stale.t, B, H, W * C * 2, P, 0b101)
    check(stale)


@pytest.mark.parametrize("M,K,N,epi,with_bias", [
    (300, 128, 192, "none", False), (300, 128, 192, "none", True), (257, 640, 128, "geglu", True)])
def test_linear_writes_inside_its_buffers(cuda_device, M, K, N, epi, with_bias):
    rows = 2 * N if epi == "geglu" else N
    x, w = rnd((M, K), 70), rnd((rows, K), 71, scale=K ** -0.5)
    bias = rnd((rows,), 72, F32) if with_bias else None
    e = dpp.DPP_EPI_GEGLU if epi == "geglu" else dpp.DPP_EPI_NONE
    d = dpp.dpp_linear_desc(M, K, N, dpp.DPP_BF16, e, 0)
    y = Guarded((M, N), BF16, 73)
    dpp.dpp_linear(d, x, w, bias, y.t)
    check(y)


def test_layernorm_writes_inside_its_buffers(cuda_device):
    T, C = 77, 320
    x = rnd((T, C), 80)
    g, b = rnd((C,), 81, F32), rnd((C,), 82, F32)
    d = dpp.dpp_ln_desc(T, C, 1e-5, dpp.DPP_BF16)
    y = Guarded((T, C), BF16, 83)
    dpp.dpp_layernorm(d, x, g, b, y.t)
    check(y)
