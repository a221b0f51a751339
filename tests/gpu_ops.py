"""Test helpers that run one op through the C ABI (ctypes binding) on cuda:0.

Inputs are CPU torch tensors from ``workloads``; outputs come back as CPU
tensors.  Nothing here computes any part of the method: it allocates device
buffers, builds descriptors and calls the library.
"""
import numpy as np
import torch

import displaced_patch_parallelism_02_b300 as dpp

CODES = {torch.float32: dpp.DPP_F32, torch.bfloat16: dpp.DPP_BF16}
KV_DTYPE = {torch.float32: torch.float32, torch.bfloat16: torch.float16}  # attention state
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}  # max-abs error / RMS of the output


def cuda(t):
    return None if t is None else t.contiguous().to("cuda")


def to_storage(a, dtype):
    """Rounds an fp64 array to a tensor's storage type (RNE) and back: the
    value a layer of that type stores for the next one to read."""
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).to(torch.float64).numpy()


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_rms_close(got, want, rel, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    rms = float(np.sqrt(np.mean(want ** 2)))
    err = float(np.max(np.abs(got - want))) if got.size else 0.0
    assert err <= rel * rms, f"{what}: max|err| {err:.4g} > {rel} x RMS {rms:.4g}"
    return err / rms if rms else 0.0


# ---------------------------------------------------------------- conv
def conv(x, stale, w, bias, P, halo=dpp.DPP_HALO_STALE, stream=None, y_init=None):
    """x, stale: [B,H,W,Ci] (device or CPU); w: [Co,Ci,3,3] torch order;
    halo: a DPP_HALO_* value; y_init: accumulate into a copy of it."""
    x = cuda(x)
    stale = cuda(stale) if stale is not None and stale.device.type == "cpu" else stale
    B, H, W, Ci = x.shape
    Co = w.shape[0]
    wd = cuda(w.permute(0, 2, 3, 1))  # [Co,3,3,Ci]
    y = (torch.empty((B, H, W, Co), dtype=x.dtype, device="cuda") if y_init is None
         else y_init.to("cuda", copy=True).contiguous())
    d = dpp.dpp_conv_desc(B, H, W, Ci, Co, P, CODES[x.dtype], int(halo), int(y_init is not None))
    dpp.dpp_conv3x3(d, x, stale, wd, cuda(bias), y, stream=stream)
    return y


# ------------------------------------------------------------ groupnorm
def gn_desc(x, G, eps, P, band_local=False, act=dpp.DPP_ACT_NONE):
    B, H, W, C = x.shape
    return dpp.dpp_gn_desc(B, H, W, C, G, P, eps, CODES[x.dtype], int(band_local), int(act))


def groupnorm(x, stats_prev, G, eps, gamma, beta, P, y=None, stream=None, band_local=False,
              act=dpp.DPP_ACT_NONE):
    """Returns (y, stats_next) as device tensors."""
    x = cuda(x)
    d = gn_desc(x, G, eps, P, band_local, act)
    B = x.shape[0]
    stats_next = torch.empty((P, B, G, 2), dtype=torch.float32, device="cuda")
    nws = dpp.dpp_groupnorm_workspace_bytes(d)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    if y is None:
        y = torch.empty_like(x)
    dpp.dpp_groupnorm(d, x, cuda(stats_prev) if stats_prev is not None else None, stats_next,
                      cuda(gamma), cuda(beta), y, ws, nws, stream=stream)
    return y, stats_next


def conv_gn(x, stale, w, bias, P, G, stream=None, y_init=None):
    """dpp_conv3x3_gn: returns (y, gn_sums [P,B,G,2] fp64) as device tensors;
    y_init: accumulate into a copy of it."""
    x = cuda(x)
    stale = cuda(stale) if stale is not None and stale.device.type == "cpu" else stale
    B, H, W, Ci = x.shape
    Co = w.shape[0]
    wd = cuda(w.permute(0, 2, 3, 1))  # [Co,3,3,Ci]
    y = (torch.empty((B, H, W, Co), dtype=x.dtype, device="cuda") if y_init is None
         else y_init.to("cuda", copy=True).contiguous())
    sums = torch.empty((P, B, G, 2), dtype=torch.float64, device="cuda")
    d = dpp.dpp_conv_desc(B, H, W, Ci, Co, P, CODES[x.dtype], 0, int(y_init is not None))
    dpp.dpp_conv3x3_gn(d, x, stale, wd, cuda(bias), y, G, sums, stream=stream)
    return y, sums


def groupnorm_apply(x, stats_prev, gn_sums, G, eps, gamma, beta, P, y=None, stream=None,
                    act=dpp.DPP_ACT_NONE):
    """dpp_groupnorm_apply: returns (y, stats_next) as device tensors."""
    x = cuda(x)
    d = gn_desc(x, G, eps, P, act=act)
    B = x.shape[0]
    stats_next = torch.empty((P, B, G, 2), dtype=torch.float32, device="cuda")
    if y is None:
        y = torch.empty_like(x)
    dpp.dpp_groupnorm_apply(d, x, cuda(stats_prev) if stats_prev is not None else None,
                            gn_sums, stats_next, cuda(gamma), cuda(beta), y, stream=stream)
    return y, stats_next


# ------------------------------------------------------------ attention
def attn_desc(x, H, W, heads, P, n_ctx=0, c_ctx=0, band_local=False, accumulate=False):
    B, N, C = x.shape
    assert N == H * W
    return dpp.dpp_attn_desc(B, H, W, C, heads, C // heads, P, n_ctx, c_ctx, CODES[x.dtype],
                             int(band_local), int(accumulate))


def self_attn(x, wts, kv_prev, H, W, heads, P, stream=None, band_local=False, y_init=None):
    """Returns (y, kv_next) as device tensors; y_init: accumulate into a copy."""
    x = cuda(x)
    B, N, C = x.shape
    d = attn_desc(x, H, W, heads, P, band_local=band_local, accumulate=y_init is not None)
    kv_next = torch.empty((B, N, 2, C), dtype=KV_DTYPE[x.dtype], device="cuda")
    y = torch.empty_like(x) if y_init is None else y_init.to("cuda", copy=True).contiguous()
    nws = dpp.dpp_self_attn_workspace_bytes(d)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    w = {k: cuda(v) for k, v in wts.items()}
    dpp.dpp_self_attn(d, x, w["wq"], w["wk"], w["wv"], w["wo"], kv_prev, kv_next, y, ws, nws,
                      stream=stream)
    return y, kv_next


def cross_attn(x, ctx, wts, H, W, heads, stream=None, y_init=None):
    x = cuda(x)
    ctx = cuda(ctx)
    d = attn_desc(x, H, W, heads, 1, ctx.shape[1], ctx.shape[2], accumulate=y_init is not None)
    y = torch.empty_like(x) if y_init is None else y_init.to("cuda", copy=True).contiguous()
    nws = dpp.dpp_cross_attn_workspace_bytes(d)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    w = {k: cuda(v) for k, v in wts.items()}
    dpp.dpp_cross_attn(d, x, ctx, w["wq"], w["wk"], w["wv"], w["wo"], y, ws, nws, stream=stream)
    return y


# ------------------------------------------------------------------ CFG
def cfg(u, c, scale, out=None, ws=None):
    u, c = cuda(u), cuda(c)
    n = u.numel()
    if out is None:
        out = torch.empty_like(u)
    sums = torch.zeros(3, dtype=torch.float64, device="cuda")
    nws = dpp.dpp_cfg_workspace_bytes(n)
    if ws is None:
        ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    dpp.dpp_cfg_combine(u, c, scale, n, out, sums, ws, nws)
    return out, sums, ws


# ------------------------------------------------------ per-token layers
def layernorm(x, gamma, beta, eps, in_place=False):
    """x: [T, C] (CPU or device); returns y as a device tensor."""
    x = cuda(x)
    T, C = x.shape
    y = x if in_place else torch.empty_like(x)
    d = dpp.dpp_ln_desc(T, C, eps, CODES[x.dtype])
    dpp.dpp_layernorm(d, x, cuda(gamma), cuda(beta), y)
    return y


def linear(x, w, bias, geglu=False, y_init=None):
    """x: [M, K]; w: [N, K] ([2N, K] with geglu); returns y [M, N] (device)."""
    x, w = cuda(x), cuda(w)
    M, K = x.shape
    N = w.shape[0] // 2 if geglu else w.shape[0]
    y = (torch.empty((M, N), dtype=x.dtype, device="cuda") if y_init is None
         else y_init.to("cuda", copy=True).contiguous())
    d = dpp.dpp_linear_desc(M, K, N, CODES[x.dtype],
                            dpp.DPP_EPI_GEGLU if geglu else dpp.DPP_EPI_NONE,
                            int(y_init is not None))
    dpp.dpp_linear(d, x, w, cuda(bias), y)
    return y


def bf16_half_ulp_max(want):
    """Half a bf16 ulp at the largest |value| of `want`: the error of storing
    the exact value in bf16, at worst."""
    m = float(np.max(np.abs(want))) if np.size(want) else 0.0
    return 0.0 if m == 0.0 else 2.0 ** (np.floor(np.log2(m)) - 8)


def assert_close_over_bf16_floor(got, want, rel, what=""):
    """Max-abs error within rel x RMS on top of the bf16 storage floor (half an
    ulp of the largest value): for heavy-tailed outputs, such as the gated
    GELU's products, whose largest values round by more than rel x RMS."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    rms = float(np.sqrt(np.mean(want ** 2)))
    floor = bf16_half_ulp_max(want)
    err = float(np.max(np.abs(got - want))) if got.size else 0.0
    assert err <= rel * rms + floor, \
        f"{what}: max|err| {err:.4g} > {rel} x RMS {rms:.4g} + floor {floor:.4g}"
    return err / rms if rms else 0.0
