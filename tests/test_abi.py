"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/dpp.h declares, and rejects bad arguments on the host before any
CUDA call (so these run on a machine without a device).

The pointers below are fake, 16-byte-aligned addresses: every call here must
fail validation, which never dereferences them.
"""
import ctypes
import os
import re

import pytest

import displaced_patch_parallelism_02_b300 as dpp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dpp.h")

A = 0x7f0000000000  # fake device addresses, far apart
Bp = 0x7f1000000000
Cp = 0x7f2000000000
Dp = 0x7f3000000000
Ep = 0x7f4000000000


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dpp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_calls_and_helpers():
    names = declared_functions()
    for n in ["dpp_conv3x3", "dpp_groupnorm", "dpp_self_attn", "dpp_cfg_combine",
              "dpp_refresh_stale", "dpp_cross_attn", "dpp_status_string", "dpp_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(dpp.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_has_every_declared_name():
    missing = [n for n in declared_functions() if not callable(getattr(dpp, n, None))]
    assert not missing, missing


def test_status_strings_and_version():
    assert dpp.dpp_status_string(dpp.DPP_OK) == "DPP_OK"
    assert dpp.dpp_status_string(dpp.DPP_ERR_ALIAS) == "DPP_ERR_ALIAS"
    assert dpp.dpp_status_string(99) == "DPP_ERR_UNKNOWN"
    assert dpp.dpp_version() >= 100


def conv(**kw):
    d = dict(B=1, H=8, W=8, C_in=16, C_out=16, P=2, dtype=dpp.DPP_BF16, halo=0)
    d.update(kw)
    return dpp.dpp_conv_desc(**d)


@pytest.mark.parametrize("kw,ptrs,want", [
    (dict(H=9), {}, dpp.DPP_ERR_INVALID_ARG),             # H % P != 0
    (dict(C_in=12), {}, dpp.DPP_ERR_INVALID_ARG),         # bf16 needs C % 8 == 0
    (dict(P=0), {}, dpp.DPP_ERR_INVALID_ARG),
    (dict(dtype=5), {}, dpp.DPP_ERR_INVALID_ARG),
    (dict(halo=3), {}, dpp.DPP_ERR_INVALID_ARG),          # not a dpp_halo value
    ({}, dict(x=0), dpp.DPP_ERR_INVALID_ARG),             # null input
    ({}, dict(x=A + 8), dpp.DPP_ERR_ALIGN),
    ({}, dict(y=A + 64), dpp.DPP_ERR_ALIAS),              # output overlaps input
    ({}, dict(y=Bp + 32), dpp.DPP_ERR_ALIAS),             # output overlaps stale
])
def test_conv_validation(kw, ptrs, want):
    p = dict(x=A, stale=Bp, w=Cp, bias=None, y=Dp)
    p.update(ptrs)
    st = dpp.dpp_conv3x3(conv(**kw), p["x"], p["stale"], p["w"], p["bias"], p["y"],
                         stream=0, raise_on_error=False)
    assert st == want


def gn(**kw):
    d = dict(B=1, H=8, W=8, C=32, G=4, P=2, eps=1e-5, dtype=dpp.DPP_BF16)
    d.update(kw)
    return dpp.dpp_gn_desc(**d)


def test_gn_workspace_query_is_pure_and_positive():
    assert dpp.dpp_groupnorm_workspace_bytes(gn()) > 0
    assert dpp.dpp_groupnorm_workspace_bytes(gn(C=30)) == 0  # invalid desc


@pytest.mark.parametrize("kw,ptrs,want", [
    (dict(C=30), {}, dpp.DPP_ERR_INVALID_ARG),            # C % G
    (dict(H=7), {}, dpp.DPP_ERR_INVALID_ARG),             # H % P
    ({}, dict(ws=0), dpp.DPP_ERR_WORKSPACE),
    ({}, dict(ws_bytes=16), dpp.DPP_ERR_WORKSPACE),
    ({}, dict(stats_prev=Ep + 16), dpp.DPP_ERR_ALIAS),    # prev overlaps next
    ({}, dict(gamma=Cp), dpp.DPP_ERR_INVALID_ARG),        # gamma without beta
    ({}, dict(y=A + 32), dpp.DPP_ERR_ALIAS),              # partial in-place overlap
    ({}, dict(stats_next=0), dpp.DPP_ERR_INVALID_ARG),
])
def test_gn_validation(kw, ptrs, want):
    d = gn(**kw)
    p = dict(x=A, stats_prev=None, stats_next=Ep, gamma=None, beta=None, y=Dp, ws=Bp,
             ws_bytes=1 << 20)
    p.update(ptrs)
    st = dpp.dpp_groupnorm(d, p["x"], p["stats_prev"], p["stats_next"], p["gamma"], p["beta"],
                           p["y"], p["ws"], p["ws_bytes"], stream=0, raise_on_error=False)
    assert st == want


def attn(**kw):
    d = dict(B=1, H=8, W=8, C=128, heads=2, head_dim=64, P=2, n_ctx=0, c_ctx=0,
             dtype=dpp.DPP_BF16)
    d.update(kw)
    return dpp.dpp_attn_desc(**d)


@pytest.mark.parametrize("kw,ptrs,want", [
    (dict(head_dim=32, C=64), {}, dpp.DPP_ERR_UNSUPPORTED),
    (dict(C=192), {}, dpp.DPP_ERR_INVALID_ARG),           # C != heads * 64
    (dict(H=9), {}, dpp.DPP_ERR_INVALID_ARG),
    ({}, dict(kv_prev=Ep + 256), dpp.DPP_ERR_ALIAS),      # stale overlaps next
    ({}, dict(ws=0), dpp.DPP_ERR_WORKSPACE),
    ({}, dict(wq=0), dpp.DPP_ERR_INVALID_ARG),
])
def test_self_attn_validation(kw, ptrs, want):
    d = attn(**kw)
    p = dict(x=A, wq=Cp, wk=Cp + 65536, wv=Cp + 2 * 65536, wo=Cp + 3 * 65536, kv_prev=None,
             kv_next=Ep, y=Dp, ws=Bp, ws_bytes=1 << 24)
    p.update(ptrs)
    st = dpp.dpp_self_attn(d, p["x"], p["wq"], p["wk"], p["wv"], p["wo"], p["kv_prev"],
                           p["kv_next"], p["y"], p["ws"], p["ws_bytes"], stream=0,
                           raise_on_error=False)
    assert st == want


def test_cross_attn_validation():
    d = attn(n_ctx=0, c_ctx=0)
    st = dpp.dpp_cross_attn(d, A, Bp, Cp, Cp, Cp, Cp, Dp, Ep, 1 << 24, stream=0,
                            raise_on_error=False)
    assert st == dpp.DPP_ERR_INVALID_ARG
    d = attn(n_ctx=77, c_ctx=2048)
    assert dpp.dpp_cross_attn_workspace_bytes(d) > 0
    st = dpp.dpp_cross_attn(d, A, Bp, Cp, Cp, Cp, Cp, Dp, Ep, 16, stream=0, raise_on_error=False)
    assert st == dpp.DPP_ERR_WORKSPACE


def test_cfg_validation():
    n = 1000
    ws = dpp.dpp_cfg_workspace_bytes(n)
    assert ws >= 16 + 3 * 8
    assert dpp.dpp_cfg_combine(A, Bp, 7.5, n, Cp + 4, None, None, 0, stream=0,
                               raise_on_error=False) == dpp.DPP_ERR_ALIGN
    assert dpp.dpp_cfg_combine(A, Bp, 7.5, n, Cp, Dp, None, 0, stream=0,
                               raise_on_error=False) == dpp.DPP_ERR_WORKSPACE
    assert dpp.dpp_cfg_combine(A, Bp, 7.5, n, A + 16, None, None, 0, stream=0,
                               raise_on_error=False) == dpp.DPP_ERR_ALIAS
    assert dpp.dpp_cfg_combine(0, Bp, 7.5, n, Cp, None, None, 0, stream=0,
                               raise_on_error=False) == dpp.DPP_ERR_INVALID_ARG


def test_refresh_validation():
    f = dpp.dpp_refresh_stale
    assert f(A, Bp, 1, 10, 64, 4, stream=0, raise_on_error=False) == dpp.DPP_ERR_INVALID_ARG
    assert f(A, Bp, 1, 8, 40, 4, stream=0, raise_on_error=False) == dpp.DPP_ERR_INVALID_ARG
    assert f(A, Bp, 1, 8, 64, 65, stream=0, raise_on_error=False) == dpp.DPP_ERR_INVALID_ARG
    assert f(A, A + 64, 1, 8, 64, 4, stream=0, raise_on_error=False) == dpp.DPP_ERR_ALIAS
    assert f(A + 8, Bp, 1, 8, 64, 4, stream=0, raise_on_error=False) == dpp.DPP_ERR_ALIGN
    # an empty mask is a valid no-op that launches nothing
    assert f(A, Bp, 1, 8, 64, 4, patch_mask=0, stream=0, raise_on_error=False) == dpp.DPP_OK


def test_refresh_halo_validation():
    f = dpp.dpp_refresh_halo
    assert f(A, Bp, 1, 10, 64, 4, stream=0, raise_on_error=False) == dpp.DPP_ERR_INVALID_ARG
    assert f(A, Bp, 1, 8, 40, 4, stream=0, raise_on_error=False) == dpp.DPP_ERR_INVALID_ARG
    assert f(A, A + 64, 1, 8, 64, 4, stream=0, raise_on_error=False) == dpp.DPP_ERR_ALIAS
    assert f(A + 8, Bp, 1, 8, 64, 4, stream=0, raise_on_error=False) == dpp.DPP_ERR_ALIGN
    assert f(A, Bp, 40000, 8, 64, 4, stream=0, raise_on_error=False) == dpp.DPP_ERR_UNSUPPORTED
    # one band has no halo: a valid no-op that launches nothing
    before = dpp.dpp_launch_count()
    assert f(A, Bp, 2, 8, 64, 1, stream=0, raise_on_error=False) == dpp.DPP_OK
    assert dpp.dpp_launch_count() == before


@pytest.mark.parametrize("kw,ptrs,want", [
    (dict(C=30), {}, dpp.DPP_ERR_INVALID_ARG),            # C % G
    (dict(G=2048, C=2048), {}, dpp.DPP_ERR_UNSUPPORTED),   # more than 1024 groups
    (dict(C=8192, G=32), {}, dpp.DPP_ERR_UNSUPPORTED),     # more than 512 vectors a pixel
    ({}, dict(x=0), dpp.DPP_ERR_INVALID_ARG),
    ({}, dict(sums=0), dpp.DPP_ERR_INVALID_ARG),
    ({}, dict(sums=Bp + 8), dpp.DPP_ERR_ALIGN),
    ({}, dict(sums=A + 64), dpp.DPP_ERR_ALIAS),            # sums inside x
])
def test_groupnorm_sums_validation(kw, ptrs, want):
    p = dict(x=A, sums=Bp)
    p.update(ptrs)
    assert dpp.dpp_groupnorm_sums(gn(**kw), p["x"], p["sums"], stream=0,
                                  raise_on_error=False) == want


@pytest.mark.parametrize("kw,ptrs,want", [
    (dict(H=7), {}, dpp.DPP_ERR_INVALID_ARG),             # H % P
    ({}, dict(sums=0), dpp.DPP_ERR_INVALID_ARG),
    ({}, dict(affine=0), dpp.DPP_ERR_INVALID_ARG),
    ({}, dict(gamma=Cp, beta=None), dpp.DPP_ERR_INVALID_ARG),
    ({}, dict(affine=Dp + 4), dpp.DPP_ERR_ALIGN),
    ({}, dict(affine=Bp + 64), dpp.DPP_ERR_ALIAS),         # affine over the sums
    ({}, dict(stats_prev=Ep + 16), dpp.DPP_ERR_ALIAS),     # prev overlaps next
])
def test_groupnorm_affine_validation(kw, ptrs, want):
    p = dict(sums=Bp, stats_prev=None, stats_next=Ep, gamma=Cp, beta=Cp + 4096, affine=Dp)
    p.update(ptrs)
    st = dpp.dpp_groupnorm_affine(gn(**kw), p["sums"], p["stats_prev"], p["stats_next"],
                                  p["gamma"], p["beta"], p["affine"], stream=0,
                                  raise_on_error=False)
    assert st == want


@pytest.mark.parametrize("kw,ptrs,want", [
    (dict(H=9), {}, dpp.DPP_ERR_INVALID_ARG),             # the conv's own checks first
    (dict(dtype=dpp.DPP_F32), {}, dpp.DPP_ERR_UNSUPPORTED),  # tensor-core conv only
    ({}, dict(affine=0), dpp.DPP_ERR_INVALID_ARG),
    ({}, dict(affine_prev=0), dpp.DPP_ERR_INVALID_ARG),     # stale halo needs the old affine
    ({}, dict(act=7), dpp.DPP_ERR_INVALID_ARG),
    ({}, dict(G=3, sums=Ep + 65536), dpp.DPP_ERR_INVALID_ARG),  # C_out % G
    ({}, dict(affine=Ep + 8), dpp.DPP_ERR_ALIGN),
    ({}, dict(affine=Dp + 256), dpp.DPP_ERR_ALIAS),         # output over the affine
    ({}, dict(sums=Dp + 512), dpp.DPP_ERR_ALIAS),           # sums inside the output
])
def test_conv_norm_validation(kw, ptrs, want):
    p = dict(x=A, stale=Bp, affine=Ep, affine_prev=Ep + 4096, act=dpp.DPP_ACT_SILU, w=Cp,
             y=Dp, G=4, sums=None)
    p.update(ptrs)
    st = dpp.dpp_conv3x3_norm(conv(**kw), p["x"], p["stale"], p["affine"], p["affine_prev"],
                              p["act"], p["w"], None, p["y"], p["G"], p["sums"], stream=0,
                              raise_on_error=False)
    assert st == want


def ln(**kw):
    d = dict(T=64, C=640, eps=1e-5, dtype=dpp.DPP_BF16)
    d.update(kw)
    return dpp.dpp_ln_desc(**d)


@pytest.mark.parametrize("kw,ptrs,want", [
    (dict(C=12), {}, dpp.DPP_ERR_INVALID_ARG),            # bf16 needs C % 8 == 0
    (dict(T=0), {}, dpp.DPP_ERR_INVALID_ARG),
    (dict(C=4096), {}, dpp.DPP_ERR_UNSUPPORTED),          # more than 256 vectors a token
    (dict(dtype=dpp.DPP_F32, C=2048), {}, dpp.DPP_ERR_UNSUPPORTED),
    (dict(eps=-1.0), {}, dpp.DPP_ERR_INVALID_ARG),
    ({}, dict(beta=None), dpp.DPP_ERR_INVALID_ARG),        # gamma without beta
    ({}, dict(x=A + 4), dpp.DPP_ERR_ALIGN),
    ({}, dict(y=A + 64), dpp.DPP_ERR_ALIAS),               # partial overlap (y == x is fine)
    ({}, dict(y=Cp + 16), dpp.DPP_ERR_ALIAS),              # output over gamma
])
def test_layernorm_validation(kw, ptrs, want):
    p = dict(x=A, gamma=Cp, beta=Dp, y=Bp)
    p.update(ptrs)
    before = dpp.dpp_launch_count()
    st = dpp.dpp_layernorm(ln(**kw), p["x"], p["gamma"], p["beta"], p["y"], stream=0,
                           raise_on_error=False)
    assert st == want and dpp.dpp_launch_count() == before


def lin(**kw):
    d = dict(M=256, K=640, N=640, dtype=dpp.DPP_BF16, epilogue=dpp.DPP_EPI_NONE, accumulate=0)
    d.update(kw)
    return dpp.dpp_linear_desc(**d)


@pytest.mark.parametrize("kw,ptrs,want", [
    (dict(dtype=dpp.DPP_F32), {}, dpp.DPP_ERR_UNSUPPORTED),
    (dict(N=32), {}, dpp.DPP_ERR_INVALID_ARG),             # N % 64
    (dict(K=12), {}, dpp.DPP_ERR_INVALID_ARG),             # K % 8
    (dict(M=0), {}, dpp.DPP_ERR_INVALID_ARG),
    (dict(epilogue=5), {}, dpp.DPP_ERR_INVALID_ARG),
    (dict(dtype=7), {}, dpp.DPP_ERR_INVALID_ARG),
    ({}, dict(x=0), dpp.DPP_ERR_INVALID_ARG),
    ({}, dict(w=Cp + 8), dpp.DPP_ERR_ALIGN),
    ({}, dict(y=A + 1024), dpp.DPP_ERR_ALIAS),             # output over x
    ({}, dict(y=Cp + 1024), dpp.DPP_ERR_ALIAS),            # output over w
    (dict(epilogue=dpp.DPP_EPI_GEGLU), dict(y=Cp + 640 * 640 * 2 + 64),
     dpp.DPP_ERR_ALIAS),                                   # output over the gate rows
])
def test_linear_validation(kw, ptrs, want):
    p = dict(x=A, w=Cp, bias=None, y=Bp)
    p.update(ptrs)
    before = dpp.dpp_launch_count()
    st = dpp.dpp_linear(lin(**kw), p["x"], p["w"], p["bias"], p["y"], stream=0,
                        raise_on_error=False)
    assert st == want and dpp.dpp_launch_count() == before


def test_error_raises_with_status_name():
    with pytest.raises(dpp.DppError, match="DPP_ERR_INVALID_ARG"):
        dpp.dpp_conv3x3(conv(H=9), A, Bp, Cp, None, Dp, stream=0)


def test_rejected_calls_launch_nothing():
    before = dpp.dpp_launch_count()
    dpp.dpp_conv3x3(conv(H=9), A, Bp, Cp, None, Dp, stream=0, raise_on_error=False)
    dpp.dpp_groupnorm(gn(C=30), A, None, Ep, None, None, Dp, Bp, 1 << 20, stream=0,
                      raise_on_error=False)
    dpp.dpp_self_attn(attn(H=9), A, Cp, Cp, Cp, Cp, None, Ep, Dp, Bp, 1 << 24, stream=0,
                      raise_on_error=False)
    dpp.dpp_refresh_stale(A, A + 64, 1, 8, 64, 4, stream=0, raise_on_error=False)
    assert dpp.dpp_launch_count() == before


def test_static_groupnorm_rejects_oversize_scratch_on_the_host():
    # 8192 one-channel groups in 64 bands of 2 images: 128 units x 8192
    # groups x 2 fp64 totals = 16 MiB of scratch
    big = gn(B=2, H=256, W=256, C=8192, G=8192, P=64)
    assert dpp.dpp_groupnorm_workspace_bytes(big) > dpp.DPP_GN_STATIC_SCRATCH_BYTES
    before = dpp.dpp_launch_count()
    st = dpp.dpp_groupnorm_static(big, A, None, Ep, None, None, Dp, stream=0,
                                  raise_on_error=False)
    assert st == dpp.DPP_ERR_WORKSPACE and dpp.dpp_launch_count() == before
    assert dpp.dpp_groupnorm_static(gn(C=30), A, None, Ep, None, None, Dp, stream=0,
                                    raise_on_error=False) == dpp.DPP_ERR_INVALID_ARG


def test_generic_workspace_query_matches_the_per_op_queries():
    g = gn()
    assert dpp.dpp_workspace_bytes(dpp.DPP_OP_GROUPNORM, g) == dpp.dpp_groupnorm_workspace_bytes(g)
    a = attn()
    assert dpp.dpp_workspace_bytes(dpp.DPP_OP_SELF_ATTN, a) == dpp.dpp_self_attn_workspace_bytes(a)
    x = attn(n_ctx=77, c_ctx=2048)
    assert dpp.dpp_workspace_bytes(dpp.DPP_OP_CROSS_ATTN, x) == \
        dpp.dpp_cross_attn_workspace_bytes(x)
    assert dpp.dpp_workspace_bytes(dpp.DPP_OP_CFG_COMBINE, 921600) == \
        dpp.dpp_cfg_workspace_bytes(921600) > 0
    assert dpp.dpp_workspace_bytes(dpp.DPP_OP_CONV3X3, conv()) == 0
    assert dpp.dpp_workspace_bytes(dpp.DPP_OP_REFRESH_STALE, conv()) == 0
    assert dpp.dpp_workspace_bytes(99, g) == 0
    assert dpp.dpp_workspace_bytes(dpp.DPP_OP_GROUPNORM, gn(C=30)) == 0


def test_block_chain_checks_weight_shapes_on_the_host():
    import torch
    from displaced_patch_parallelism_02_b300 import chain
    C, F, X = 64, 256, 32
    shapes = chain.weight_shapes(C, F, X)
    w = {k: torch.zeros(s, dtype=torch.float32 if len(s) == 1 else torch.bfloat16)
         for k, s in shapes.items()}
    assert chain.check_weights(w, C, F, X, torch.device("cpu")) is w
    bad = dict(w, ff1_w=torch.zeros((F, C), dtype=torch.bfloat16))  # gate rows missing
    with pytest.raises(ValueError, match="ff1_w"):
        chain.check_weights(bad, C, F, X, torch.device("cpu"))
    with pytest.raises(ValueError, match="missing"):
        chain.check_weights({k: v for k, v in w.items() if k != "wo"}, C, F, X,
                            torch.device("cpu"))
    bad = dict(w, conv1_w=torch.zeros((C, C, 3, 3), dtype=torch.bfloat16))  # not channels-last
    with pytest.raises(ValueError, match="conv1_w"):
        chain.check_weights(bad, C, F, X, torch.device("cpu"))


def test_wait_selftest_validation():
    before = dpp.dpp_launch_count()
    assert dpp.dpp_wait_selftest(2, A, stream=0, raise_on_error=False) == dpp.DPP_ERR_INVALID_ARG
    assert dpp.dpp_wait_selftest(0, None, stream=0, raise_on_error=False) == \
        dpp.DPP_ERR_INVALID_ARG
    assert dpp.dpp_wait_selftest(0, A + 4, stream=0, raise_on_error=False) == dpp.DPP_ERR_ALIGN
    assert dpp.dpp_launch_count() == before


def test_block_chain_step_checks_its_inputs_on_the_host():
    import torch
    from displaced_patch_parallelism_02_b300 import chain
    C, F, X = 64, 256, 32
    w = {k: torch.zeros(s, dtype=torch.float32 if len(s) == 1 else torch.bfloat16)
         for k, s in chain.weight_shapes(C, F, X).items()}
    bc = chain.BlockChain(1, 8, 8, C, 1, 2, 8, 5, X, w, "cpu")
    x = torch.zeros(1, 8, 8, C, dtype=torch.bfloat16)
    ctx = torch.zeros(1, 5, X, dtype=torch.bfloat16)
    n0 = dpp.dpp_launch_count()
    with pytest.raises(ValueError, match="x:"):
        bc.step(torch.zeros(1, 8, 4, C, dtype=torch.bfloat16), ctx)
    with pytest.raises(ValueError, match="x:"):
        bc.step(x.float(), ctx)
    with pytest.raises(ValueError, match="ctx:"):
        bc.step(x, torch.zeros(1, 5, 16, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="x:"):
        bc.step(torch.zeros(1, 8, 8, 2 * C, dtype=torch.bfloat16)[..., :C], ctx)  # strided
    assert dpp.dpp_launch_count() == n0 and bc.k == 0


def test_opbench_parses_its_options_and_needs_a_device():
    import torch
    from displaced_patch_parallelism_02_b300 import opbench
    with pytest.raises(SystemExit) as e:
        opbench.main(["--help"])
    assert e.value.code == 0
    with pytest.raises(SystemExit):
        opbench.main(["no_such_op"])
    if not torch.cuda.is_available():
        with pytest.raises(AssertionError, match="CUDA device"):
            opbench.main(["linear", "--M", "128"])


def test_library_is_built_from_these_sources():
    """The library carries the SHA-256 of the sources and flags it was built
    from; build() rebuilds it when that differs from the files here, so a
    prebuilt library cannot stand in for edited sources."""
    import importlib.util
    path = os.path.join(ROOT, "displaced_patch_parallelism_02_b300", "build.py")
    spec = importlib.util.spec_from_file_location("_dpp_build_check", path)
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    assert dpp.dpp_source_hash() == b.source_hash()
    assert b.library_hash() == b.source_hash()
    assert b.library_hash(os.path.join(ROOT, "no_such_library.so")) is None


def test_cached_cross_attention_arguments_checked_on_the_host():
    d = dpp.dpp_attn_desc(1, 4, 4, 64, 1, 64, 1, 77, 96, dpp.DPP_BF16, 0, 0)
    before = dpp.dpp_launch_count()
    st = dpp.dpp_cross_attn_kv(d, A, Bp, Cp, None, stream=0, raise_on_error=False)
    assert st == dpp.DPP_ERR_INVALID_ARG
    st = dpp.dpp_cross_attn_kv(d, A + 8, Bp, Cp, Dp, stream=0, raise_on_error=False)
    assert st == dpp.DPP_ERR_ALIGN
    n = dpp.dpp_cross_attn_cached_workspace_bytes(d)
    assert n > 0
    st = dpp.dpp_cross_attn_cached(d, A, Bp, Cp, Dp, Ep, None, 0, stream=0, raise_on_error=False)
    assert st == dpp.DPP_ERR_WORKSPACE
    assert dpp.dpp_launch_count() == before
