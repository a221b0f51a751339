"""dpp_groupnorm_static: GroupNorm for callers that cannot allocate device memory.

Such callers (plugins inside a host program that owns the device-memory
budget, or hot paths that must not call cudaMalloc because it may synchronise
the device) get the partial-sum scratch from a static device array in the
library.  This checks, through the C ABI, that two calls in a row -- the
synchronous step and a displaced step fed by the first call's published
partials -- match the workspace entry point dpp_groupnorm within the bf16 /
fp32 tolerances of the other parity tests.  It lives in a file of its own,
collected last, and passes alone in a fresh process as well as after the
other tests.
"""
import numpy as np
import pytest
import torch

import displaced_patch_parallelism_02_b300 as dpp
import workloads as wl
from tests import gpu_ops as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,W,C,Gn,P,dt", [
    (2, 480, 480, 320, 32, 8, torch.bfloat16),   # the 3840px latent
    (2, 12, 7, 40, 8, 3, torch.bfloat16),        # ragged chunks, groups straddling vectors
    (1, 32, 32, 64, 32, 2, torch.float32),
])
def test_static_scratch_groupnorm_matches_workspace_entry_point(cuda_device, B, H, W, C, Gn, P,
                                                                dt):
    name = "bf16" if dt == torch.bfloat16 else "f32"
    S = wl.normal((B, H, W, C), 900, dtype=name).cuda()
    F = wl.perturbed(wl.normal((B, H, W, C), 900, dtype=name), 901, 0.05).cuda()
    gamma, beta = (t.cuda() for t in wl.gn_affine(C, 9))
    d = G.gn_desc(F, Gn, 1e-5, P)
    assert dpp.dpp_groupnorm_workspace_bytes(d) <= dpp.DPP_GN_STATIC_SCRATCH_BYTES
    stats = lambda: torch.empty((P, B, Gn, 2), dtype=torch.float32, device="cuda")

    # reference: the entry point with a caller workspace
    y_ref0, st_ref0 = G.groupnorm(S, None, Gn, 1e-5, gamma, beta, P)
    y_ref1, st_ref1 = G.groupnorm(F, st_ref0, Gn, 1e-5, gamma, beta, P)

    # two calls in a row on the static scratch: synchronous, then displaced
    y0, st0 = torch.empty_like(S), stats()
    dpp.dpp_groupnorm_static(d, S, None, st0, gamma, beta, y0)
    y1, st1 = torch.empty_like(F), stats()
    dpp.dpp_groupnorm_static(d, F, st0, st1, gamma, beta, y1)
    torch.cuda.synchronize()

    tol = G.TOL[dt]
    G.assert_rms_close(G.f64(y0), G.f64(y_ref0), tol, "static groupnorm, call 1")
    G.assert_rms_close(G.f64(y1), G.f64(y_ref1), tol, "static groupnorm, call 2")
    np.testing.assert_allclose(st1.cpu().numpy(), st_ref1.cpu().numpy(), rtol=1e-6, atol=1e-3)
    assert dpp.dpp_device_status() == dpp.DPP_OK
