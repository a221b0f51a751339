"""Adaptive parallelism switching (Hydiff summaries, gist.science section
自适应并行切换; Avetisyan, Адаптивное переключение): the library's host-side
controller (dpp_switch_init / dpp_switch_update) against the oracle's
switch_stages, stage for stage.

The controller is host logic, so its parity runs without a GPU.  The one GPU
test drives it the way a sampler does: each step's discrepancy comes from the
sums dpp_cfg_combine writes, while the oracle reads the same maps in fp64.
Both sides take the threshold decisions in fp64.
"""
import math

import numpy as np
import pytest
import torch

import displaced_patch_parallelism_02_b300 as dpp
import oracle
import workloads as wl


def run_controller(ds, flat_tol, rise_tol, patience):
    s = dpp.dpp_switch_state()
    dpp.dpp_switch_init(s, flat_tol, rise_tol, patience)
    return [dpp.dpp_switch_update(s, d) for d in ds]


def u_curve(rng, n, noise):
    # decline, a flat valley, a late rise: the shape the pages describe
    t = np.linspace(0.0, 1.0, n)
    base = 0.05 + 0.6 * np.exp(-8.0 * t) + 0.4 * np.clip(t - 0.7, 0.0, None) ** 2
    return list(np.abs(base * (1.0 + noise * rng.standard_normal(n))))


@pytest.mark.parametrize("patience", [1, 2, 3, 4])
@pytest.mark.parametrize("noise", [0.0, 0.01, 0.05])
def test_controller_matches_oracle_on_u_curves(patience, noise):
    rng = np.random.default_rng(100 * patience + int(noise * 1000))
    for trial in range(40):
        d = u_curve(rng, int(rng.integers(1, 80)), noise)
        ft, rt = float(rng.uniform(0.005, 0.1)), float(rng.uniform(0.0, 0.2))
        assert run_controller(d, ft, rt, patience) == oracle.switch_stages(d, ft, rt, patience)


def test_controller_matches_oracle_on_random_walks_with_bad_entries():
    rng = np.random.default_rng(9)
    for trial in range(300):
        n = int(rng.integers(0, 50))
        d = list(np.abs(1.0 + np.cumsum(0.05 * rng.standard_normal(n))))
        for _ in range(int(rng.integers(0, 4))):
            if n:
                d[int(rng.integers(0, n))] = [float("nan"), -0.5, 0.0, math.inf][
                    int(rng.integers(0, 4))]
        p = int(rng.integers(1, 5))
        ft, rt = float(rng.uniform(0.0, 0.1)), float(rng.uniform(0.0, 0.1))
        assert run_controller(d, ft, rt, p) == oracle.switch_stages(d, ft, rt, p)


def test_controller_worked_example_and_state():
    from tests.test_oracle_pins import SWITCH_SERIES, SWITCH_STAGES
    s = dpp.dpp_switch_state()
    dpp.dpp_switch_init(s, 0.05, 0.10, 2)
    got = [dpp.dpp_switch_update(s, d) for d in SWITCH_SERIES]
    assert got == SWITCH_STAGES
    assert s.stage == dpp.DPP_STAGE_FULLY_CONNECTING and s.steps == len(SWITCH_SERIES)
    dpp.dpp_switch_init(s, 0.05, 0.10, 0)  # patience below 1 reads as 1
    assert s.patience == 1 and s.stage == dpp.DPP_STAGE_WARMUP and s.steps == 0


@pytest.mark.gpu
def test_controller_driven_by_cfg_sums(cuda_device):
    # eps_c = eps_u + a_t * z: the rel-MAE of step t is a_t * E|z| / E|eps_u|
    n = 4 * 96 * 96
    u = wl.normal((n,), 501, dtype="f32")
    z = wl.normal((n,), 502, dtype="f32")
    a = [0.9 * 0.5 ** t + 0.08 for t in range(10)] + [0.08] * 6 + \
        [0.08 * 1.15 ** k for k in range(1, 10)]
    sums = torch.zeros(3, dtype=torch.float64, device="cuda")
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    nws = dpp.dpp_cfg_workspace_bytes(n)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    ud = u.cuda()
    s = dpp.dpp_switch_state()
    dpp.dpp_switch_init(s, 0.03, 0.05, 2)
    got, ref_d = [], []
    for at in a:
        c = (u.double() + at * z.double()).float()
        dpp.dpp_cfg_combine(ud, c.cuda(), 7.5, n, out, sums, ws, nws)
        h = sums.cpu().numpy()
        got.append(dpp.dpp_switch_update(s, float(h[0] / h[1])))
        _, ref_sums = oracle.cfg_combine(u.double().numpy(), c.double().numpy(), 7.5)
        ref_d.append(oracle.rel_mae(ref_sums))
    want = oracle.switch_stages(ref_d, 0.03, 0.05, 2)
    assert got == want
    assert want[0] == 0 and 1 in want and want[-1] == 2
