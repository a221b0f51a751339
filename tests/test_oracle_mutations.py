"""Planted mistakes in the oracle must each fail at least one pin.

Each mutation below is a plausible slip (a transposed tap, the wrong halo
source, a biased/unbiased variance mix-up, a missing softmax scale, a swapped
guidance operand, an off-by-one band ...).  It is monkeypatched into the
oracle on the CPU and the pins of test_oracle_pins are re-run against it.
"""
import numpy as np
import pytest

import oracle
import oracle.blocks as ob
import oracle.displaced as od
import tests.test_oracle_pins as pins


def _conv_row_transposed(rows_in, Wt, W):
    return _orig_conv_row(rows_in, np.swapaxes(Wt, 2, 3), W)


_orig_conv_row = od._conv_row


def _displaced_conv_fresh_halo(F, S, Wt, bias, P, out_rows=None, first_layer=False):
    return _orig_displaced_conv(F, S, Wt, bias, P, out_rows, True)


_orig_displaced_conv = od.displaced_conv3x3


def _displaced_conv_neighbours_stale(F, S, Wt, bias, P, out_rows=None, first_layer=False):
    B, H, W, _ = F.shape
    rows = range(H) if out_rows is None else list(out_rows)
    out = np.zeros((B, len(rows), W, Wt.shape[0]))
    for k, h in enumerate(rows):
        src = [None if not 0 <= r < H else (F[:, r] if r == h else S[:, r])
               for r in (h - 1, h, h + 1)]
        out[:, k] = od._conv_row(src, Wt, W) + (0 if bias is None else bias)
    return out


def _groupnorm_unbiased(X, G, eps, gamma=None, beta=None):
    B, H, W, C = X.shape
    Xg = X.reshape(B, H * W, G, C // G)
    mean = Xg.mean(axis=(1, 3), keepdims=True)
    n = H * W * C // G
    var = ((Xg - mean) ** 2).sum(axis=(1, 3), keepdims=True) / (n - 1)
    Y = ((Xg - mean) / np.sqrt(var + eps)).reshape(B, H, W, C)
    return Y * gamma + beta if gamma is not None else Y


def _groupnorm_eps_outside(X, G, eps, gamma=None, beta=None):
    B, H, W, C = X.shape
    Xg = X.reshape(B, H * W, G, C // G)
    mean = Xg.mean(axis=(1, 3), keepdims=True)
    var = ((Xg - mean) ** 2).mean(axis=(1, 3), keepdims=True)
    Y = ((Xg - mean) / (np.sqrt(var) + eps)).reshape(B, H, W, C)
    return Y * gamma + beta if gamma is not None else Y


def _groupnorm_channel_groups_strided(X, G, eps, gamma=None, beta=None):
    # groups taken as channels c % G instead of consecutive blocks
    B, H, W, C = X.shape
    Xg = X.reshape(B, H * W, C // G, G)
    mean = Xg.mean(axis=(1, 2), keepdims=True)
    var = ((Xg - mean) ** 2).mean(axis=(1, 2), keepdims=True)
    Y = ((Xg - mean) / np.sqrt(var + eps)).reshape(B, H, W, C)
    return Y * gamma + beta if gamma is not None else Y


def _composite_swapped(F, S, P, p, axis=1):
    return _orig_composite(S, F, P, p, axis)


_orig_composite = od.composite


def _attention_unscaled(Q, K, V, heads):
    return _orig_attention(Q * np.sqrt(Q.shape[1] // heads), K, V, heads)


_orig_attention = od.attention_heads


def _partials_all_rows(X, G, P):
    B, H, W, C = X.shape
    out = np.zeros((P, B, G, 2))
    Xg = X.reshape(B, H * W, G, C // G)
    out[:, :, :, 0] = Xg.sum(axis=(1, 3)) / P
    out[:, :, :, 1] = (Xg ** 2).sum(axis=(1, 3)) / P
    return out


def _cfg_wrong_base(eps_u, eps_c, scale):
    out, sums = _orig_cfg(eps_u, eps_c, scale)
    return np.asarray(eps_c) + scale * (np.asarray(eps_c) - np.asarray(eps_u)), sums


_orig_cfg = od.cfg_combine


def _rel_mae_by_cond(sums):
    return float(sums[0] / sums[2])


def _refresh_off_by_one(fresh, stale, P, patch_mask=None, axis=1):
    out = np.array(stale, copy=True)
    n = fresh.shape[axis]
    for p in range(P):
        if patch_mask is not None and not (patch_mask >> p) & 1:
            continue
        lo, hi = od.patch_rows(n, P, p)
        idx = [slice(None)] * fresh.ndim
        idx[axis] = slice(lo, min(hi + 1, n))
        out[tuple(idx)] = fresh[tuple(idx)]
    return out


def _naive_conv_reads_neighbours(F, Wt, bias, P, out_rows=None):
    return od.conv3x3(F, Wt, bias, out_rows)


def _naive_gn_image_statistics(F, G, eps, gamma, beta, P):
    return od.groupnorm(F, G, eps, gamma, beta)


def _naive_attention_all_keys(F, Wq, Wk, Wv, Wo, heads, P):
    return od.displaced_self_attention(F, F, Wq, Wk, Wv, Wo, heads, P)


def _switch_variant(absolute_drop=False, rise_vs_previous=False, short_window=False):
    def stages(ds, flat_tol, rise_tol, patience):
        patience = max(1, int(patience))
        v = [float(x) for x in ds if x >= 0.0]
        w = patience - 1 if short_window and patience > 1 else patience

        def drop(j):
            if absolute_drop:
                return v[j - 1] - v[j]
            return (v[j - 1] - v[j]) / v[j - 1] if v[j - 1] > 0.0 else 0.0

        def ref(j, tau1):
            return v[j - 1] if rise_vs_previous else min(v[tau1:j + 1])

        tau1 = next((t for t in range(w, len(v))
                     if all(drop(j) < flat_tol for j in range(t - w + 1, t + 1))), None)
        tau2 = None
        if tau1 is not None:
            tau2 = next((t for t in range(tau1 + w, len(v))
                         if all(v[j] > ref(j, tau1) * (1.0 + rise_tol)
                                for j in range(t - w + 1, t + 1))), None)
        out = [2 if tau2 is not None and t >= tau2 else 1 if tau1 is not None and t >= tau1
               else 0 for t in range(len(v))]
        res, k, last = [], 0, 0
        for x in ds:
            if x >= 0.0:
                last = out[k]
                k += 1
            res.append(last)
        return res
    return stages


def _geglu_gate_first(X, W1, b1):
    Hd = ob.linear(X, W1, b1)
    n = Hd.shape[-1] // 2
    return ob.gelu(Hd[..., :n]) * Hd[..., n:]


def _resnet_no_silu_after_gn2(x, states, prm, P, G, eps):
    st = states or {}
    g1 = ob.silu(od.displaced_groupnorm(x, st.get("gn1", x), G, eps, prm["gn1_g"],
                                        prm["gn1_b"], P))
    h = od.displaced_conv3x3(g1, st.get("conv1", g1), prm["conv1_w"], prm["conv1_b"], P)
    g2 = od.displaced_groupnorm(h, st.get("gn2", h), G, eps, prm["gn2_g"], prm["gn2_b"], P)
    y = od.displaced_conv3x3(g2, st.get("conv2", g2), prm["conv2_w"], prm["conv2_b"], P)
    return x + y, {"gn1": x, "conv1": g1, "gn2": h, "conv2": g2}


def _resnet_states_swapped(x, states, prm, P, G, eps):
    out, st = _orig_resnet(x, states, prm, P, G, eps)
    st = dict(st)
    st["conv1"], st["conv2"] = st["conv2"], st["conv1"]
    return out, st


_orig_resnet = ob.resnet_block


MUTATIONS = {
    "conv_taps_transposed": [("_conv_row", _conv_row_transposed)],
    "conv_halo_fresh": [("displaced_conv3x3", _displaced_conv_fresh_halo)],
    "conv_own_neighbours_stale": [("displaced_conv3x3", _displaced_conv_neighbours_stale)],
    "gn_unbiased_variance": [("groupnorm", _groupnorm_unbiased)],
    "gn_eps_outside_sqrt": [("groupnorm", _groupnorm_eps_outside)],
    "gn_strided_groups": [("groupnorm", _groupnorm_channel_groups_strided)],
    "gn_partials_all_rows": [("groupnorm_partials", _partials_all_rows)],
    "composite_swapped": [("composite", _composite_swapped)],
    "attention_unscaled": [("attention_heads", _attention_unscaled)],
    "cfg_wrong_base": [("cfg_combine", _cfg_wrong_base)],
    "rel_mae_by_cond": [("rel_mae", _rel_mae_by_cond)],
    "refresh_off_by_one": [("refresh_stale", _refresh_off_by_one)],
    "naive_conv_reads_neighbours": [("naive_conv3x3", _naive_conv_reads_neighbours)],
    "naive_gn_image_statistics": [("naive_groupnorm", _naive_gn_image_statistics)],
    "naive_attention_all_keys": [("naive_self_attention", _naive_attention_all_keys)],
    "switch_absolute_drop": [("switch_stages", _switch_variant(absolute_drop=True))],
    "switch_rise_vs_previous": [("switch_stages", _switch_variant(rise_vs_previous=True))],
    "switch_short_window": [("switch_stages", _switch_variant(short_window=True))],
    "geglu_gate_first": [("blocks.geglu", _geglu_gate_first)],
    "resnet_no_silu_after_gn2": [("blocks.resnet_block", _resnet_no_silu_after_gn2)],
    "resnet_states_swapped": [("blocks.resnet_block", _resnet_states_swapped)],
}


def _all_pins():
    calls = []
    for name in dir(pins):
        fn = getattr(pins, name)
        if not name.startswith("test_") or not callable(fn):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if not params:
            calls.append((name, fn, {}))
            continue
        argnames = [a.strip() for a in params[0].args[0].split(",")]
        for vals in params[0].args[1]:
            vals = vals if isinstance(vals, tuple) else (vals,)
            calls.append((name, fn, dict(zip(argnames, vals))))
    return calls


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(mutation, monkeypatch):
    for attr, repl in MUTATIONS[mutation]:
        if attr.startswith("blocks."):
            monkeypatch.setattr(ob, attr.split(".", 1)[1], repl)
            continue
        monkeypatch.setattr(od, attr, repl)
        if hasattr(oracle, attr):
            monkeypatch.setattr(oracle, attr, repl)
    failed = []
    for name, fn, kw in _all_pins():
        try:
            fn(**kw)
        except (AssertionError, ValueError, IndexError):
            failed.append(name)
    assert failed, f"no pin caught the planted mistake {mutation}"
