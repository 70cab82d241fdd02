"""Pins of the float64 oracle to facts other than itself.

* central finite differences of the oracle's own forward, every input element
  perturbed, under an objective that includes the final-state region (the
  SSM_SCAN_BACK page, "The oracle is a float64 finite difference");
* the five planted defects of that page's verification table must each fail
  the same check by a wide margin, and the check must count what it compared;
* the chunkwise (K1..K5) form of the combined_backward.rs page must equal the
  serial recurrence to rounding;
* closed forms: A = 0 (a prefix sum), dy = 0 (pure decay of the seed), the
  unrolled sum for the forward, and a two-step case worked by hand;
* Euler identities (homogeneity) and chaining two calls through s0 / ds_final;
* cross-variant reductions (MIMO with R = 1 is Mamba-2; Mamba-2 with P = 1 and
  a decay constant over the state is Mamba-1).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import chunkwise
from selective_state_space_ssd_gb300 import inputs as synth
from selective_state_space_ssd_gb300.configs import CONFIGS, scaled

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

TINY = CONFIGS["mamba2_tiny_fp32"]
M1_TINY = dict(variant="mamba1", dtype="f32", batch=2, seqlen=24, nheads=3, headdim=1, dstate=4, ngroups=1,
               chunk=8, mimo_rank=1)
MIMO_TINY = dict(variant="mimo", dtype="f32", batch=1, seqlen=16, nheads=2, headdim=3, dstate=4, ngroups=2,
                 chunk=4, mimo_rank=2)
M2_GROUPS = dict(variant="mamba2", dtype="f32", batch=2, seqlen=32, nheads=4, headdim=3, dstate=5, ngroups=2,
                 chunk=8, mimo_rank=1)


def f64(cfg, seed=0):
    return synth.as_float64(synth.make_inputs(cfg, seed=seed))


def rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ----------------------------------------------------------- finite differences
def _objective(variant, inp):
    out = oracle.forward(variant, inp, nthreads=1)
    return float(np.sum(inp["dy"] * out["y"]) + np.sum(inp["ds_final"] * out["s_final"]))


def _fd_check(variant, inp, mutation=0):
    """Return (worst relative error over the gradients, elements perturbed)."""
    grads = oracle.backward(variant, inp, nthreads=1, mutation=mutation)
    names = {"x": "dx", "dt_raw": "ddt_raw", "A": "dA", "B": "dB", "C": "dC", "s0": "ds0"}
    worst, count = 0.0, 0
    for src, gname in names.items():
        if inp.get(src) is None or gname not in grads:
            continue
        theta = inp[src]
        fd = np.empty_like(theta)
        flat = theta.reshape(-1)
        for i in range(flat.size):
            h = 1e-6 * max(1.0, abs(flat[i]))
            plus = dict(inp)
            minus = dict(inp)
            tp, tm = theta.copy(), theta.copy()
            tp.reshape(-1)[i] += h
            tm.reshape(-1)[i] -= h
            plus[src], minus[src] = tp, tm
            fd.reshape(-1)[i] = (_objective(variant, plus) - _objective(variant, minus)) / (2 * h)
            count += 1
        worst = max(worst, rel(grads[gname], fd))
    return worst, count


FD_PASS = 1e-6


@pytest.mark.parametrize("variant,cfg", [("mamba2", TINY), ("mamba1", M1_TINY), ("mimo", MIMO_TINY),
                                         ("mamba2", M2_GROUPS)])
def test_backward_matches_finite_differences(variant, cfg):
    inp = f64(cfg)
    worst, count = _fd_check(variant, inp)
    sizes = sum(inp[k].size for k in ("x", "dt_raw", "A", "B", "C", "s0") if inp.get(k) is not None)
    assert count == sizes and count > 0  # every element was perturbed
    assert worst < FD_PASS, worst


@pytest.mark.parametrize("mutation", [1, 2, 3, 4, 5])
def test_planted_defects_are_caught(mutation):
    inp = f64(TINY)
    worst, count = _fd_check("mamba2", inp, mutation=mutation)
    assert count == 1730  # x 1024 + dt_raw 128 + A 2 + B 256 + C 256 + s0 64
    assert worst > 100 * FD_PASS, (mutation, worst)


@pytest.mark.parametrize("mutation", [1, 2, 3, 4])
def test_planted_defects_are_caught_mimo(mutation):
    inp = f64(MIMO_TINY)
    worst, _ = _fd_check("mimo", inp, mutation=mutation)
    assert worst > 100 * FD_PASS, (mutation, worst)


@pytest.mark.parametrize("mutation", [1, 2, 3, 4, 5])
def test_planted_defects_are_caught_mamba1(mutation):
    inp = f64(M1_TINY)
    worst, _ = _fd_check("mamba1", inp, mutation=mutation)
    assert worst > 100 * FD_PASS, (mutation, worst)


# --------------------------------------------------------------- chunkwise form
@pytest.mark.parametrize("cfg", [TINY, M2_GROUPS, scaled(TINY, batch=2, seqlen=96, nheads=3, headdim=5,
                                                            dstate=7, chunk=32),
                                 # a tail chunk: T not a multiple of the chunk length, and T below it
                                 scaled(M2_GROUPS, seqlen=37), scaled(TINY, seqlen=13)])
def test_serial_equals_chunkwise_mamba2(cfg):
    inp = f64(cfg)
    L = cfg["chunk"]
    fs = oracle.forward("mamba2", inp)
    fc = chunkwise.mamba2_forward(inp["x"], inp["dt_raw"], inp["A"], inp["B"], inp["C"], inp["s0"], L)
    for k in ("y", "s_final"):
        assert rel(fc[k], fs[k]) < 1e-12, k
    bs = oracle.backward("mamba2", inp)
    bc = chunkwise.mamba2_backward(inp["dy"], inp["ds_final"], inp["x"], inp["dt_raw"], inp["A"], inp["B"],
                                   inp["C"], inp["s0"], L)
    for k in ("dx", "ddt_raw", "dA", "dB", "dC", "ds0"):
        assert rel(bc[k], bs[k]) < 1e-11, k


@pytest.mark.parametrize("cfg", [MIMO_TINY, scaled(MIMO_TINY, batch=2, seqlen=48, mimo_rank=3, chunk=16),
                                 scaled(MIMO_TINY, batch=2, seqlen=19, mimo_rank=3, chunk=8)])
def test_serial_equals_chunkwise_mimo(cfg):
    inp = f64(cfg)
    L = cfg["chunk"]
    fs = oracle.forward("mimo", inp)
    fc = chunkwise.mimo_forward(inp["x"], inp["dt_raw"], inp["B"], inp["C"], inp["s0"], L)
    for k in ("y", "s_final"):
        assert rel(fc[k], fs[k]) < 1e-12, k
    bs = oracle.mimo_backward(inp["dy"], inp["ds_final"], inp["x"], inp["dt_raw"], inp["B"], inp["C"], inp["s0"])
    bc = chunkwise.mimo_backward(inp["dy"], inp["ds_final"], inp["x"], inp["dt_raw"], inp["B"], inp["C"],
                                 inp["s0"], L)
    for k in ("dv", "dda", "dB", "dC", "ds0"):
        assert rel(bc[k], bs[k]) < 1e-11, k


# ------------------------------------------------------------------ closed forms
def _softplus(z):
    return np.log1p(np.exp(z))  # no overflow at the generator's range


def test_closed_form_A_zero_is_prefix_sum():
    inp = f64(TINY)
    inp["A"] = np.zeros_like(inp["A"])
    x, B, C, s0, dy, dsf = inp["x"], inp["B"], inp["C"], inp["s0"], inp["dy"], inp["ds_final"]
    d = _softplus(inp["dt_raw"])                                    # [b,T,H]
    # s_t = s0 + sum_{tau<=t} d_tau x_tau (outer) B_tau
    incr = np.einsum("bth,bthp,btn->bthpn", d, x, B[:, :, 0])
    S = s0[:, None] + np.cumsum(incr, axis=1)                      # [b,T,H,P,N]
    y = np.einsum("bthpn,btn->bthp", S, C[:, :, 0])
    f = oracle.forward("mamba2", inp)
    assert rel(f["y"], y) < 1e-13
    assert rel(f["s_final"], S[:, -1]) < 1e-13
    # dS_t = ds_final + sum_{tau>=t} dy_tau (outer) C_tau (no decay)
    outer = np.einsum("bthp,btn->bthpn", dy, C[:, :, 0])
    dS = dsf[:, None] + np.cumsum(outer[:, ::-1], axis=1)[:, ::-1]
    S_prev = np.concatenate([s0[:, None], S[:, :-1]], axis=1)
    g = oracle.backward("mamba2", inp)
    assert rel(g["ds0"], dS[:, 0]) < 1e-13
    assert rel(g["dA"], np.einsum("bth,bthpn,bthpn->h", d, dS, S_prev)) < 1e-12
    assert rel(g["dx"], d[..., None] * np.einsum("bthpn,btn->bthp", dS, B[:, :, 0])) < 1e-13


def test_mamba1_closed_form_A_zero():
    """Mamba-1 at A = 0 (every decay 1): s_t = s0 + sum_{tau<=t} dt' x (x) B per channel, and the backward is made
    of running sums: dS_t = ds_final + sum_{tau>=t} dy C; dx = dt' <dS_t, B_t>, dB_t = sum_d dS_t dt' x,
    dC_t = sum_d s_t dy, ds0 = dS_0, dA[d,n] = sum_t dt' dS_t s_{t-1}, ddt_raw = sigmoid(z) x <dS_t, B_t>."""
    cfg = scaled(M1_TINY, batch=2, seqlen=11, nheads=3, dstate=4)
    inp = f64(cfg)
    inp["A"] = np.zeros_like(inp["A"])
    x, B, C, s0, dy, dsf = inp["x"], inp["B"], inp["C"], inp["s0"], inp["dy"], inp["ds_final"]
    z = inp["dt_raw"]
    d = _softplus(z)                                                  # [b,T,D]
    S = s0[:, None] + np.cumsum(np.einsum("btd,btn->btdn", d * x, B), axis=1)   # [b,T,D,N]
    f = oracle.forward("mamba1", inp)
    assert rel(f["y"], np.einsum("btdn,btn->btd", S, C)) < 1e-13
    assert rel(f["s_final"], S[:, -1]) < 1e-13
    dS = dsf[:, None] + np.cumsum(np.einsum("btd,btn->btdn", dy, C)[:, ::-1], axis=1)[:, ::-1]
    S_prev = np.concatenate([s0[:, None], S[:, :-1]], axis=1)
    g = oracle.backward("mamba1", inp)
    dSB = np.einsum("btdn,btn->btd", dS, B)
    assert rel(g["dx"], d * dSB) < 1e-13
    assert rel(g["dB"], np.einsum("btdn,btd->btn", dS, d * x)) < 1e-13
    assert rel(g["dC"], np.einsum("btdn,btd->btn", S, dy)) < 1e-13
    assert rel(g["ds0"], dS[:, 0]) < 1e-13
    assert rel(g["dA"], np.einsum("btd,btdn,btdn->dn", d, dS, S_prev)) < 1e-12
    assert rel(g["ddt_raw"], x * dSB / (1.0 + np.exp(-z))) < 1e-12


def test_closed_form_dy_zero_is_pure_decay():
    inp = f64(TINY)
    inp["dy"] = np.zeros_like(inp["dy"])
    g = oracle.backward("mamba2", inp)
    total = np.sum(_softplus(inp["dt_raw"]) * inp["A"][None, None, :], axis=1)  # [b,H]
    assert rel(g["ds0"], np.exp(total)[:, :, None, None] * inp["ds_final"]) < 1e-13
    assert np.all(g["dC"] == 0.0)  # dC_t = dy_t . s_t only
    assert np.max(np.abs(g["dx"])) > 0.0  # the seed still reaches x through dS


def test_forward_equals_unrolled_sum():
    """y_t = C_t . [exp(sum_{k<=t} da_k) s0 + sum_{tau<=t} exp(sum_{tau<k<=t} da_k) d_tau x_tau B_tau]."""
    cfg = scaled(TINY, seqlen=12, headdim=3, dstate=2)
    inp = f64(cfg)
    x, B, C, s0 = inp["x"], inp["B"], inp["C"], inp["s0"]
    d = _softplus(inp["dt_raw"])
    da = d * inp["A"][None, None, :]
    b, T, H, P = x.shape
    y = np.zeros_like(x)
    for bb in range(b):
        for h in range(H):
            for t in range(T):
                st = math.exp(sum(da[bb, k, h] for k in range(t + 1))) * s0[bb, h]
                for tau in range(t + 1):
                    w = math.exp(sum(da[bb, k, h] for k in range(tau + 1, t + 1))) * d[bb, tau, h]
                    st = st + w * np.outer(x[bb, tau, h], B[bb, tau, 0])
                y[bb, t, h] = st @ C[bb, t, 0]
    assert rel(oracle.forward("mamba2", inp)["y"], y) < 1e-13


def test_mamba1_forward_equals_unrolled_sum():
    """Mamba-1, one decay per state: y_t[d] = sum_n C_t[n] [exp(sum_{k<=t} dt'_k A[d,n]) s0[d,n]
    + sum_{tau<=t} exp(sum_{tau<k<=t} dt'_k A[d,n]) dt'_tau x_tau[d] B_tau[n]], written out with no recurrence;
    the states' decays differ, so a decay shared across n (or taken from the wrong index) fails it."""
    cfg = scaled(M1_TINY, batch=1, seqlen=9, nheads=3, dstate=3)
    inp = f64(cfg)
    x, B, C, s0, A = inp["x"], inp["B"], inp["C"], inp["s0"], inp["A"]
    d = _softplus(inp["dt_raw"])                                      # [b,T,D]
    b, T, D = x.shape
    N = A.shape[1]
    assert np.ptp(A, axis=1).min() > 0                                # distinct decays per state
    y = np.zeros_like(x)
    sf = np.zeros((b, D, N))
    for bb in range(b):
        for dd in range(D):
            for t in range(T):
                for n in range(N):
                    st = math.exp(sum(d[bb, k, dd] * A[dd, n] for k in range(t + 1))) * s0[bb, dd, n]
                    for tau in range(t + 1):
                        w = math.exp(sum(d[bb, k, dd] * A[dd, n] for k in range(tau + 1, t + 1)))
                        st += w * d[bb, tau, dd] * x[bb, tau, dd] * B[bb, tau, n]
                    y[bb, t, dd] += C[bb, t, n] * st
                    if t == T - 1:
                        sf[bb, dd, n] = st
    f = oracle.forward("mamba1", inp)
    assert rel(f["y"], y) < 1e-13
    assert rel(f["s_final"], sf) < 1e-13


def test_hand_worked_two_steps():
    with open(os.path.join(GOLDEN, "hand_worked_T2.json")) as f:
        gold = json.load(f)
    i = gold["inputs"]
    inp = {"x": np.array(i["x"]).reshape(1, 2, 1, 1), "dt_raw": np.array(i["dt_raw"]).reshape(1, 2, 1),
           "A": np.array([i["A"]]), "B": np.array(i["B"]).reshape(1, 2, 1, 1),
           "C": np.array(i["C"]).reshape(1, 2, 1, 1), "s0": np.array(i["s0"]).reshape(1, 1, 1, 1),
           "dy": np.array(i["dy"]).reshape(1, 2, 1, 1), "ds_final": np.array(i["ds_final"]).reshape(1, 1, 1, 1)}
    L = math.log(2.0)

    def ev(e):
        return [eval(s, {"L": L}) for s in e] if isinstance(e, list) else [eval(e, {"L": L})]

    got = dict(oracle.forward("mamba2", inp))
    got.update(oracle.backward("mamba2", inp))
    compared = 0
    for k, expr in gold["expected"].items():
        np.testing.assert_allclose(np.asarray(got[k]).reshape(-1), ev(expr), rtol=1e-14, atol=1e-14, err_msg=k)
        compared += 1
    assert compared == 8


# -------------------------------------------------------- homogeneity identities
def _inner(a, b):
    return float(np.sum(np.asarray(a) * np.asarray(b)))


@pytest.mark.parametrize("variant,cfg", [("mamba2", TINY), ("mamba2", M2_GROUPS), ("mamba1", M1_TINY),
                                         ("mimo", MIMO_TINY)])
def test_euler_identities(variant, cfg):
    inp = f64(cfg)
    f = oracle.forward(variant, inp)
    g = oracle.backward(variant, inp)
    lhs = _inner(inp["dy"], f["y"]) + _inner(inp["ds_final"], f["s_final"])
    scale = abs(lhs) + _inner(np.abs(inp["dy"]), np.abs(f["y"]))
    assert abs(lhs - (_inner(g["dx"], inp["x"]) + _inner(g["ds0"], inp["s0"]))) < 1e-12 * scale
    assert abs(lhs - (_inner(g["dB"], inp["B"]) + _inner(g["ds0"], inp["s0"]))) < 1e-12 * scale
    assert abs(_inner(inp["dy"], f["y"]) - _inner(g["dC"], inp["C"])) < 1e-12 * scale


# -------------------------------------------------------------------- chaining
def _split(inp, t0, variant):
    tdim = 1
    a, b = {}, {}
    for k, v in inp.items():
        if v is None or k in ("A", "s0", "ds_final"):
            a[k] = b[k] = v
        else:
            a[k], b[k] = np.split(v, [t0], axis=tdim)
    return a, b


@pytest.mark.parametrize("variant,cfg", [("mamba2", TINY), ("mamba1", M1_TINY), ("mimo", MIMO_TINY)])
def test_chaining_two_calls_equals_one(variant, cfg):
    inp = f64(cfg)
    t0 = cfg["seqlen"] // 2
    first, second = _split(inp, t0, variant)
    f1 = oracle.forward(variant, first)
    second["s0"] = f1["s_final"]
    f2 = oracle.forward(variant, second)
    full = oracle.forward(variant, inp)
    assert rel(np.concatenate([f1["y"], f2["y"]], axis=1), full["y"]) < 1e-13
    assert rel(f2["s_final"], full["s_final"]) < 1e-13
    g2 = oracle.backward(variant, second)
    first["ds_final"] = g2["ds0"]
    g1 = oracle.backward(variant, first)
    g = oracle.backward(variant, inp)
    for k in ("dx", "ddt_raw", "dB", "dC"):
        assert rel(np.concatenate([g1[k], g2[k]], axis=1), g[k]) < 1e-12, k
    assert rel(g1["ds0"], g["ds0"]) < 1e-12
    if "dA" in g:
        assert rel(g1["dA"] + g2["dA"], g["dA"]) < 1e-12


# ------------------------------------------------------ cross-variant reductions
def test_mimo_rank_one_is_mamba2():
    cfg = scaled(TINY, batch=2, nheads=3)
    inp = f64(cfg)
    d = _softplus(inp["dt_raw"])
    b, T, H, P = inp["x"].shape
    N = inp["B"].shape[-1]
    v = (d[..., None] * inp["x"])[:, :, None]                      # [b,T,1,H,P]
    Bh = np.broadcast_to(inp["B"][:, :, None, 0:1, :], (b, T, 1, H, N)).copy()
    Ch = np.broadcast_to(inp["C"][:, :, None, 0:1, :], (b, T, 1, H, N)).copy()
    da = d * inp["A"][None, None, :]
    fm = oracle.mimo_forward(v, da, Bh, Ch, inp["s0"])
    f2 = oracle.forward("mamba2", inp)
    assert rel(fm["y"][:, :, 0], f2["y"]) < 1e-13
    assert rel(fm["s_final"], f2["s_final"]) < 1e-13
    gm = oracle.mimo_backward(inp["dy"][:, :, None], inp["ds_final"], v, da, Bh, Ch, inp["s0"])
    g2 = oracle.backward("mamba2", inp)
    assert rel(d[..., None] * gm["dv"][:, :, 0], g2["dx"]) < 1e-12
    assert rel(gm["dB"][:, :, 0].sum(axis=2), g2["dB"][:, :, 0]) < 1e-12
    assert rel(gm["dC"][:, :, 0].sum(axis=2), g2["dC"][:, :, 0]) < 1e-12
    assert rel(np.sum(gm["dda"] * d, axis=(0, 1)), g2["dA"]) < 1e-12
    assert rel(gm["ds0"], g2["ds0"]) < 1e-12


def test_mimo_closed_form_da_zero_all_ranks_of_a_step():
    """da = 0: the MIMO state is a running sum of every rank's v (x) B, and y_{t,r} reads the state after ALL R
    rank terms of step t (ranks r' > r included), so a within-step causal mask (r' <= r) fails this; the
    backward's dS_t = ds_final + sum_{tau >= t, r} dy (x) C gives dv, dB, dC, ds0 and dda = <dS_t, s_{t-1}>."""
    rng = np.random.default_rng(21)
    b, T, R, H, P, N = 2, 7, 3, 2, 3, 4
    v = rng.standard_normal((b, T, R, H, P))
    B = rng.standard_normal((b, T, R, H, N)) / 2
    C = rng.standard_normal((b, T, R, H, N)) / 2
    s0 = 0.1 * rng.standard_normal((b, H, P, N))
    dy = rng.standard_normal((b, T, R, H, P))
    dsf = rng.standard_normal((b, H, P, N))
    da = np.zeros((b, T, H))
    incr = np.einsum("btrhp,btrhn->bthpn", v, B)                      # all R ranks of step t
    S = s0[:, None] + np.cumsum(incr, axis=1)                          # [b,T,H,P,N]: state after step t
    y = np.einsum("bthpn,btrhn->btrhp", S, C)
    f = oracle.mimo_forward(v, da, B, C, s0)
    assert rel(f["y"], y) < 1e-13
    assert rel(f["s_final"], S[:, -1]) < 1e-13
    outer = np.einsum("btrhp,btrhn->bthpn", dy, C)
    dS = dsf[:, None] + np.cumsum(outer[:, ::-1], axis=1)[:, ::-1]    # gradient of the state after step t
    S_prev = np.concatenate([s0[:, None], S[:, :-1]], axis=1)
    g = oracle.mimo_backward(dy, dsf, v, da, B, C, s0)
    assert rel(g["dv"], np.einsum("bthpn,btrhn->btrhp", dS, B)) < 1e-13
    assert rel(g["dB"], np.einsum("bthpn,btrhp->btrhn", dS, v)) < 1e-13
    assert rel(g["dC"], np.einsum("bthpn,btrhp->btrhn", S, dy)) < 1e-13
    assert rel(g["ds0"], dS[:, 0]) < 1e-13
    assert rel(g["dda"], np.einsum("bthpn,bthpn->bth", dS, S_prev)) < 1e-12
    # the within-step causal reading differs at every rank but the last: the pin has power
    # (rank r sees the state before step t plus ranks q <= r of it)
    causal = np.einsum("bthpn,btrhn->btrhp", S_prev, C) + np.einsum(
        "btqhp,btqhn,btrhn,rq->btrhp", v, B, C, np.tril(np.ones((R, R))))
    assert rel(causal[:, :, :-1], y[:, :, :-1]) > 1e-3
    assert rel(causal[:, :, -1], y[:, :, -1]) < 1e-13


def test_mamba2_width_one_is_mamba1_with_flat_decay():
    m1 = M1_TINY
    inp1 = f64(m1)
    b, T, D = inp1["x"].shape
    N = inp1["A"].shape[1]
    inp1["A"] = np.repeat(inp1["A"][:, :1], N, axis=1)             # constant over the state
    inp2 = {"x": inp1["x"][..., None], "dt_raw": inp1["dt_raw"], "A": inp1["A"][:, 0].copy(),
            "B": inp1["B"][:, :, None], "C": inp1["C"][:, :, None], "s0": inp1["s0"][:, :, None],
            "dy": inp1["dy"][..., None], "ds_final": inp1["ds_final"][:, :, None]}
    f1 = oracle.forward("mamba1", inp1)
    f2 = oracle.forward("mamba2", inp2)
    assert rel(f2["y"][..., 0], f1["y"]) < 1e-13
    g1 = oracle.backward("mamba1", inp1)
    g2 = oracle.backward("mamba2", inp2)
    assert rel(g2["dx"][..., 0], g1["dx"]) < 1e-12
    assert rel(g2["ddt_raw"], g1["ddt_raw"]) < 1e-12
    assert rel(g2["dB"][:, :, 0], g1["dB"]) < 1e-12
    assert rel(g2["dC"][:, :, 0], g1["dC"]) < 1e-12
    assert rel(g2["dA"], g1["dA"].sum(axis=1)) < 1e-12
    assert rel(g2["ds0"][:, :, 0], g1["ds0"]) < 1e-12


def test_backward_is_independent_of_thread_count():
    inp = f64(scaled(M2_GROUPS, nheads=8, ngroups=2))
    g1 = oracle.backward("mamba2", inp, nthreads=1)
    g4 = oracle.backward("mamba2", inp, nthreads=4)
    for k in g1:
        assert np.array_equal(g1[k], g4[k]), k


@pytest.mark.parametrize("variant,cfg", [("mamba2", scaled(M2_GROUPS, seqlen=21)), ("mamba1", scaled(M1_TINY, seqlen=19)),
                                         ("mimo", scaled(MIMO_TINY, seqlen=13))])
def test_tail_steps_are_identity_steps(variant, cfg):
    """The tail chunk's missing steps, read as dt_raw = -inf (dt' = 0, da = 0;
    MIMO: da = 0) with x = B = C = dy = 0, leave the state unchanged: the serial recurrence
    over T steps padded with such steps to the next chunk multiple gives the
    unpadded outputs on the real steps, the same s_final and ds0, and zero
    gradients on the padding (but MIMO's da gradient there, which does not
    vanish at da = 0).  The kernels compute the tail chunk this way and store
    nothing for the padding."""
    inp = f64(cfg)
    T = cfg["seqlen"]
    Tp = -(-T // cfg["chunk"]) * cfg["chunk"] + cfg["chunk"]  # a whole extra chunk of padding as well
    pad = {}
    for k, v in inp.items():
        if v is None or k in ("A", "s0", "ds_final"):
            pad[k] = v
            continue
        w = np.zeros((v.shape[0], Tp) + v.shape[2:])
        w[:, :T] = v
        if k == "dt_raw":  # dt' = softplus(-inf) = 0; MIMO's slot carries da itself, which pads as 0
            w[:, T:] = 0.0 if variant == "mimo" else -np.inf
        pad[k] = w
    f, fp = oracle.forward(variant, inp), oracle.forward(variant, pad)
    b, bp = oracle.backward(variant, inp), oracle.backward(variant, pad)
    assert np.array_equal(fp["s_final"], f["s_final"]) and np.array_equal(fp["y"][:, :T], f["y"])
    assert not np.any(fp["y"][:, T:])
    for k, v in b.items():
        if v is None:
            continue
        if k in ("ds0", "dA"):
            assert rel(bp[k], v) < 1e-13, k
        else:
            assert rel(bp[k][:, :T], v) < 1e-13, k
            if not (variant == "mimo" and k == "ddt_raw"):  # MIMO's da gradient is e^da <dS, s>, nonzero
                assert not np.any(bp[k][:, T:]), k
