"""Pins of the float64 KDA oracle (oracle/kda.py) to facts other than itself.

* Central finite differences of the oracle's own forward, perturbing every
  element of q, k, v, g, beta and s0, under the non-uniform objective
  <do, o> + <ds_final, s_final> (so the seed of the reverse loop is tested),
  must match its backward to about 1e-8 relative.
* Each of five planted defects (among them the page's warning: dropping the
  delta-rule path -k (x) dr from dS_dec) must fail that check by more than 100x
  its gate.
* Closed forms: beta = 0 leaves pure per-row decay of s0; with one-hot keys
  and beta = 1 the delta rule overwrites row j of the state with v_t exactly;
  a two-step example worked by hand fixes that o_t reads the updated state.
* Euler identities (o is linear in q; o and s_final are jointly linear in
  (v, s0)), chaining two calls through s_final / ds0, and the GVA sum against
  explicitly repeated query / key heads.
"""
import numpy as np
import pytest

from oracle.kda import KDA_MUTATIONS, kda_backward, kda_forward
from selective_state_space_ssd_gb300 import inputs as synth
from selective_state_space_ssd_gb300.configs import KDA_CONFIGS

TINY = KDA_CONFIGS["kda_tiny_fp32"]
MICRO = dict(TINY, seqlen=6, nheads=1, value_heads=2, key_dim=4, value_dim=3)
NAMES = ("q", "k", "v", "g", "beta", "s0")
GRADS = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "s0": "ds0"}


def _inputs(cfg, seed=0):
    return synth.as_float64(synth.make_kda_inputs(cfg, seed=seed))


def _objective(inp, scale, wo, ws):
    f = kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["s0"], scale)
    return float(np.sum(wo * f["o"]) + np.sum(ws * f["s_final"]))


def _fd_errors(cfg, mutation=0, seed=0):
    """max |analytic - FD| / max |FD| per input, and the number of perturbed elements."""
    inp = _inputs(cfg, seed)
    scale = synth.kda_scale(cfg)
    wo, ws = inp["do"], inp["ds_final"]
    an = kda_backward(wo, ws, inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["s0"], scale,
                      mutation=mutation)
    errs, count = {}, 0
    for name in NAMES:
        x = inp[name]
        fd = np.zeros_like(x)
        flat, fdf = x.reshape(-1), fd.reshape(-1)
        for i in range(flat.size):
            h = 1e-6 * max(1.0, abs(flat[i]))
            old = flat[i]
            flat[i] = old + h
            jp = _objective(inp, scale, wo, ws)
            flat[i] = old - h
            jm = _objective(inp, scale, wo, ws)
            flat[i] = old
            fdf[i] = (jp - jm) / (2 * h)
            count += 1
        errs[name] = float(np.max(np.abs(an[GRADS[name]] - fd)) / max(np.max(np.abs(fd)), 1e-30))
    return errs, count


GATE = 1e-7


def test_backward_matches_central_differences_on_every_element():
    errs, count = _fd_errors(TINY)
    b, T, H, HV, K, V = (TINY[n] for n in ("batch", "seqlen", "nheads", "value_heads", "key_dim", "value_dim"))
    assert count == 2 * b * T * H * K + b * T * HV * (V + K + 1) + b * HV * K * V == 1856
    assert max(errs.values()) < GATE, errs


@pytest.mark.parametrize("mutation", sorted(m for m in KDA_MUTATIONS if m))
def test_every_planted_defect_fails_the_check(mutation):
    errs, _ = _fd_errors(MICRO, mutation=mutation, seed=3)
    assert max(errs.values()) > 100 * GATE, (KDA_MUTATIONS[mutation], errs)


def test_beta_zero_is_pure_decay():
    inp = _inputs(TINY, seed=1)
    inp["beta"] = np.zeros_like(inp["beta"])
    scale = synth.kda_scale(TINY)
    f = kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["s0"], scale)
    G = TINY["value_heads"] // TINY["nheads"]
    cum = np.cumsum(inp["g"], axis=1)                                   # [b,T,HV,K]
    for t in range(TINY["seqlen"]):
        S_t = np.exp(cum[:, t])[..., None] * inp["s0"]
        qh = np.repeat(inp["q"][:, t], G, axis=1) * scale
        np.testing.assert_allclose(f["o"][:, t], np.einsum("bhk,bhkv->bhv", qh, S_t), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(f["s_final"], np.exp(cum[:, -1])[..., None] * inp["s0"], rtol=1e-12, atol=1e-14)
    g = kda_backward(inp["do"], inp["ds_final"], inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["s0"],
                     scale)
    assert np.all(g["dv"] == 0)


def test_one_hot_keys_with_beta_one_overwrite_a_row():
    """k_t = e_j, beta_t = 1: S_t = S_dec + e_j (v_t - S_dec[j]) sets row j to v_t, so the final row j is
    v at the last step that wrote it, decayed by the gates of that row after it."""
    cfg = dict(TINY, seqlen=12)
    inp = _inputs(cfg, seed=2)
    rng = np.random.default_rng(5)
    b, T, H, K = inp["q"].shape
    HV = inp["v"].shape[2]
    G = HV // H
    rows = rng.integers(0, K, size=(b, T, H))
    inp["k"] = np.zeros_like(inp["k"])
    for bb in range(b):
        for t in range(T):
            for h in range(H):
                inp["k"][bb, t, h, rows[bb, t, h]] = 1.0
    inp["beta"] = np.ones_like(inp["beta"])
    f = kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["s0"], 1.0)
    for bb in range(b):
        for hv in range(HV):
            h = hv // G
            for j in range(K):
                writes = [t for t in range(T) if rows[bb, t, h] == j]
                if writes:
                    tl = writes[-1]
                    want = np.exp(np.sum(inp["g"][bb, tl + 1:, hv, j])) * inp["v"][bb, tl, hv]
                else:
                    want = np.exp(np.sum(inp["g"][bb, :, hv, j])) * inp["s0"][bb, hv, j]
                np.testing.assert_allclose(f["s_final"][bb, hv, j], want, rtol=1e-12, atol=1e-14)


def test_output_reads_the_updated_state():
    """F6 reads S_t, after the delta-rule update F5: with s0 = 0, one-hot key e_j and beta = 1 at the first step,
    S_1 = e_j (x) v_1, so o_1 = scale q_1[j] v_1 (reading S_dec instead would give 0).  A second step with key
    e_i (i != j), beta = 1/2 and log-decay g keeps row j decayed by exp(g_2[j]) and writes half of v_2 into row i:
    o_2 = scale (q_2[j] exp(g_2[j]) v_1 + q_2[i] v_2 / 2); all worked out by hand here."""
    b, T, H, HV, K, V = 1, 2, 1, 1, 3, 2
    j, i = 2, 0
    q = np.zeros((b, T, H, K))
    q[0, 0] = [0.3, -0.7, 1.5]
    q[0, 1] = [2.0, 0.4, -1.1]
    k = np.zeros((b, T, H, K))
    k[0, 0, 0, j] = 1.0
    k[0, 1, 0, i] = 1.0
    v = np.array([[[[0.8, -1.2]], [[0.5, 2.0]]]])                     # [b,T,HV,V]
    g = np.zeros((b, T, HV, K))
    g[0, 1, 0] = [-0.2, -0.3, -0.6]
    beta = np.array([[[1.0], [0.5]]])                                  # [b,T,HV]
    scale = 0.25
    f = kda_forward(q, k, v, g, beta, None, scale)
    o1 = scale * q[0, 0, 0, j] * v[0, 0, 0]
    o2 = scale * (q[0, 1, 0, j] * np.exp(g[0, 1, 0, j]) * v[0, 0, 0] + q[0, 1, 0, i] * 0.5 * v[0, 1, 0])
    np.testing.assert_allclose(f["o"][0, 0, 0], o1, rtol=0, atol=1e-15)
    np.testing.assert_allclose(f["o"][0, 1, 0], o2, rtol=0, atol=1e-15)
    S = np.zeros((K, V))
    S[j] = np.exp(g[0, 1, 0, j]) * v[0, 0, 0]
    S[i] = 0.5 * v[0, 1, 0]
    np.testing.assert_allclose(f["s_final"][0, 0], S, rtol=0, atol=1e-15)


def test_euler_identities():
    inp = _inputs(TINY, seed=4)
    scale = synth.kda_scale(TINY)
    f = kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["s0"], scale)
    g = kda_backward(inp["do"], inp["ds_final"], inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["s0"],
                     scale)
    lhs_o = np.sum(inp["do"] * f["o"])
    lhs = lhs_o + np.sum(inp["ds_final"] * f["s_final"])
    assert abs(np.sum(g["dq"] * inp["q"]) - lhs_o) <= 1e-12 * max(1.0, abs(lhs_o))
    rhs = np.sum(g["dv"] * inp["v"]) + np.sum(g["ds0"] * inp["s0"])
    assert abs(rhs - lhs) <= 1e-12 * max(1.0, abs(lhs))


def test_chaining_two_calls_equals_one():
    inp = _inputs(TINY, seed=6)
    scale = synth.kda_scale(TINY)
    T1 = 7
    cut = lambda a, sl: a[:, sl]
    full_f = kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["s0"], scale)
    full_b = kda_backward(inp["do"], inp["ds_final"], inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                          inp["s0"], scale)
    a, b_ = slice(0, T1), slice(T1, None)
    f1 = kda_forward(*(cut(inp[n], a) for n in ("q", "k", "v", "g", "beta")), inp["s0"], scale)
    f2 = kda_forward(*(cut(inp[n], b_) for n in ("q", "k", "v", "g", "beta")), f1["s_final"], scale)
    np.testing.assert_allclose(np.concatenate([f1["o"], f2["o"]], axis=1), full_f["o"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(f2["s_final"], full_f["s_final"], rtol=1e-12, atol=1e-13)
    g2 = kda_backward(cut(inp["do"], b_), inp["ds_final"], *(cut(inp[n], b_) for n in ("q", "k", "v", "g", "beta")),
                      f1["s_final"], scale)
    g1 = kda_backward(cut(inp["do"], a), g2["ds0"], *(cut(inp[n], a) for n in ("q", "k", "v", "g", "beta")),
                      inp["s0"], scale)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_allclose(np.concatenate([g1[name], g2[name]], axis=1), full_b[name], rtol=1e-10,
                                   atol=1e-12)
    np.testing.assert_allclose(g1["ds0"], full_b["ds0"], rtol=1e-10, atol=1e-12)


def test_grouped_heads_equal_repeated_heads_summed():
    """GVA: value head hv reads query / key head hv // G, and dq, dk of a query / key head are the sums over its
    G value heads -- the same as repeating q, k per value head (G = 1) and summing those gradients by hand."""
    inp = _inputs(TINY, seed=7)
    scale = synth.kda_scale(TINY)
    G = TINY["value_heads"] // TINY["nheads"]
    rep = {n: np.repeat(inp[n], G, axis=2) for n in ("q", "k")}
    a = kda_backward(inp["do"], inp["ds_final"], inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["s0"],
                     scale)
    r = kda_backward(inp["do"], inp["ds_final"], rep["q"], rep["k"], inp["v"], inp["g"], inp["beta"], inp["s0"],
                     scale)
    b, T, H, K = inp["q"].shape
    for name in ("dq", "dk"):
        summed = r[name].reshape(b, T, H, G, K).sum(axis=3)
        np.testing.assert_allclose(a[name], summed, rtol=1e-12, atol=1e-14)
    for name in ("dv", "dg", "dbeta", "ds0"):
        np.testing.assert_allclose(a[name], r[name], rtol=1e-12, atol=1e-14)
