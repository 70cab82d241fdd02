"""Float64 oracle for the KDA delta-rule recurrence and its BPTT backward.

TEST INFRASTRUCTURE, like the rest of this package: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s oracle legs may import it, and
it imports nothing from the CUDA library.

It follows the notes page "sec-10.tex" (section "反向传播推导"): the forward
recap F1-F6 and the reverse-time loop of steps 1-6, with the state of every
step stored (store-all).  Per batch element and value head, with state S of
shape [K, V]:

    F1  S_dec = exp(g_t) (.) S_{t-1}          (g_t: one log-decay per key row)
    F2  p_t   = k_t^T S_dec                    [V]
    F3  r_t   = v_t - p_t
    F4  a_t   = beta_t k_t                     [K]
    F5  S_t   = S_dec + a_t (x) r_t
    F6  o_t   = q_t^T S_t                      with q_t already multiplied by `scale`

Grouped value heads (GVA): value head hv reads query / key head hv // G,
G = HV / H; the backward sums the per-value-head dq, dk over the G heads of
each query / key head (the page's view + sum) and multiplies dq by `scale`.

Shapes (row-major): q, k [b,T,H,K]; v [b,T,HV,V]; g [b,T,HV,K];
beta [b,T,HV]; s0, s_final [b,HV,K,V]; o [b,T,HV,V].

Readings where the page is silent: q and k enter as given (the recurrence
normalises nothing); the reverse loop is seeded with the gradient of the final
state ds_final (the VJP of (o, s_final)), and its last dS is ds0.

``mutation`` (backward only) plants one defect, for the tests that show the
finite-difference check catches it; 0 is the correct VJP.
"""
from __future__ import annotations

import numpy as np

KDA_MUTATIONS = {
    0: "none",
    1: "drop the delta-rule path -k (x) dr from dS_dec",
    2: "seed the state gradient with zeros",
    3: "drop o's own contribution q (x) do to dS",
    4: "use S_dec where S_t belongs in dq",
    5: "carry dS_dec back without the decay exp(g)",
}


def _f64(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _expand(x, G):
    """Query / key head h -> the G value heads h*G .. h*G+G-1: [b,T,H,K] -> [b,T,H*G,K]."""
    return np.repeat(x, G, axis=2)


def kda_forward(q, k, v, g, beta, s0=None, scale=1.0, keep=False):
    """o and s_final of the recurrence F1-F6.  With keep=True also returns the
    per-step S_dec, r and a (store-all), which the backward needs."""
    q, k, v, g, beta, s0 = map(_f64, (q, k, v, g, beta, s0))
    b, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    assert HV % H == 0
    G = HV // H
    qe, ke = _expand(q, G) * scale, _expand(k, G)
    S = np.zeros((b, HV, K, V)) if s0 is None else s0.copy()
    o = np.zeros((b, T, HV, V))
    Sdec_all = np.zeros((T, b, HV, K, V)) if keep else None
    r_all = np.zeros((T, b, HV, V)) if keep else None
    a_all = np.zeros((T, b, HV, K)) if keep else None
    for t in range(T):
        Sdec = np.exp(g[:, t])[..., :, None] * S                       # F1
        p = np.einsum("bhk,bhkv->bhv", ke[:, t], Sdec)                  # F2
        r = v[:, t] - p                                                 # F3
        a = beta[:, t][..., None] * ke[:, t]                            # F4
        S = Sdec + a[..., :, None] * r[..., None, :]                    # F5
        o[:, t] = np.einsum("bhk,bhkv->bhv", qe[:, t], S)               # F6
        if keep:
            Sdec_all[t], r_all[t], a_all[t] = Sdec, r, a
    out = {"o": o, "s_final": S}
    if keep:
        out.update(Sdec=Sdec_all, r=r_all, a=a_all)
    return out


def kda_backward(do, ds_final, q, k, v, g, beta, s0=None, scale=1.0, mutation=0):
    """Gradients dq, dk [b,T,H,K], dv [b,T,HV,V], dg [b,T,HV,K], dbeta [b,T,HV]
    and ds0 [b,HV,K,V] of <do, o> + <ds_final, s_final>: the page's steps 1-6,
    t from T-1 down to 0, on the stored per-step intermediates."""
    do, ds_final = _f64(do), _f64(ds_final)
    q, k, g, beta = _f64(q), _f64(k), _f64(g), _f64(beta)
    fw = kda_forward(q, k, v, g, beta, s0, scale, keep=True)
    b, T, H, K = q.shape
    HV, V = do.shape[2], do.shape[3]
    G = HV // H
    qe, ke = _expand(q, G) * scale, _expand(k, G)
    dS = np.zeros_like(ds_final) if mutation == 2 else ds_final.copy()   # dS_acc, seeded with ds_final
    dq_e = np.zeros((b, T, HV, K))
    dk_e = np.zeros((b, T, HV, K))
    dv = np.zeros((b, T, HV, V))
    dg = np.zeros((b, T, HV, K))
    dbeta = np.zeros((b, T, HV))
    for t in range(T - 1, -1, -1):
        Sdec, r, a = fw["Sdec"][t], fw["r"][t], fw["a"][t]
        qt, kt, do_t = qe[:, t], ke[:, t], do[:, t]
        S_t = Sdec + a[..., :, None] * r[..., None, :]
        # step 1: o_t = q_t^T S_t
        if mutation != 3:
            dS = dS + qt[..., :, None] * do_t[..., None, :]
        dq_e[:, t] = np.einsum("bhv,bhkv->bhk", do_t, Sdec if mutation == 4 else S_t)
        # step 2: S_t = S_dec + a_t (x) r_t
        da = np.einsum("bhv,bhkv->bhk", r, dS)
        dr = np.einsum("bhk,bhkv->bhv", a, dS)
        # step 3: a_t = beta_t k_t
        dbeta[:, t] = np.einsum("bhk,bhk->bh", kt, da)
        dk_a = beta[:, t][..., None] * da
        # step 4: r_t = v_t - k_t^T S_dec
        dv[:, t] = dr
        dk_r = -np.einsum("bhv,bhkv->bhk", dr, Sdec)
        dSdec_r = -kt[..., :, None] * dr[..., None, :]
        # step 5: both paths into S_dec, then S_dec = exp(g_t) (.) S_{t-1}
        dSdec = dS if mutation == 1 else dS + dSdec_r
        dg[:, t] = np.einsum("bhkv,bhkv->bhk", Sdec, dSdec)
        dk_e[:, t] = dk_a + dk_r
        dS = dSdec if mutation == 5 else np.exp(g[:, t])[..., :, None] * dSdec
    # step 6: the value heads' dq, dk summed onto their query / key head (view + sum); dq carries the scale
    dq = dq_e.reshape(b, T, H, G, K).sum(axis=3) * scale
    dk = dk_e.reshape(b, T, H, G, K).sum(axis=3)
    return {"dq": dq, "dk": dk, "dv": dv, "dg": dg, "dbeta": dbeta, "ds0": dS}
