"""Chunkwise (K1..K5) float64 form of the scan and its recompute backward.

TEST INFRASTRUCTURE (see oracle/__init__.py).  Written with numpy from the
algebra of the Mamba-3 page "combined_backward.rs" (burn-mamba,
double_ssd/ssd/serial_recalculated):

* K1  in-chunk inclusive cumsum of da ("K1 — pre-combined Δ·A → intra-chunk
  cumsum"); the chunk-end value is the last element.
* K2  CB = C Bᵀ over the fused length L·R ("K2 — CB matrix").
* K3  chunk-end state from a zero start, with decay exp(cumA_last − cumA)
  (k3_ssd_chunk_state_extended).
* K4  state passing S_{c+1} = exp(cumA_end) S_c + intra_c ("K4 backward step"
  recap).
* K5  y = exp(cumA_t) C S_cᵀ (BLUE) + (CB ∘ decay ∘ mask) v (ORANGE); the
  mask keeps source s for target t iff ⌊s/R⌋ ≤ ⌊t/R⌋ and is applied as −inf
  before the exponential ("ORANGE backward").

The page builds T as nchunks · chunk_len.  Here T may be any length: the last
chunk is shorter (T − (nc − 1)·L steps) and every chunk formula runs on the
steps it has; its chunk end is its own last step.

The backward follows the page's order: recompute K1..K4, walk the chunks in
reverse carrying the state gradient (BLUE + ORANGE + K4 backward), then the
K3, K2 and K1 backwards and the sums of all contributions.

Its only purpose is to be compared with the serial store-all oracle in
``ssd_oracle.c``: two different algorithms that must agree to rounding.
It shares no code with that file.
"""
from __future__ import annotations

import numpy as np


def _softplus(z):
    return np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z)))


def _sigmoid(z):
    return np.where(z >= 0, 1.0 / (1.0 + np.exp(-np.abs(z))), np.exp(-np.abs(z)) / (1.0 + np.exp(-np.abs(z))))


def _mask_mimo(L, R):
    t = np.arange(L * R) // R
    return t[None, :] <= t[:, None]  # [target, source]


def _unit_forward(v, da, Bm, Cm, s0, L):
    """One (batch, head) unit.  v [T,R,P], da [T], Bm/Cm [T,R,N], s0 [P,N].
    Returns y [T,R,P], s_final [P,N] and the chunk-input states [nc,P,N]."""
    T, R, P = v.shape
    N = Bm.shape[2]
    nc = -(-T // L)
    S = s0.copy()
    y = np.empty_like(v)
    S_in = np.empty((nc, P, N))
    for c in range(nc):
        sl = slice(c * L, min((c + 1) * L, T))
        Lc = sl.stop - sl.start
        LR = Lc * R
        keep = _mask_mimo(Lc, R)
        vf = v[sl].reshape(LR, P)
        Bf = Bm[sl].reshape(LR, N)
        Cf = Cm[sl].reshape(LR, N)
        cum = np.cumsum(da[sl])                          # K1
        cum_f = np.repeat(cum, R)                        # fused position -> cumA
        CB = Cf @ Bf.T                                   # K2
        decay_end = np.exp(cum[-1] - cum_f)              # K3
        intra = (decay_end[:, None] * vf).T @ Bf
        diff = np.where(keep, cum_f[:, None] - cum_f[None, :], -np.inf)
        decay_in = np.exp(diff)
        y_blue = np.exp(cum_f)[:, None] * (Cf @ S.T)     # K5 BLUE
        y_orange = (CB * decay_in) @ vf                  # K5 ORANGE
        y[sl] = (y_blue + y_orange).reshape(Lc, R, P)
        S_in[c] = S
        S = np.exp(cum[-1]) * S + intra                  # K4
    return y, S, S_in


def _unit_backward(dy, dS_final, v, da, Bm, Cm, s0, L):
    """Recompute backward of one unit; returns dv, dda, dB, dC, ds0."""
    T, R, P = v.shape
    N = Bm.shape[2]
    nc = -(-T // L)
    _, _, S_in = _unit_forward(v, da, Bm, Cm, s0, L)     # recompute K1..K4
    dv = np.zeros_like(v)
    dda = np.zeros_like(da)
    dB = np.zeros_like(Bm)
    dC = np.zeros_like(Cm)
    dS = dS_final.copy()
    for c in reversed(range(nc)):
        sl = slice(c * L, min((c + 1) * L, T))
        Lc = sl.stop - sl.start
        LR = Lc * R
        keep = _mask_mimo(Lc, R)
        vf = v[sl].reshape(LR, P)
        Bf = Bm[sl].reshape(LR, N)
        Cf = Cm[sl].reshape(LR, N)
        dyf = dy[sl].reshape(LR, P)
        cum = np.cumsum(da[sl])
        cum_f = np.repeat(cum, R)
        CB = Cf @ Bf.T
        Sc = S_in[c]
        # BLUE backward: blue[i,p] = exp(cum_i) sum_n C[i,n] S[p,n]
        dch = dyf * np.exp(cum_f)[:, None]
        dS_blue = (Cf.T @ dch).T                         # [P,N]
        dC_blue = dch @ Sc                               # [LR,N]
        d_cum_f = np.sum(dyf * (Cf @ Sc.T) * np.exp(cum_f)[:, None], axis=1)
        # ORANGE backward: W = CB * decay_in, orange = W v
        diff = np.where(keep, cum_f[:, None] - cum_f[None, :], -np.inf)
        decay_in = np.exp(diff)
        W = CB * decay_in
        dW = dyf @ vf.T
        dv_orange = W.T @ dyf
        dCB = dW * decay_in
        d_diff = dW * CB * decay_in
        d_cum_f += d_diff.sum(axis=1) - d_diff.sum(axis=0)
        # K3 backward: intra = (decay_end * v)^T B, gradient dS (= d intra)
        decay_end = np.exp(cum[-1] - cum_f)
        d_decayed_v = Bf @ dS.T                          # [LR,P]
        dB_k3 = (decay_end[:, None] * vf) @ dS           # [LR,N]
        dv_k3 = d_decayed_v * decay_end[:, None]
        d_decay_end = np.sum(d_decayed_v * vf, axis=1) * decay_end
        d_cum_f -= d_decay_end
        d_cum_last = d_decay_end.sum()
        # K4 backward: S_{c+1} = exp(cum_end) S_c + intra_c
        a_end = np.exp(cum[-1])
        d_cum_last += a_end * np.sum(dS * Sc)
        # K2 backward
        dC_k2 = dCB @ Bf
        dB_k2 = dCB.T @ Cf
        # fold the fused positions back onto the chunk's L steps, then K1
        d_cum = d_cum_f.reshape(Lc, R).sum(axis=1)
        d_cum[-1] += d_cum_last
        dda[sl] = np.cumsum(d_cum[::-1])[::-1]           # suffix sums
        dv[sl] = (dv_orange + dv_k3).reshape(Lc, R, P)
        dB[sl] = (dB_k2 + dB_k3).reshape(Lc, R, N)
        dC[sl] = (dC_k2 + dC_blue).reshape(Lc, R, N)
        dS = a_end * dS + dS_blue
    return dv, dda, dB, dC, dS


# ---------------------------------------------------------------- MIMO form
def mimo_forward(v, da, B, C, s0, L):
    v, da, B, C, s0 = (np.asarray(a, dtype=np.float64) for a in (v, da, B, C, s0))
    b, T, R, H, P = v.shape
    y = np.empty_like(v)
    s_final = np.empty((b, H, P, B.shape[4]))
    for bb in range(b):
        for h in range(H):
            yy, sf, _ = _unit_forward(v[bb, :, :, h], da[bb, :, h], B[bb, :, :, h], C[bb, :, :, h], s0[bb, h], L)
            y[bb, :, :, h] = yy
            s_final[bb, h] = sf
    return {"y": y, "s_final": s_final}


def mimo_backward(dy, ds_final, v, da, B, C, s0, L):
    dy, ds_final, v, da, B, C, s0 = (np.asarray(a, dtype=np.float64) for a in (dy, ds_final, v, da, B, C, s0))
    b, T, R, H, P = v.shape
    out = {"dv": np.empty_like(v), "dda": np.empty_like(da), "dB": np.empty_like(B), "dC": np.empty_like(C),
           "ds0": np.empty_like(s0)}
    for bb in range(b):
        for h in range(H):
            dv, dda, dB, dC, ds0 = _unit_backward(dy[bb, :, :, h], ds_final[bb, h], v[bb, :, :, h],
                                                  da[bb, :, h], B[bb, :, :, h], C[bb, :, :, h], s0[bb, h], L)
            out["dv"][bb, :, :, h] = dv
            out["dda"][bb, :, h] = dda
            out["dB"][bb, :, :, h] = dB
            out["dC"][bb, :, :, h] = dC
            out["ds0"][bb, h] = ds0
    return out


# ------------------------------------------------------------- Mamba-2 form
def mamba2_forward(x, dt_raw, A, B, C, s0, L):
    """Mamba-2 through the R = 1 chunk form: v = dt' x, da = dt' A_h, and
    every head of group g reads that group's B and C."""
    x, dt_raw, A, B, C, s0 = (np.asarray(a, dtype=np.float64) for a in (x, dt_raw, A, B, C, s0))
    b, T, H, P = x.shape
    G = B.shape[2]
    dtp = _softplus(dt_raw)
    y = np.empty_like(x)
    s_final = np.empty_like(s0)
    for bb in range(b):
        for h in range(H):
            g = h // (H // G)
            v = (dtp[bb, :, h, None] * x[bb, :, h])[:, None, :]
            yy, sf, _ = _unit_forward(v, dtp[bb, :, h] * A[h], B[bb, :, g][:, None], C[bb, :, g][:, None],
                                      s0[bb, h], L)
            y[bb, :, h] = yy[:, 0]
            s_final[bb, h] = sf
    return {"y": y, "s_final": s_final}


def mamba2_backward(dy, ds_final, x, dt_raw, A, B, C, s0, L):
    dy, ds_final, x, dt_raw, A, B, C, s0 = (np.asarray(a, dtype=np.float64)
                                            for a in (dy, ds_final, x, dt_raw, A, B, C, s0))
    b, T, H, P = x.shape
    G = B.shape[2]
    dtp = _softplus(dt_raw)
    out = {"dx": np.empty_like(x), "ddt_raw": np.empty_like(dt_raw), "dA": np.zeros_like(A),
           "dB": np.zeros_like(B), "dC": np.zeros_like(C), "ds0": np.empty_like(s0)}
    for bb in range(b):
        for h in range(H):
            g = h // (H // G)
            d = dtp[bb, :, h]
            v = (d[:, None] * x[bb, :, h])[:, None, :]
            dv, dda, dBh, dCh, ds0 = _unit_backward(dy[bb, :, h][:, None], ds_final[bb, h], v, d * A[h],
                                                    B[bb, :, g][:, None], C[bb, :, g][:, None], s0[bb, h], L)
            dv = dv[:, 0]
            out["dx"][bb, :, h] = d[:, None] * dv
            ddtp = np.sum(dv * x[bb, :, h], axis=1) + A[h] * dda
            out["ddt_raw"][bb, :, h] = ddtp * _sigmoid(dt_raw[bb, :, h])
            out["dA"][h] += np.sum(dda * d)
            out["dB"][bb, :, g] += dBh[:, 0]
            out["dC"][bb, :, g] += dCh[:, 0]
            out["ds0"][bb, h] = ds0
    return out
