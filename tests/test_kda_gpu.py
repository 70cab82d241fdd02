"""GPU parity of the KDA delta-rule kernels (through the C ABI) with the
float64 oracle (oracle/kda.py), element by element, max|gpu - ref| / max|ref|
within the fp32 bound 1e-4 for every output.

Cases cover: the tiny shape of the oracle's pins; key and value widths that
are not multiples of the warp layout (masked key rows past K; V = 45: a last
column warp with one live column of four, and two backward CTAs, the second
with idle warps) with T not a multiple of the 8-step checkpoint segment; a zero initial state; one, two
and four value heads per query / key head; head dimension 128.  At the full
workload size (b=2, T=1024, 16 value heads, K=V=128) one query / key head
group is checked against the oracle (its G value heads are independent of
the rest), and the Euler identities of the recurrence hold over all of it.
The backward is bitwise repeatable.
"""
import numpy as np
import pytest
import torch

from oracle.kda import kda_backward, kda_forward
from selective_state_space_ssd_gb300 import binding
from selective_state_space_ssd_gb300 import inputs as synth
from selective_state_space_ssd_gb300.configs import KDA_CONFIGS

from parity import rel_err

pytestmark = pytest.mark.gpu

TOL = 1e-4
BASE = KDA_CONFIGS["kda_tiny_fp32"]
CASES = {
    "tiny": BASE,
    "ragged": dict(BASE, batch=2, seqlen=37, nheads=1, value_heads=2, key_dim=40, value_dim=20),
    "ragged_cols": dict(BASE, batch=1, seqlen=29, nheads=1, value_heads=2, key_dim=37, value_dim=45),
    # degenerate: one step; widths below one warp's layout (5 key rows, 3 of a warp's 4 value columns)
    "one_step": dict(BASE, batch=2, seqlen=1),
    "narrow": dict(BASE, batch=1, seqlen=3, nheads=1, value_heads=1, key_dim=5, value_dim=3),
    "gva4": dict(BASE, batch=1, seqlen=48, nheads=1, value_heads=4, key_dim=32, value_dim=16),
    "dim128": dict(BASE, batch=1, seqlen=100, nheads=2, value_heads=4, key_dim=128, value_dim=128),
    "one_value_head": dict(BASE, batch=2, seqlen=50, nheads=3, value_heads=3, key_dim=64, value_dim=40),
}
OUT_F = ("o", "s_final")
OUT_B = ("dq", "dk", "dv", "dg", "dbeta", "ds0")


def _run(cfg, cpu, zero_s0=False):
    dev = {k: v.cuda() for k, v in cpu.items()}
    s0 = None if zero_s0 else dev["s0"]
    o, sf = binding.kda_forward(cfg, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], s0)
    g = binding.kda_backward(cfg, dev["do"], dev["ds_final"], dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], s0)
    torch.cuda.synchronize()
    return dict(g, o=o, s_final=sf)


def _oracle(cfg, cpu, zero_s0=False):
    f = synth.as_float64(cpu)
    s0 = None if zero_s0 else f["s0"]
    scale = synth.kda_scale(cfg)
    out = kda_forward(f["q"], f["k"], f["v"], f["g"], f["beta"], s0, scale)
    out.update(kda_backward(f["do"], f["ds_final"], f["q"], f["k"], f["v"], f["g"], f["beta"], s0, scale))
    return out


@pytest.mark.parametrize("name", sorted(CASES))
def test_kda_matches_the_oracle(name):
    cfg = CASES[name]
    cpu = synth.make_kda_inputs(cfg, seed=11)
    got, ref = _run(cfg, cpu), _oracle(cfg, cpu)
    errs = {k: rel_err(got[k], ref[k]) for k in OUT_F + OUT_B}
    assert max(errs.values()) <= TOL, errs


def test_kda_zero_initial_state():
    cfg = CASES["ragged"]
    cpu = synth.make_kda_inputs(cfg, seed=12, zero_s0=True)
    got, ref = _run(cfg, cpu, zero_s0=True), _oracle(cfg, cpu, zero_s0=True)
    errs = {k: rel_err(got[k], ref[k]) for k in OUT_F + OUT_B}
    assert max(errs.values()) <= TOL, errs


def test_kda_backward_is_bitwise_repeatable():
    cfg = CASES["dim128"]
    cpu = synth.make_kda_inputs(cfg, seed=13)
    a, b = _run(cfg, cpu), _run(cfg, cpu)
    for k in OUT_F + OUT_B:
        assert torch.equal(a[k], b[k]), k


def test_kda_full_size_one_group_and_euler_identities():
    cfg = KDA_CONFIGS["kda_fp32"]
    cpu = synth.make_kda_inputs(cfg, seed=14)
    got = _run(cfg, cpu)
    G = cfg["value_heads"] // cfg["nheads"]
    bb, h = 1, 3  # one batch element, one query / key head and its G value heads
    vs = slice(h * G, (h + 1) * G)
    sub = {"q": cpu["q"][bb:bb + 1, :, h:h + 1], "k": cpu["k"][bb:bb + 1, :, h:h + 1]}
    for n in ("v", "g", "beta", "do"):
        sub[n] = cpu[n][bb:bb + 1, :, vs]
    for n in ("s0", "ds_final"):
        sub[n] = cpu[n][bb:bb + 1, vs]
    ref = _oracle(dict(cfg, batch=1, nheads=1, value_heads=G), sub)
    pick = {"q": lambda t: t[bb:bb + 1, :, h:h + 1], "k": lambda t: t[bb:bb + 1, :, h:h + 1]}
    errs = {}
    for k in OUT_F + OUT_B:
        x = got[k]
        if k in ("dq", "dk"):
            x = x[bb:bb + 1, :, h:h + 1]
        elif k in ("s_final", "ds0"):
            x = x[bb:bb + 1, vs]
        else:
            x = x[bb:bb + 1, :, vs]
        errs[k] = rel_err(x, ref[k])
    assert max(errs.values()) <= TOL, errs
    # o is linear in q; o and s_final are jointly linear in (v, s0): exact for any correct VJP at any size
    f = {k: v.double() for k, v in cpu.items()}
    g = {k: v.double().cpu() for k, v in got.items()}
    do_o = float((f["do"] * g["o"]).sum())
    lhs = do_o + float((f["ds_final"] * g["s_final"]).sum())
    assert abs(float((g["dq"] * f["q"]).sum()) - do_o) <= 1e-4 * max(1.0, abs(do_o))
    rhs = float((g["dv"] * f["v"]).sum() + (g["ds0"] * f["s0"]).sum())
    assert abs(rhs - lhs) <= 1e-4 * max(1.0, abs(lhs))
