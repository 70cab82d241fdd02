"""The benchmark's measurement model, checked without a GPU: the algorithmic
bytes, FLOPs and exponentials of a forward + backward pair at the workloads'
sizes, and a byte count for every kernel the library launches (so that the
roofline of whichever kernel dominates a step is never left undefined)."""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from selective_state_space_ssd_gb300.configs import CONFIGS, KDA_CONFIGS  # noqa: E402

CSRC = os.path.join(ROOT, "selective_state_space_ssd_gb300", "csrc")


def test_headline_bytes_and_flops():
    """Mamba-2 2.7B layer: leaf inputs and outputs 370.1 MB forward + 562.0 MB
    backward; 7 (2 L P N) + 3 (2 L^2 P) FLOPs per (b, chunk, head) and
    4 (2 L^2 N) per (b, chunk, group)."""
    cfg = CONFIGS["mamba2_2p7b_bf16"]
    fb, bb = bench.algorithmic_bytes(cfg)
    assert round(fb / 1e6, 1) == 370.1 and round(bb / 1e6, 1) == 562.0
    b, T, H, P, N, L, G = 4, 4096, 80, 64, 128, 64, 1
    nc = T // L
    flops = b * nc * (H * (7 * 2 * L * P * N + 3 * 2 * L * L * P) + G * 4 * 2 * L * L * N)
    assert bench.tensor_flops(cfg) == flops
    assert round(flops / 1e9, 1) == 183.6


def test_mamba1_decays():
    """One decay per (step, channel, state) in the forward and again in the
    backward's replay: 2 b T D N = 805.3 M at the Mamba-1 workload."""
    cfg = CONFIGS["mamba1_fp32"]
    assert bench.exp_count(cfg) == 2 * 8 * 2048 * 1536 * 16
    assert bench.exp_count(CONFIGS["mamba2_2p7b_bf16"]) == 0


def _launch_names():
    names = set()
    for f in os.listdir(CSRC):
        with open(os.path.join(CSRC, f)) as fh:
            names.update(re.findall(r'SSD_LAUNCH\(\s*"(\w+)"', fh.read()))
        with open(os.path.join(CSRC, f)) as fh:
            src = fh.read()
        # launch names chosen at run time (the scan launch)
        if "k_tc_scan_pair_cb" in src:
            names.update(re.findall(r'"(k_tc_\w+_cb)"', src))
    return names


def test_every_launch_has_a_byte_count():
    names = _launch_names()
    assert {"k_tc_bwd_chunk", "k_tc_fwd_chunk", "k_tc_scan_pair_cb", "k_m1_backward", "k_chunk_bwd"} <= names
    kda = {n for n in names if n.startswith("k_kda")}
    assert kda == {"k_kda_forward", "k_kda_checkpoints", "k_kda_backward", "k_kda_rows", "k_kda_gva"}
    for cfg in CONFIGS.values():
        for n in names - kda:
            assert bench.kernel_bytes(n, cfg) is not None, (n, cfg["variant"])
    for cfg in KDA_CONFIGS.values():
        for n in kda:
            assert bench.kernel_bytes(n, cfg) > 0, n


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_step_roofline_is_positive(name):
    cfg = CONFIGS[name]
    fb, bb = bench.algorithmic_bytes(cfg)
    assert fb > 0 and bb > fb  # the backward re-reads the leaves and writes six gradients


def test_tensor_core_path_choice():
    assert bench.tc_path(CONFIGS["mamba2_2p7b_bf16"]) and bench.tc_path(CONFIGS["mimo_r4_bf16"])
    assert not bench.tc_path(CONFIGS["mamba2_tiny_fp32"]) and not bench.tc_path(CONFIGS["mamba1_fp32"])
    assert bench.path_dtype(CONFIGS["mimo_r4_bf16"]) == "bf16"


def test_roofline_takes_the_bytes_of_the_pass_the_kernel_runs_in():
    cfg = CONFIGS["mamba2_2p7b_bf16"]
    fb, bb = bench.algorithmic_bytes(cfg)
    assert bench.kernel_direction_bytes("k_tc_fwd_chunk", cfg) == fb
    assert bench.kernel_direction_bytes("k_tc_states_cb", cfg) == fb
    assert bench.kernel_direction_bytes("k_tc_bwd_chunk", cfg) == bb
    assert bench.kernel_direction_bytes("k_tc_scan_pair_cb", cfg) == bb
    # the design bytes of the backward chunk kernel include the chunk states it reads: more than the pass's own
    assert bench.kernel_bytes("k_tc_bwd_chunk", cfg) > bb


def test_parity_errors_are_relative_to_the_reference_maximum():
    import numpy as np
    import torch
    ref = {"y": np.array([1.0, -4.0, 2.0]), "dx": np.array([0.5, 0.25])}
    gpu = {"y": torch.tensor([1.0, -4.0, 2.2]), "dx": torch.tensor([0.5, 0.25]), "dB": torch.zeros(1)}
    errs = bench.parity_errors(gpu, ref)
    assert set(errs) == {"y", "dx"}
    assert abs(errs["y"] - 0.2 / 4.0) < 1e-6 and errs["dx"] == 0.0


def test_mimo_executed_flops_count_the_fused_sequence():
    cfg = CONFIGS["mimo_r4_bf16"]
    # the tensor-core kernels run chunks of 64 fused positions instead of the pages' L * R = 256: the L x L terms
    # shrink by R, the L x N terms stay
    assert bench.tensor_flops(cfg, executed=True) < bench.tensor_flops(cfg)
    m2 = CONFIGS["mamba2_2p7b_bf16"]
    assert bench.tensor_flops(m2, executed=True) == bench.tensor_flops(m2)


@pytest.mark.parametrize("dt,steps", [(40.0, 3), (0.5, 200), (2.0, 60)])
def test_reference_arm_caps_its_timed_passes(dt, steps, monkeypatch, capsys):
    """The reference arm's steps are whole-workload oracle passes: it times at most REF_BUDGET_S of them (at least
    3, at most --steps) and reports how many ran.  The oracle is replaced by a stub that reports dt seconds."""
    calls = []

    def fake_time_oracle(cfg, inputs=None, whole=False, **kw):
        calls.append(whole)
        return 1.0, dt, 4, "stub", cfg, inputs, None

    monkeypatch.setattr(bench, "time_oracle", fake_time_oracle)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "200", "--warmup", "3"])
    monkeypatch.delenv("RANK", raising=False)
    assert bench.main() == 0
    line = __import__("json").loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == steps and line["steps_requested"] == 200
    assert len(calls) == 3 + steps and all(calls)
    assert line["ms_per_step"] == pytest.approx(1e3 * dt)
