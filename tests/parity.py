"""Helpers shared by the GPU parity tests: run the CUDA library through its
C ABI and the float64 oracle on the same seeded inputs, and compare them with
the metric max|gpu - ref| / max|ref| per output."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from selective_state_space_ssd_gb300 import binding
from selective_state_space_ssd_gb300 import inputs as synth

# max|err| / max|ref| bounds: fp32 path, and bf16 inputs with fp32 accumulation
TOL = {"f32": 1e-4, "bf16": 2e-2}
OUTPUTS = ("y", "s_final", "dx", "ddt_raw", "dA", "dB", "dC", "ds0")


def to_device(inp: dict, device="cuda") -> dict:
    return {k: (None if v is None else v.to(device)) for k, v in inp.items()}


def zero_workspace(cfg: dict, backward: bool, device="cuda"):
    prob = binding.problem(cfg)
    n = binding.ssd_workspace_size(prob, backward)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device), n


def status_word(ws) -> int:
    """The device status word kept in the first 4 bytes of the workspace."""
    return int(ws[:4].view(torch.int32).item())


def run_gpu(cfg: dict, dev_inputs: dict, s0_null: bool = False) -> dict:
    t = dev_inputs
    s0 = None if s0_null else t["s0"]
    wsf = zero_workspace(cfg, False)
    wsb = zero_workspace(cfg, True)
    y, sf = binding.forward(cfg, t["x"], t["dt_raw"], t["A"], t["B"], t["C"], s0, workspace=wsf)
    g = binding.backward(cfg, t["dy"], t["ds_final"], t["x"], t["dt_raw"], t["A"], t["B"], t["C"], s0, workspace=wsb)
    torch.cuda.synchronize()
    assert status_word(wsf[0]) == 0 and status_word(wsb[0]) == 0, "a device-side bounded wait gave up"
    out = {"y": y, "s_final": sf}
    out.update(g)
    return out


def run_oracle(cfg: dict, cpu_inputs: dict) -> dict:
    f64 = synth.as_float64(cpu_inputs)
    out = dict(oracle.forward(cfg["variant"], f64))
    out.update(oracle.backward(cfg["variant"], f64))
    return out


def rel_err(gpu, ref) -> float:
    g = gpu.detach().float().cpu().numpy().astype(np.float64) if hasattr(gpu, "detach") else np.asarray(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite values in GPU output"
    denom = float(np.max(np.abs(r)))
    return float(np.max(np.abs(g - r))) / max(denom, 1e-30)


def compare(cfg: dict, gpu: dict, ref: dict, tol: float | None = None, names=OUTPUTS) -> dict:
    """Relative error of every output both sides have; asserts each is within
    tolerance and that at least the six gradients and y/s_final were checked."""
    tol = TOL[cfg["dtype"]] if tol is None else tol
    errs = {}
    for k in names:
        if k in ref and ref[k] is not None and gpu.get(k) is not None:
            errs[k] = rel_err(gpu[k], ref[k])
    expected = 7 if cfg["variant"] == "mimo" else 8
    assert len(errs) == expected, sorted(errs)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"outside {tol}: {bad}; all: {errs}"
    return errs
