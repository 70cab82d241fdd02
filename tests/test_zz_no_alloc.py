"""ssd_forward_static: the forward for callers that cannot allocate device
memory (for example code running inside a framework that owns every GPU
allocation, or a loop that must not allocate after start-up).  It takes no
workspace and uses the library's fixed 32 MiB device array instead.

Each case calls it through the C ABI twice in a row, on different inputs, and
compares both results with ssd_forward (which uses a caller workspace) within
the parity tolerance of the other GPU tests.  After each call the array's
device status word must read 0 (no bounded wait gave up).  The outputs are
allocated before the calls, and the second call must leave both torch's
allocated bytes and the device's free bytes unchanged.  A problem whose
scratch exceeds the fixed array must be refused with SSD_ERR_TOO_LARGE before
anything runs.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from selective_state_space_ssd_gb300 import binding
from selective_state_space_ssd_gb300 import inputs as synth
from selective_state_space_ssd_gb300.configs import CONFIGS, scaled

from parity import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu

CASES = {
    # CUDA-core path: its scratch holds the chunk states
    "mamba2_tiny_fp32": CONFIGS["mamba2_tiny_fp32"],
    # tensor-core path: its scratch holds the bf16 chunk states and C B^T
    "mamba2_bf16_tc": scaled(CONFIGS["mamba2_130m_bf16"], batch=2, seqlen=256, nheads=4),
    # MIMO on the tensor-core kernels (the fused sequence): chunk states and C B^T of 3 heads in the scratch
    "mimo_bf16": scaled(CONFIGS["mimo_r4_bf16"], batch=1, seqlen=256, nheads=3, ngroups=3),
    "mamba1_fp32": scaled(CONFIGS["mamba1_fp32"], batch=2, seqlen=256, nheads=40),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_static_forward_matches_workspace_forward_twice(name, cuda_lib):
    cfg = CASES[name]
    tol = TOL[cfg["dtype"]]
    prob = binding.problem(cfg)
    assert binding.ssd_forward_static_status(read=False)[0] == 0  # the start-up step: module loaded
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs each time
        t = to_device(synth.make_inputs(cfg, seed=seed))
        y_ref, sf_ref = binding.forward(cfg, t["x"], t["dt_raw"], t["A"], t["B"], t["C"], t["s0"])
        y = torch.empty_like(t["x"])
        sf = torch.empty_like(t["ds_final"])
        torch.cuda.synchronize()
        before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
        binding.ssd_forward_static(prob, t["x"], t["dt_raw"], t["A"], t["B"], t["C"], t["s0"], y, sf)
        torch.cuda.synchronize()
        after = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
        if call == 1:
            assert after == before, f"the second call allocated device memory: {before} -> {after}"
        assert binding.ssd_forward_static_status() == (0, 0)
        assert rel_err(y, y_ref.double().cpu().numpy()) <= tol
        assert rel_err(sf, sf_ref.double().cpu().numpy()) <= tol


def test_static_forward_refuses_problems_beyond_its_array(cuda_lib):
    big = CONFIGS["mimo_r4_bf16"]  # its CUDA-core forward needs 268 MB of chunk states
    prob = binding.problem(big)
    need = binding.ssd_workspace_size(prob, False)
    assert need > 32 << 20
    # rejected during validation: nothing is dereferenced or launched
    fake = 1 << 20
    st = cuda_lib.ssd_forward_static(ctypes.byref(prob), fake, fake, None, fake, fake, None, fake, fake, None)
    assert st == 9  # SSD_ERR_TOO_LARGE
    assert "32 MiB" in binding.ssd_status_string(st)
