"""Failure detection: a bounded device-side wait that runs out.

Every wait of the tensor-core kernels on one of their barriers gives up after
a time limit, writes a nonzero code into the device status word and returns.
ssd_wait_selftest makes one such wait run out on purpose (one thread waits on
a barrier that nothing completes, with a limit of a few milliseconds), with
no copy, MMA or TMEM allocation in flight.  The test checks that the call
returns, that the word then reads SSD_ERR_TIMEOUT with the self-test's code,
and that the context stays usable: a forward + backward afterwards on the
same stream matches the oracle and leaves its own status words at 0.
"""
import pytest
import torch

from selective_state_space_ssd_gb300 import binding
from selective_state_space_ssd_gb300 import inputs as synth
from selective_state_space_ssd_gb300.configs import CONFIGS, scaled

from parity import compare, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_TIMEOUT = 0, 1, 7


def test_wait_runs_out_and_reports_through_the_status_word(cuda_lib):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert binding.ssd_read_status(ws) == (SSD_OK, 0)
    assert binding.ssd_wait_selftest(ws, 5000) == SSD_OK  # 5 ms limit
    st, code = binding.ssd_read_status(ws)
    assert (st, code) == (SSD_ERR_TIMEOUT, 1)
    # the limit is checked on the host; nothing is launched for a bad one
    assert binding.ssd_wait_selftest(ws, 0) == SSD_ERR_INVALID_ARG
    assert binding.ssd_wait_selftest(ws, 2_000_001) == SSD_ERR_INVALID_ARG
    assert binding.ssd_read_status(ws) == (SSD_ERR_TIMEOUT, 1)  # untouched by the refused calls


def test_context_is_usable_after_a_wait_ran_out(cuda_lib):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert binding.ssd_wait_selftest(ws, 2000) == SSD_OK
    assert binding.ssd_read_status(ws)[0] == SSD_ERR_TIMEOUT
    cfg = scaled(CONFIGS["mamba2_2p7b_bf16"], batch=1, seqlen=192, nheads=2)  # the tensor-core kernels
    cpu = synth.make_inputs(cfg, seed=5)
    got = run_gpu(cfg, to_device(cpu))  # asserts both workspaces' status words are 0
    compare(cfg, got, run_oracle(cfg, cpu))
