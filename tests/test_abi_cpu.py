"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
symbol the header declares, and validates its arguments on the host (no
kernel is launched by any call here: every call fails validation first)."""
import ctypes
import os
import re
import subprocess

import pytest

from selective_state_space_ssd_gb300 import binding
from selective_state_space_ssd_gb300.configs import CONFIGS, scaled

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssd.h")


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z_]+)\s*\(", text)))


def test_header_declares_the_abi():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_loads_and_exports_every_declared_symbol(cuda_lib):
    for name in declared_functions():
        assert hasattr(cuda_lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (ssd_[a-z_]+)\b", out))
    assert set(declared_functions()) <= exported
    assert cuda_lib.ssd_version() >= 100


def test_library_is_built_for_sm_103a():
    out = subprocess.run(["cuobjdump", "--list-elf", binding.library_path()], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout


def test_status_strings(cuda_lib):
    for code in range(0, 10):
        s = binding.ssd_status_string(code)
        assert s.startswith("SSD_")
    assert binding.ssd_status_string(99) == "SSD_ERR_UNKNOWN"


def _status(fn, *args):
    return fn(*args)


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_workspace_query_accepts_every_config(cuda_lib, name):
    p = binding.problem(CONFIGS[name])
    fwd = binding.ssd_workspace_size(p, False)
    bwd = binding.ssd_workspace_size(p, True)
    assert fwd >= 0 and bwd > 0


@pytest.mark.parametrize("over,code", [
    (dict(ngroups=3), 2),                   # H % G != 0
    (dict(headdim=0), 2),
    (dict(dstate=300), 2),                  # beyond this build's limit
    (dict(chunk=512), 2),                   # chunk beyond this build's limit
    (dict(chunk=0), 2),
    (dict(seqlen=0), 2),
    (dict(seqlen=100), 0),                  # T % chunk != 0: a tail chunk of 4 steps
    (dict(chunk=128), 0),                   # chunk > T: one partial chunk
])
def test_shape_validation(cuda_lib, over, code):
    cfg = scaled(CONFIGS["mamba2_tiny_fp32"], **over)
    p = binding.problem(cfg)
    n = ctypes.c_size_t(0)
    assert cuda_lib.ssd_workspace_size(ctypes.byref(p), 0, ctypes.byref(n)) == code


def test_variant_specific_validation(cuda_lib):
    n = ctypes.c_size_t(0)
    m1 = binding.problem(scaled(CONFIGS["mamba1_fp32"], dtype="bf16"))
    assert cuda_lib.ssd_workspace_size(ctypes.byref(m1), 1, ctypes.byref(n)) == 3  # SSD_ERR_DTYPE
    m1 = binding.problem(scaled(CONFIGS["mamba1_fp32"], headdim=2))
    assert cuda_lib.ssd_workspace_size(ctypes.byref(m1), 1, ctypes.byref(n)) == 2
    bad = binding.problem(CONFIGS["mamba2_tiny_fp32"])
    bad.variant = 7
    assert cuda_lib.ssd_workspace_size(ctypes.byref(bad), 1, ctypes.byref(n)) == 1
    assert cuda_lib.ssd_workspace_size(None, 1, ctypes.byref(n)) == 1


def test_pointer_validation_launches_nothing(cuda_lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("uses fake device addresses; host-only check")
    p = binding.problem(CONFIGS["mamba2_tiny_fp32"])
    fake = 1 << 20  # never dereferenced: validation rejects the call first
    # NULL required buffer
    st = cuda_lib.ssd_forward(ctypes.byref(p), None, fake, fake, fake, fake, None, fake, fake, fake, 1 << 30, None)
    assert st == 1
    # misaligned buffer
    st = cuda_lib.ssd_forward(ctypes.byref(p), fake + 4, fake, fake, fake, fake, None, fake, fake, fake, 1 << 30,
                              None)
    assert st == 4
    # workspace too small
    need = binding.ssd_workspace_size(p, False)
    st = cuda_lib.ssd_forward(ctypes.byref(p), fake, fake, fake, fake, fake, None, fake, fake, fake, need - 1, None)
    assert st == 5
    # MIMO requires A == NULL and dA == NULL
    pm = binding.problem(CONFIGS["mimo_r4_bf16"])
    st = cuda_lib.ssd_forward(ctypes.byref(pm), fake, fake, fake, fake, fake, None, fake, fake, fake, 1 << 40, None)
    assert st == 1
    need = binding.ssd_workspace_size(p, True)
    # prob, dy, ds_final, x, dt_raw, A, B, C, s0, dx, ddt_raw, dA, dB, dC, ds0, ws, ws_bytes, stream
    st = cuda_lib.ssd_backward(ctypes.byref(p), fake, None, fake, fake, fake, fake, fake, None,
                               fake, fake, fake, fake, fake, fake, fake, need, None)
    assert st == 1  # ds_final is required: it is the seed of the reverse recurrence
    st = cuda_lib.ssd_backward(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, None,
                               fake, fake, fake, fake, fake, fake, fake, need - 1, None)
    assert st == 5


def test_states_stash_validation(cuda_lib):
    """The stashed-states pair exists for the tensor-core problems only; its
    size is the bf16 chunk-state tensor; bad buffers fail on the host."""
    import torch
    tc = binding.problem(CONFIGS["mamba2_2p7b_bf16"])
    c = CONFIGS["mamba2_2p7b_bf16"]
    assert binding.ssd_states_size(tc) == (c["batch"] * c["nheads"] * (c["seqlen"] // c["chunk"]) * c["dstate"] *
                                           c["headdim"] * 2)
    n = ctypes.c_size_t(0)
    for name in ("mamba2_tiny_fp32", "mamba1_fp32", "mimo_r4_bf16"):
        p = binding.problem(CONFIGS[name])
        assert cuda_lib.ssd_states_size(ctypes.byref(p), ctypes.byref(n)) == 2  # SSD_ERR_SHAPE
    assert cuda_lib.ssd_states_size(ctypes.byref(tc), None) == 1
    if torch.cuda.is_available():
        return  # the rest uses fake device addresses
    fake = 1 << 20
    need_s = binding.ssd_states_size(tc)
    need_f = binding.ssd_workspace_size(tc, False)
    need_b = binding.ssd_workspace_size(tc, True)
    args = [fake] * 6 + [None, fake, fake]  # x, dt_raw, A, B, C, (s0), y, s_final
    st = cuda_lib.ssd_forward_stash(ctypes.byref(tc), *args[:5], None, fake, fake, None, need_s, fake, need_f, None)
    assert st == 1  # no states buffer
    st = cuda_lib.ssd_forward_stash(ctypes.byref(tc), *args[:5], None, fake, fake, fake, need_s - 1, fake, need_f,
                                    None)
    assert st == 5  # states buffer too small
    st = cuda_lib.ssd_forward_stash(ctypes.byref(tc), *args[:5], None, fake, fake, fake + 8, need_s, fake, need_f,
                                    None)
    assert st == 4  # misaligned states buffer
    # prob, dy, ds_final, x, dt_raw, A, B, C, states, states_bytes, dx, ddt_raw, dA, dB, dC, ds0, ws, ws_bytes, stream
    st = cuda_lib.ssd_backward_stashed(ctypes.byref(tc), fake, fake, fake, fake, fake, fake, fake, fake, need_s,
                                       fake, fake, fake, fake, fake, fake, fake, need_b - 1, None)
    assert st == 5
    st = cuda_lib.ssd_backward_stashed(ctypes.byref(tc), fake, fake, fake, fake, fake, fake, fake, None, need_s,
                                       fake, fake, fake, fake, fake, fake, fake, need_b, None)
    assert st == 1
    small = binding.problem(CONFIGS["mamba2_tiny_fp32"])
    st = cuda_lib.ssd_backward_stashed(ctypes.byref(small), fake, fake, fake, fake, fake, fake, fake, fake, need_s,
                                       fake, fake, fake, fake, fake, fake, fake, need_b, None)
    assert st == 2


def test_tail_chunk_sizes_the_workspace_by_ceil(cuda_lib):
    """T not a multiple of the chunk: the states of nc = ceil(T / L) chunks."""
    tc = CONFIGS["mamba2_2p7b_bf16"]
    full = binding.ssd_states_size(binding.problem(scaled(tc, seqlen=4096)))
    ragged = binding.ssd_states_size(binding.problem(scaled(tc, seqlen=4096 - 63)))
    assert ragged == full
    assert binding.ssd_states_size(binding.problem(scaled(tc, seqlen=4096 + 1))) == full * 65 // 64


def test_checkpoint_validation(cuda_lib):
    """The checkpoint pair exists for the tensor-core problems only; its size is
    b*H*ceil(nc/K)*P*N fp32 values; K < 1 and bad buffers fail on the host."""
    import torch
    c = CONFIGS["mamba2_2p7b_bf16"]
    tc = binding.problem(c)
    nc = c["seqlen"] // c["chunk"]
    for every in (1, 3, 8, 64, 1000):
        nk = -(-nc // every)
        assert binding.ssd_checkpoints_size(tc, every) == c["batch"] * c["nheads"] * nk * c["headdim"] * c["dstate"] * 4
    n = ctypes.c_size_t(0)
    assert cuda_lib.ssd_checkpoints_size(ctypes.byref(tc), 0, ctypes.byref(n)) == 1  # SSD_ERR_INVALID_ARG
    assert cuda_lib.ssd_checkpoints_size(ctypes.byref(tc), -2, ctypes.byref(n)) == 1
    assert cuda_lib.ssd_checkpoints_size(ctypes.byref(tc), (1 << 30) + 1, ctypes.byref(n)) == 1
    assert cuda_lib.ssd_checkpoints_size(ctypes.byref(tc), 8, None) == 1
    for name in ("mamba2_tiny_fp32", "mamba1_fp32", "mimo_r4_bf16"):
        p = binding.problem(CONFIGS[name])
        assert cuda_lib.ssd_checkpoints_size(ctypes.byref(p), 8, ctypes.byref(n)) == 2  # SSD_ERR_SHAPE
    if torch.cuda.is_available():
        return  # the rest uses fake device addresses
    fake = 1 << 20
    need_k = binding.ssd_checkpoints_size(tc, 8)
    need_f = binding.ssd_workspace_size(tc, False)
    need_b = binding.ssd_workspace_size(tc, True)
    fwd = cuda_lib.ssd_forward_checkpointed
    # prob, x, dt_raw, A, B, C, s0, y, s_final, every, ckpt, ckpt_bytes, ws, ws_bytes, stream
    assert fwd(ctypes.byref(tc), fake, fake, fake, fake, fake, None, fake, fake, 8, None, need_k, fake, need_f,
               None) == 1  # no checkpoint buffer
    assert fwd(ctypes.byref(tc), fake, fake, fake, fake, fake, None, fake, fake, 8, fake, need_k - 1, fake, need_f,
               None) == 5  # too small
    assert fwd(ctypes.byref(tc), fake, fake, fake, fake, fake, None, fake, fake, 8, fake + 8, need_k, fake, need_f,
               None) == 4  # misaligned
    assert fwd(ctypes.byref(tc), fake, fake, fake, fake, fake, None, fake, fake, 0, fake, need_k, fake, need_f,
               None) == 1  # K = 0
    bwd = cuda_lib.ssd_backward_checkpointed
    # prob, dy, ds_final, x, dt_raw, A, B, C, every, ckpt, ckpt_bytes, dx, ddt_raw, dA, dB, dC, ds0, ws, ws_bytes, stream
    assert bwd(ctypes.byref(tc), fake, fake, fake, fake, fake, fake, fake, 8, fake, need_k, fake, fake, fake, fake,
               fake, fake, fake, need_b - 1, None) == 5  # workspace too small
    assert bwd(ctypes.byref(tc), fake, fake, fake, fake, fake, fake, fake, 8, fake, need_k, fake, fake, fake, fake,
               fake, fake, None, need_b, None) == 1  # no workspace


def test_kda_validation(cuda_lib):
    """KDA sizes: the forward needs only the status word; the backward's workspace holds the checkpoints every
    8 steps, the CTAs' row sums and the per-value-head dq, dk (the replay scratch is in shared memory); bad sizes
    are refused on the host."""
    from selective_state_space_ssd_gb300.configs import KDA_CONFIGS
    c = KDA_CONFIGS["kda_fp32"]
    p = binding.kda_problem(c)
    assert binding.ssd_kda_workspace_size(p, False) == 256
    b, T, HV, K, V = c["batch"], c["seqlen"], c["value_heads"], c["key_dim"], c["value_dim"]
    need = binding.ssd_kda_workspace_size(p, True)
    nw = V // 4          # column warps of 4 value columns
    nsplit = nw // 8     # backward CTAs of eight column warps
    floats = (b * HV * (-(-T // 8)) * nw * 512             # lane-major checkpoints of every warp slice (K x 4)
              + b * T * HV * nsplit * (4 * K + 1)          # the CTAs' row sums
              + 2 * b * T * HV * K)                        # dq, dk per value head
    assert floats * 4 <= need <= floats * 4 + 256 * 6
    n = ctypes.c_size_t(0)
    for over, code in [(dict(key_dim=129), 2), (dict(value_dim=129), 2), (dict(value_heads=6, nheads=4), 2),
                       (dict(seqlen=0), 1), (dict(key_dim=0), 1)]:
        bad = binding.kda_problem(dict(c, **over))
        assert cuda_lib.ssd_kda_workspace_size(ctypes.byref(bad), 1, ctypes.byref(n)) == code, over
    assert cuda_lib.ssd_kda_workspace_size(ctypes.byref(p), 1, None) == 1
    fake = 1 << 20
    # prob, q, k, v, g, beta, s0, scale, o, s_final, ws, ws_bytes, stream: NULL q, misaligned o, small workspace
    assert cuda_lib.ssd_kda_forward(ctypes.byref(p), None, fake, fake, fake, fake, None, 0.1, fake, fake, fake, 256,
                                    None) == 1
    assert cuda_lib.ssd_kda_forward(ctypes.byref(p), fake, fake, fake, fake, fake, None, 0.1, fake + 4, fake, fake,
                                    256, None) == 4
    assert cuda_lib.ssd_kda_forward(ctypes.byref(p), fake, fake, fake, fake, fake, None, 0.1, fake, fake, fake, 255,
                                    None) == 5
    args = [fake] * 7 + [None]  # do, ds_final, q, k, v, g, beta, (s0)
    assert cuda_lib.ssd_kda_backward(ctypes.byref(p), *args, 0.1, *([fake] * 6), fake, need - 1, None) == 5
