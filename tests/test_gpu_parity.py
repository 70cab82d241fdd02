"""Parity of the CUDA library (called through its C ABI) with the float64
oracle on the same seeded inputs, element by element, for every output.

Small cases span several chunks and ragged sizes (head/state widths that are
not multiples of any tile, odd head counts, several groups); the full-size
cases run the five workloads exactly as the benchmark launches them.
"""
import numpy as np
import pytest
import torch

from selective_state_space_ssd_gb300 import binding
from selective_state_space_ssd_gb300 import inputs as synth
from selective_state_space_ssd_gb300.configs import CONFIGS, scaled

import oracle
from parity import TOL, compare, rel_err, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

M2_BF16 = CONFIGS["mamba2_130m_bf16"]
MIMO = CONFIGS["mimo_r4_bf16"]
M1 = CONFIGS["mamba1_fp32"]

SMALL = {
    "tiny_fp32": CONFIGS["mamba2_tiny_fp32"],
    "m2_fp32_ragged_groups": dict(variant="mamba2", dtype="f32", batch=2, seqlen=96, nheads=6, headdim=5, dstate=7,
                                  ngroups=3, chunk=32, mimo_rank=1),
    "m2_bf16_tiles": scaled(M2_BF16, batch=2, seqlen=256, nheads=4, ngroups=2),
    "m2_bf16_ragged": scaled(M2_BF16, batch=1, seqlen=192, nheads=3, headdim=24, dstate=40, ngroups=1),
    "m2_bf16_single_chunk": scaled(M2_BF16, batch=1, seqlen=64, nheads=2),
    # tensor-core kernels' item ranges: one head per group (every head is a run of its own), and more
    # (chunk, head) items than SMs with five heads per group (short runs, chunks split over CTAs)
    "m2_bf16_head_per_group": scaled(M2_BF16, batch=2, seqlen=256, nheads=4, ngroups=4),
    "m2_bf16_split_runs": scaled(M2_BF16, batch=4, seqlen=512, nheads=10, ngroups=2),
    "m1_small": scaled(M1, batch=2, seqlen=256, nheads=40),
    "m1_ragged": scaled(M1, batch=1, seqlen=96, nheads=37, dstate=5, chunk=32),
    "mimo_bf16_tiles": scaled(MIMO, batch=1, seqlen=256, nheads=3, ngroups=3),
    "mimo_ragged": scaled(MIMO, batch=2, seqlen=48, nheads=2, ngroups=2, headdim=20, dstate=24, chunk=16,
                          mimo_rank=3),
    "mimo_fp32": scaled(MIMO, dtype="f32", batch=1, seqlen=128, nheads=2, ngroups=2, headdim=16, dstate=32,
                        chunk=32),
    # a tail chunk (T not a multiple of the chunk length): tensor-core path with tails of 17 and 63 steps and
    # a sequence shorter than one chunk; the CUDA-core paths of every variant
    "m2_bf16_tail": scaled(M2_BF16, batch=2, seqlen=3 * 64 + 17, nheads=4, ngroups=2),
    "m2_bf16_tail63": scaled(M2_BF16, batch=3, seqlen=127, nheads=3),
    "m2_bf16_short": scaled(M2_BF16, batch=3, seqlen=40, nheads=2),
    "m2_fp32_tail": dict(variant="mamba2", dtype="f32", batch=2, seqlen=100, nheads=6, headdim=5, dstate=7,
                         ngroups=3, chunk=32, mimo_rank=1),
    "m1_tail": scaled(M1, batch=2, seqlen=100, nheads=40, chunk=32),
    # Mamba-1 lane layouts: 16 threads a channel (N = 32), 2 (N = 3) and 1 (N = 2)
    "m1_n32": scaled(M1, batch=1, seqlen=72, nheads=13, dstate=32),
    "m1_n3": scaled(M1, batch=2, seqlen=40, nheads=70, dstate=3),
    "m1_n2": scaled(M1, batch=1, seqlen=33, nheads=150, dstate=2),
    "mimo_tail": scaled(MIMO, batch=2, seqlen=50, nheads=2, ngroups=2, headdim=20, dstate=24, chunk=16,
                        mimo_rank=3),
    # MIMO on the tensor-core kernels (the fused sequence of T * R positions in chunks of 64): rank 4 with a
    # tail (200 = 3 * 64 + 8 positions), ranks 2 and 1
    "mimo_tc_tail": scaled(MIMO, batch=2, seqlen=50, nheads=3, ngroups=3),
    "mimo_tc_r2": scaled(MIMO, batch=1, seqlen=96, nheads=2, ngroups=2, mimo_rank=2),
    "mimo_tc_r1": scaled(MIMO, batch=2, seqlen=80, nheads=2, ngroups=2, mimo_rank=1),
    # the degenerate sequence of one step: a single chunk with 63 (tensor-core) or chunk - 1 empty steps
    "tiny_fp32_one_step": dict(CONFIGS["mamba2_tiny_fp32"], seqlen=1),
    "m2_bf16_one_step": scaled(M2_BF16, batch=2, seqlen=1, nheads=3),
    "m1_one_step": scaled(M1, batch=1, seqlen=1, nheads=40),
    "mimo_tc_one_step": scaled(MIMO, batch=1, seqlen=1, nheads=2, ngroups=2),
}


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return cuda_lib


@pytest.mark.parametrize("name", sorted(SMALL))
def test_parity_small(name):
    cfg = SMALL[name]
    cpu = synth.make_inputs(cfg, seed=1)
    gpu = run_gpu(cfg, to_device(cpu))
    compare(cfg, gpu, run_oracle(cfg, cpu))


@pytest.mark.parametrize("name", ["tiny_fp32", "m2_bf16_tiles", "m1_small", "mimo_bf16_tiles"])
def test_null_s0_equals_zero_state(name):
    cfg = SMALL[name]
    cpu = synth.make_inputs(cfg, seed=2, zero_s0=True)
    dev = to_device(cpu)
    a = run_gpu(cfg, dev, s0_null=True)
    b = run_gpu(cfg, dev, s0_null=False)
    for k in a:
        if a[k] is not None:
            assert torch.equal(a[k], b[k]), k
    compare(cfg, a, run_oracle(cfg, cpu))


@pytest.mark.parametrize("name", ["tiny_fp32", "m2_bf16_tiles", "m1_small", "mimo_bf16_tiles", "m2_bf16_tail",
                                  "mimo_tc_tail"])
def test_backward_is_bitwise_deterministic(name):
    cfg = SMALL[name]
    dev = to_device(synth.make_inputs(cfg, seed=3))
    a = run_gpu(cfg, dev)
    b = run_gpu(cfg, dev)
    for k in a:
        if a[k] is not None:
            assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("name", ["m2_bf16_tiles", "m2_bf16_split_runs", "m2_bf16_tail", "full_2p7b"])
def test_stashed_states_give_the_recompute_bits(name):
    """ssd_forward_stash returns ssd_forward's bits and a chunk-state stash;
    ssd_backward_stashed from that stash returns ssd_backward's bits (which the
    other tests hold to the oracle), with and without s0."""
    cfg = CONFIGS["mamba2_2p7b_bf16"] if name == "full_2p7b" else SMALL[name]
    for zero_s0 in (False, True):
        dev = to_device(synth.make_inputs(cfg, seed=6, zero_s0=zero_s0))
        s0 = None if zero_s0 else dev["s0"]
        y, sf = binding.forward(cfg, dev["x"], dev["dt_raw"], dev["A"], dev["B"], dev["C"], s0)
        y2, sf2, states = binding.forward_stash(cfg, dev["x"], dev["dt_raw"], dev["A"], dev["B"], dev["C"], s0)
        g = binding.backward(cfg, dev["dy"], dev["ds_final"], dev["x"], dev["dt_raw"], dev["A"], dev["B"], dev["C"],
                             s0)
        g2 = binding.backward_stashed(cfg, dev["dy"], dev["ds_final"], dev["x"], dev["dt_raw"], dev["A"], dev["B"],
                                      dev["C"], states)
        torch.cuda.synchronize()
        assert torch.equal(y, y2) and torch.equal(sf, sf2)
        for k in g:
            assert torch.equal(g[k], g2[k]), k
        # the stash's first tile of every (batch, head) is s0 in bf16, laid out [N][P]
        nc = -(-cfg["seqlen"] // cfg["chunk"])
        st = states.view(torch.bfloat16).view(cfg["batch"], cfg["nheads"], nc, cfg["dstate"], cfg["headdim"])
        want = torch.zeros_like(st[:, :, 0]) if zero_s0 else dev["s0"].transpose(-1, -2).to(torch.bfloat16)
        assert torch.equal(st[:, :, 0], want)


@pytest.mark.parametrize("name,every", [("m2_bf16_tiles", 1), ("m2_bf16_tiles", 2), ("m2_bf16_split_runs", 3),
                                        ("m2_bf16_tail", 2), ("m2_bf16_tail", 64), ("full_2p7b", 8)])
def test_checkpointed_backward_gives_the_recompute_bits(name, every):
    """ssd_forward_checkpointed returns ssd_forward's bits plus fp32 checkpoints
    every K chunks; ssd_backward_checkpointed, which replays the chunk states in
    segments of K chunks from them, returns ssd_backward's bits (which the other
    tests hold to the oracle), with and without s0, for K = 1, several K that
    leave a short last segment, and K >= the chunk count (s0 only)."""
    cfg = CONFIGS["mamba2_2p7b_bf16"] if name == "full_2p7b" else SMALL[name]
    for zero_s0 in (False, True):
        dev = to_device(synth.make_inputs(cfg, seed=7, zero_s0=zero_s0))
        s0 = None if zero_s0 else dev["s0"]
        y, sf = binding.forward(cfg, dev["x"], dev["dt_raw"], dev["A"], dev["B"], dev["C"], s0)
        y2, sf2, ck = binding.forward_checkpointed(cfg, dev["x"], dev["dt_raw"], dev["A"], dev["B"], dev["C"], s0,
                                                   every=every)
        g = binding.backward(cfg, dev["dy"], dev["ds_final"], dev["x"], dev["dt_raw"], dev["A"], dev["B"], dev["C"],
                             s0)
        g2 = binding.backward_checkpointed(cfg, dev["dy"], dev["ds_final"], dev["x"], dev["dt_raw"], dev["A"],
                                           dev["B"], dev["C"], ck, every=every)
        torch.cuda.synchronize()
        assert torch.equal(y, y2) and torch.equal(sf, sf2)
        for k in g:
            assert torch.equal(g[k], g2[k]), k
        # entry 0 of every (batch, head) is s0 itself (fp32, [P][N]), or zeros
        want = torch.zeros_like(ck[:, :, 0]) if zero_s0 else dev["s0"]
        assert torch.equal(ck[:, :, 0], want)


def test_checkpoints_are_the_states_at_the_chunk_boundaries():
    """Entry k of the checkpoints is the state entering chunk k*K: the oracle's
    s_final of the sequence cut after k*K chunks, within the bf16 tolerance."""
    cfg = SMALL["m2_bf16_split_runs"]
    every = 2
    cpu = synth.make_inputs(cfg, seed=8)
    dev = to_device(cpu)
    _, _, ck = binding.forward_checkpointed(cfg, dev["x"], dev["dt_raw"], dev["A"], dev["B"], dev["C"], dev["s0"],
                                            every=every)
    torch.cuda.synchronize()
    L = cfg["chunk"]
    nc = -(-cfg["seqlen"] // L)
    assert ck.shape[2] == -(-nc // every) >= 2
    f64 = synth.as_float64(cpu)
    for k in range(1, ck.shape[2]):
        T1 = k * every * L
        cut = dict(f64, x=f64["x"][:, :T1], dt_raw=f64["dt_raw"][:, :T1], B=f64["B"][:, :T1], C=f64["C"][:, :T1])
        ref = oracle.forward("mamba2", cut)["s_final"]
        assert rel_err(ck[:, :, k], ref) <= TOL[cfg["dtype"]], k


def test_zero_seed_and_zero_dy():
    """dy = 0 leaves only the decayed seed: ds0 = exp(sum da) ds_final, dC = 0."""
    cfg = SMALL["m2_bf16_tiles"]
    cpu = synth.make_inputs(cfg, seed=4)
    cpu["dy"] = torch.zeros_like(cpu["dy"])
    gpu = run_gpu(cfg, to_device(cpu))
    assert torch.count_nonzero(gpu["dC"]) == 0
    compare(cfg, gpu, run_oracle(cfg, cpu))


@pytest.mark.parametrize("T0", [128, 100])
def test_chaining_two_calls_equals_one(T0):
    """Splitting T and chaining s_final -> s0 (forward) and ds0 -> ds_final
    (backward) reproduces one call: at a chunk boundary, and at T0 = 100,
    where both pieces end in a tail chunk (100 = 64 + 36, 156 = 2 * 64 + 28)."""
    cfg = SMALL["m2_bf16_tiles"]
    cpu = synth.make_inputs(cfg, seed=5)
    dev = to_device(cpu)
    half = scaled(cfg, seqlen=T0)
    rest = scaled(cfg, seqlen=cfg["seqlen"] - T0)

    def cut(t, lo, hi):
        return t[:, lo:hi].contiguous()

    first = {k: (v if k in ("A", "s0", "ds_final") else cut(v, 0, T0)) for k, v in dev.items()}
    second = {k: (v if k in ("A", "s0", "ds_final") else cut(v, T0, cfg["seqlen"])) for k, v in dev.items()}
    y1, s1 = binding.forward(half, first["x"], first["dt_raw"], first["A"], first["B"], first["C"], first["s0"])
    y2, s2 = binding.forward(rest, second["x"], second["dt_raw"], second["A"], second["B"], second["C"], s1)
    g2 = binding.backward(rest, second["dy"], second["ds_final"], second["x"], second["dt_raw"], second["A"],
                          second["B"], second["C"], s1)
    g1 = binding.backward(half, first["dy"], g2["ds0"], first["x"], first["dt_raw"], first["A"], first["B"],
                          first["C"], first["s0"])
    torch.cuda.synchronize()
    chained = {"y": torch.cat([y1, y2], 1), "s_final": s2, "dx": torch.cat([g1["dx"], g2["dx"]], 1),
               "ddt_raw": torch.cat([g1["ddt_raw"], g2["ddt_raw"]], 1), "dA": g1["dA"] + g2["dA"],
               "dB": torch.cat([g1["dB"], g2["dB"]], 1), "dC": torch.cat([g1["dC"], g2["dC"]], 1),
               "ds0": g1["ds0"]}
    compare(cfg, chained, run_oracle(cfg, cpu))


def _inner(a, b):
    return float((a.double() * b.double()).sum())


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_full_size_parity(name):
    """The workloads at their full sizes, in the configuration the benchmark
    launches, against the oracle on every output.  MIMO compares batch 0 (its
    sequences are independent and nothing is reduced across them); the others
    run the whole oracle."""
    cfg = CONFIGS[name]
    cpu = synth.make_inputs(cfg, seed=0)
    gpu = run_gpu(cfg, to_device(cpu))
    if cfg["variant"] == "mimo":
        one = scaled(cfg, batch=1)
        ref = run_oracle(one, {k: (None if v is None else v[:1]) for k, v in cpu.items()})
        gpu = {k: (None if v is None else v[:1]) for k, v in gpu.items()}
        compare(one, gpu, ref)
    else:
        compare(cfg, gpu, run_oracle(cfg, cpu))
    # homogeneity identities hold for any correct VJP at any size
    dev = to_device(cpu)
    lhs = _inner(dev["dy"], gpu["y"]) if cfg["variant"] != "mimo" else None
    if lhs is not None:
        scale = float((dev["dy"].double().abs() * gpu["y"].double().abs()).sum())
        assert abs(lhs - _inner(gpu["dC"], dev["C"])) < 3e-2 * scale


def test_full_size_tail_chunk():
    """The 2.7B layer shape with T = 4063 (63 full chunks and a tail of 31
    steps) on the tensor-core path, against the oracle on every output."""
    cfg = scaled(CONFIGS["mamba2_2p7b_bf16"], seqlen=4063)
    cpu = synth.make_inputs(cfg, seed=0)
    compare(cfg, run_gpu(cfg, to_device(cpu)), run_oracle(cfg, cpu))
