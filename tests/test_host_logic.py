"""Host-side logic that needs no GPU: the seeded input generators' options and
the benchmark's argument defaults."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from diagonal_state_space_gb300.workloads import WORKLOADS, make_inputs, make_layer_inputs  # noqa: E402


def test_bidirectional_inputs_extend_the_causal_ones():
    a = make_layer_inputs(2, 10, 8, 4, seed=5)
    b = make_layer_inputs(2, 10, 8, 4, seed=5, bidirectional=True)
    for k in ("u", "lambda_", "log_dt", "b_tilde", "c_tilde", "d"):
        assert np.array_equal(a[k], b[k])            # the same draws, in the same order
    c2 = b["c_tilde2"]
    assert c2.shape == (8, 8) and c2.dtype == np.complex64 and c2.flags.c_contiguous
    assert np.array_equal(c2[:, :4], b["c_tilde"])
    assert not np.array_equal(c2[:, 4:], b["c_tilde"])   # the backward half is its own draw
    # same distribution as C~: real and imaginary parts ~ N(0, 1/(2H))
    big = make_layer_inputs(1, 1, 256, 256, seed=1, bidirectional=True)["c_tilde2"][:, 256:]
    assert abs(np.std(big.real) - np.sqrt(1 / 512)) < 0.002
    assert abs(np.std(big.imag) - np.sqrt(1 / 512)) < 0.002


def test_generators_are_deterministic_per_seed():
    a = make_layer_inputs(3, 17, 8, 6, seed=11, varying_dt=True, bidirectional=True)
    b = make_layer_inputs(3, 17, 8, 6, seed=11, varying_dt=True, bidirectional=True)
    for k in a:
        assert np.array_equal(a[k], b[k])


def test_next_row_workloads_are_declared():
    assert WORKLOADS["pathx_bf16_bidir"].bidirectional
    w = WORKLOADS["pathx_bf16_bilinear"]
    assert (w.method, w.clip_re, w.dt_scale) == ("bilinear", -1e-4, 0.5)
    s = WORKLOADS["stream"]
    assert s.streaming and s.u_dtype == "f32"
    inp = make_inputs(s)
    assert inp["u"].shape == (s.B, s.L, s.H)


def test_bench_defaults_per_workload(monkeypatch):
    import bench

    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert (a.workload, a.steps, a.warmup, a.e2e_steps, a.gpus, a.impl) == ("pathx_bf16", 2000, 50, 30, 1,
                                                                         "ours")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "stream"])
    a = bench.parse()
    assert (a.steps, a.warmup, a.e2e_steps) == (20, 3, 3)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "stream", "--steps", "7"])
    assert bench.parse().steps == 7


def test_algorithmic_bytes_of_the_long_sequence_workload():
    import bench

    w = WORKLOADS["pathx_bf16"]
    # u and y in bf16 plus lambda_bar, B_bar, C~ (complex fp32) and D
    expect = 8 * 16384 * 128 * 4 + 8 * 128 + 2 * 8 * 128 * 128 + 4 * 128
    assert bench.algorithmic_bytes(w, 2, 2) == expect == 67372544
    wb = WORKLOADS["pathx_bf16_bidir"]
    assert bench.algorithmic_bytes(wb, 2, 2) == expect + 8 * 128 * 128
