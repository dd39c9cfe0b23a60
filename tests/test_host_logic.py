"""Host-side logic that needs no GPU: the seeded input generators' options and
the benchmark's argument defaults."""
import json
import os
import subprocess
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


def test_stack_flops_count_the_nine_products_of_a_layer():
    import bench

    B, L, H, P, nl = 32, 1024, 512, 256, 6
    T = B * L
    # (M, N, K) of every product one layer issues (s5_ssm_forward_states,
    # s5_gate_residual, s5_gate_backward, s5_ssm_backward)
    products = [(T, 2 * P, H),   # Bu = z B_bar^T
                (T, H, 2 * P),   # y = X C'^T
                (T, H, H),       # a = h W^T
                (T, H, H),       # W^T act
                (H, H, T),       # dW = act^T h
                (T, 2 * P, H),   # x_hat = ybar C'
                (T, H, 2 * P),   # Re(B_bar^H s)
                (2 * P, H, T),   # dB_bar = S^T z
                (H, 2 * P, T)]   # G = ybar^T X (dC~)
    assert bench.stack_flops(B, L, H, P, nl) == nl * sum(2 * m * n * k for m, n, k in products)
    assert bench.stack_flops(B, L, H, P, nl) == 927712935936
    # a shape with 2P != H keeps the two kinds apart
    assert bench.stack_flops(2, 77, 64, 48, 1) == 2 * 154 * (6 * 64 * 96 + 3 * 64 * 64)


def test_reference_arm_prints_one_contract_line():
    # the float64 oracle on the host: no GPU is involved
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "small", "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] == d["cpu_baseline"]["value"] == d["e2e"]["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    # one sequence of the workload per step, timed as tokens per second
    w = WORKLOADS["small"]
    assert abs(d["value"] - w.L / (d["ms_per_step"] / 1e3)) <= 1e-6 * d["value"]


class _DoneProcess:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_sampler_takes_the_median_and_the_throttle_reasons():
    import bench

    s = bench.ClockSampler(None)
    s.proc = _DoneProcess()
    # index, sm, max sm, power, active, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    s.out.write("0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active\n"
                "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                "0, [N/A], 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    c = s.stop()
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    s = bench.ClockSampler(None)
    s.proc = _DoneProcess()
    s.out.write("0, 1500, 2070, 700.0, 0x48, Active, Not Active, Active, Not Active\n")
    assert s.stop()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_traffic_is_reported_only_for_the_captured_source_and_workload(tmp_path, monkeypatch):
    import hashlib

    import bench

    src = tmp_path / "kernel.cu"
    src.write_text("// kernel source\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(
        {"k": {"workload": "pathx_bf16 (B=8 ...)", "source_sha256": sha, "dram_bytes_per_launch": 1234}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("k", str(src), "pathx_bf16") == 1234.0
    assert bench.traffic_for("k", str(src), "fp32") is None          # another workload
    assert bench.traffic_for("other", str(src), "pathx_bf16") is None
    src.write_text("// kernel source, edited\n")                     # changed since the capture
    assert bench.traffic_for("k", str(src), "pathx_bf16") is None



# --------------------------------------------------------------------------
# The float-float constants of the discretisation kernel (csrc/s5_ff.cuh):
# 1/n! pairs and the three-part splits of ln 2 and pi/2, checked against the
# exact rationals (pi from Machin's formula, ln 2 from sum 1/(k 2^k)).
# --------------------------------------------------------------------------
def _ff_header():
    path = os.path.join(ROOT, "diagonal_state_space_gb300", "csrc", "s5_ff.cuh")
    return open(path).read()


def _hexf(tok):
    tok = tok.rstrip("f")
    return float.fromhex(tok) if "x" in tok else float(tok)


def test_ff_inverse_factorials_are_exact_to_float_float():
    import math
    import re
    from fractions import Fraction

    src = _ff_header()
    pairs = re.findall(r"case (\d+): return \{([-0-9a-fx.p+]+)f?, ([-0-9a-fx.p+]+)f?\};", src)
    assert len(pairs) == 17
    for n, hi, lo in pairs:
        exact = Fraction(1, math.factorial(int(n)))
        hi, lo = Fraction(_hexf(hi)), Fraction(_hexf(lo))
        # hi is the nearest float; hi + lo within 2^-48 of 1/n! (relative)
        assert abs(hi - exact) <= exact * Fraction(1, 2 ** 24)
        assert abs(hi + lo - exact) <= exact * Fraction(1, 2 ** 48)


def test_ff_cody_waite_splits():
    import re
    from decimal import Decimal, getcontext
    from fractions import Fraction

    getcontext().prec = 60

    def atan_inv(n):
        x, s, k = Decimal(1) / n, Decimal(0), 0
        t = x
        while abs(t) > Decimal(10) ** -58:
            s += (t / (2 * k + 1)) * (1 if k % 2 == 0 else -1)
            t *= x * x
            k += 1
        return s

    pi = 16 * atan_inv(5) - 4 * atan_inv(239)
    ln2 = sum(Decimal(1) / (k * Decimal(2) ** k) for k in range(1, 200))
    src = _ff_header()

    def consts(name):
        m = re.search(name + r"_1 = ([-0-9a-fx.p+]+)f, " + name + r"_2 = ([-0-9a-fx.p+]+)f, "
                      + name + r"_3 = ([-0-9a-fx.p+]+)f;", src)
        return [Fraction(_hexf(t)) for t in m.groups()]

    for name, exact in (("LN2", Fraction(ln2)), ("PIO2", Fraction(pi / 2))):
        c1, c2, c3 = consts(name)
        assert abs(c1 + c2 + c3 - exact) <= exact * Fraction(1, 2 ** 64)
        # the first part has at most 12 significant bits
        m, e = c1.numerator, c1.denominator
        assert e & (e - 1) == 0 and m < 2 ** 12
