"""Host logic of bench.py that needs no GPU: the clock record keeps only the
samples taken inside the timed region, the tensor-core denominator follows the
length of the timed region, and the summary flags fractions above one."""
import importlib.util
import os
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _row(t, sm, reasons=("Not Active",) * 4):
    stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(int(t))) + f".{int(round((t % 1) * 1000)):03d}"
    return ", ".join([stamp, "0", str(sm), "2070", "900.0", "0x0", *reasons])


def test_clock_record_keeps_timed_region_samples(tmp_path):
    b = _bench()
    c = b.Clocks(0)
    base = int(time.time()) + 0.0
    rows = [_row(base + 0.00, 2070), _row(base + 0.10, 1500, ("Not Active", "Not Active", "Not Active", "Active")),
            _row(base + 0.12, 1600, ("Not Active", "Not Active", "Not Active", "Active")),
            _row(base + 0.14, 1700), _row(base + 0.50, 2070)]
    f = open(tmp_path / "clk.csv", "w+")
    f.write("\n".join(rows) + "\n")
    c.f, c.proc = f, _FakeProc()
    c.t0, c.t1 = base + 0.095, base + 0.145
    out = c.stop()
    assert out["samples_in_timed_region"] == 3
    assert out["sm_mhz"] == 1600.0
    assert out["reasons"] == ["sw_power_cap"]


def test_tensor_peak_follows_region_length():
    b = _bench()
    pk = {"bf16_tflops": 1925.9, "bf16_tflops_sustained": 1745.7, "hbm_gbs": 6667.9, "src": "measured"}
    assert b.pick_tensor_peak(pk, 82.0)[0] == 1925.9
    assert b.pick_tensor_peak(pk, 950.0)[0] == 1745.7
    # a long region whose clock record shows the board at its power cap: sustained
    assert b.pick_tensor_peak(pk, 950.0, {"sm_mhz": 1650.0, "sm_max_mhz": 2070.0})[0] == 1745.7
    # a long region at full clock (waiting on a slow host link, not power-capped): burst
    assert b.pick_tensor_peak(pk, 950.0, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})[0] == 1925.9
    assert b.pick_tensor_peak(pk, 950.0, {"sm_mhz": None, "sm_max_mhz": None})[0] == 1745.7


def test_summary_flags_fraction_above_one():
    b = _bench()
    pk = {"bf16_tflops": 1000.0, "bf16_tflops_sustained": 900.0, "hbm_gbs": 1000.0, "src": "measured"}
    prof = {"gemm.a": {"launches": 2, "ms": 2.0, "flops": 2.2e12, "bytes": 0.0},      # 1100 TFLOP/s
            "norm": {"launches": 1, "ms": 1.0, "flops": 0.0, "bytes": 0.5e9}}          # 500 GB/s
    r = {"units": 100, "ms": 10.0, "ms_e2e": 11.0, "ms_prof": 10.0, "prof": prof, "config": {}, "launches": 3,
         "clocks": {}, "h2d": 0, "d2h": 0, "extra": None}
    out = b.summarize(r, "layer", 1, 1, pk)
    assert out["kernels_frac_above_1"] == ["gemm.a"]
    assert out["roofline"]["kernel"] == "gemm_bf16_tc" and out["roofline"]["frac"] == 1.1
    assert out["kernels"]["norm"]["frac"] == 0.5
    assert abs(out["value"] - 10000.0) < 1e-9
