"""bench.py's extra workload sections: every name a section calls exists in the module, so that
the default run (all sections) cannot fail on a missing function after a refactor."""
import builtins
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_every_section_resolves():
    bench = _bench()
    assert bench.SECTIONS, "no sections"
    for name, fn in bench.SECTIONS.items():
        assert callable(fn), name
        for ref in fn.__code__.co_names:
            # attribute names of the arguments (F.fp8_..., torch....) are not module globals
            if ref in fn.__code__.co_varnames:
                continue
            if fn.__name__ == "<lambda>":
                assert hasattr(bench, ref) or hasattr(builtins, ref), f"{name}: {ref} undefined"


class _DoneProcess:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        pass


def _sampler_from_rows(bench, rows, memory):
    import tempfile
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.memory = memory
    cs.n_fields = 10 if memory else 8
    cs.proc = _DoneProcess()
    fd, cs.path = tempfile.mkstemp()
    os.close(fd)
    with open(cs.path, "w") as f:
        f.write("".join(r + "\n" for r in rows))
    return cs.stop()


def test_clock_sampler_summary():
    """The clocks summary of the JSON line: median SM clock, max power, the throttle reasons
    seen Active, and (extras) the memory clock and HBM temperature; N/A becomes null."""
    bench = _bench()
    rows = ["1590, 2032, 1088.2, 0x4, Not Active, Not Active, Not Active, Active",
            "1610, 2032, 1001.0, 0x4, Not Active, Not Active, Not Active, Active",
            "1600, 2032, 1050.5, 0x0, Not Active, Active, Not Active, Not Active",
            "garbage line"]
    out = _sampler_from_rows(bench, rows, memory=False)
    assert out == {"sm_mhz": 1600.0, "sm_max_mhz": 2032.0, "power_w_max": 1088.2, "samples": 3,
                   "reasons": ["hw_thermal_slowdown", "sw_power_cap"]}
    rows = [r + ", 3996, N/A" for r in rows[:3]]
    out = _sampler_from_rows(bench, rows, memory=True)
    assert out["mem_mhz_min"] == 3996.0 and out["hbm_temp_c_max"] is None
    import json
    assert "NaN" not in json.dumps(out)
    assert _sampler_from_rows(bench, [], memory=True) is None


def test_fp8_peak_follows_sampled_clocks():
    """The step's GEMM is compared with the burst peak unless the timed region's clocks show the
    power-capped state the sustained figure was measured in."""
    bench = _bench()
    peaks = {"hbm_gbs": 6425.0, "bf16_tflops": 1808.6, "bf16_tflops_sustained": 1390.4,
             "sustained_sm_mhz": 1192.0}
    full = {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []}
    peak, burst, note = bench.choose_fp8_peak(peaks, full)
    assert peak == burst == 2 * 1808.6 and "burst" in note
    assert bench.choose_fp8_peak(peaks, None)[0] == 2 * 1808.6
    # power cap at a clock well above the one the sustained figure was taken at: still burst
    warm = {"sm_mhz": 1560.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"]}
    assert bench.choose_fp8_peak(peaks, warm)[0] == 2 * 1808.6
    capped = {"sm_mhz": 1200.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"]}
    peak, burst, note = bench.choose_fp8_peak(peaks, capped)
    assert peak == 2 * 1390.4 and burst == 2 * 1808.6 and "sustained" in note
    # no recorded clock for the sustained figure: burst
    assert bench.choose_fp8_peak(dict(peaks, sustained_sm_mhz=None), capped)[0] == 2 * 1808.6
