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
