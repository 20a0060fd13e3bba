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
