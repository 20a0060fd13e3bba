"""Build libfp8bs.so in-tree with nvcc for sm_103a.

Run ``python -m fp8_fine_grained_23_b300.build`` (or call :func:`build`). The library links the
CUDA runtime statically and has no PyTorch dependency; it is placed next to this file so that
it travels with the source tree. Division and subnormal handling stay IEEE (no fast-math,
``-prec-div=true``, ``-ftz=false``), which the bit-exact quantizer contract depends on.
"""
from __future__ import annotations

import glob
import os
import re
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libfp8bs.so")
# Debug build with a serialised pipeline (GEMMs: one operand stage, one scale slot, one TMEM
# accumulator): every role waits for the previous one at every step, so a missing or misplaced
# barrier shows up as a different result or a timeout. Tests only.
SERIAL_LIB_PATH = os.path.join(PKG, "libfp8bs_serial.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(d) > t for d in deps)


# The GEMM kernels split registers between warpgroups with setmaxnreg; the split adds up to
# exactly 168 registers per thread at launch (384 threads), so the build insists on that count.
GEMM_LAUNCH_REGS = 168


def resource_report(ptxas_log: str) -> dict[str, dict[str, int]]:
    """Per-kernel registers / spill bytes parsed from ``-Xptxas -v`` output."""
    out: dict[str, dict[str, int]] = {}
    name = None
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            name = m.group(1)
            out[name] = {}
            continue
        if name is None:
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            out[name]["spill_stores"] = int(m.group(1))
            out[name]["spill_loads"] = int(m.group(2))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            out[name]["registers"] = int(m.group(1))
    return out


def build(force: bool = False, verbose_ptxas: bool = False, serial: bool = False) -> str:
    path = SERIAL_LIB_PATH if serial else LIB_PATH
    if not force and not _stale(path):
        return path
    tmp = path + f".tmp{os.getpid()}"
    cmd = [_nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-prec-div=true", "-prec-sqrt=true",
           "-ftz=false", "-Xptxas=-v", "-Xcompiler", "-fPIC,-O2,-Wall", "-shared", "-cudart",
           "static", *(["-DFP8BS_SERIAL_PIPELINE"] if serial else []), "-I", INCLUDE, "-I", CSRC,
           *sources(), "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("nvcc failed building libfp8bs.so")
    report = resource_report(res.stdout + res.stderr)
    for name, r in report.items():
        if "gemm_kernel" in name and r.get("registers") != GEMM_LAUNCH_REGS:
            os.remove(tmp)
            raise RuntimeError(f"{name}: {r.get('registers')} registers at launch, the "
                               f"setmaxnreg split needs exactly {GEMM_LAUNCH_REGS}")
    if verbose_ptxas:
        for name, r in report.items():
            print(f"{name}: {r}")
    os.replace(tmp, path)
    return path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                serial="--serial" in sys.argv))
