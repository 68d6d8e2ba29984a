"""Host logic of the library's per-device caches (no GPU needed).

CUDA function attributes, occupancy answers and symbol addresses belong to a
device, so libdv keeps them in a table keyed by the device id
(csrc/per_device.h).  The C++ check below is compiled with the host compiler
and run: every device id computes its own value once, and ids outside the
table are never cached."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "contextual_sparsity_decode_gb300", "csrc")


def test_cache_is_keyed_by_device_id(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "per_device_test"
    src = os.path.join(ROOT, "tests", "host_cc", "per_device_test.cc")
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, src, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"


def test_every_cached_attribute_uses_the_per_device_table():
    """No CUDA source keeps a device attribute, an occupancy answer or a
    device property in a process-wide variable."""
    import re
    device_calls = re.compile(r"cudaFuncSetAttribute|cudaOccupancy|cudaDeviceGetAttribute|cudaGetSymbolAddress")
    for name in sorted(os.listdir(CSRC)):
        if not name.endswith((".cu", ".cuh")):
            continue
        src = open(os.path.join(CSRC, name)).read()
        for m in re.finditer(r"static\s+(?:const\s+)?(bool|int)\s+\w+[^;]*", src):
            stmt_end = src.find(";", m.end())
            window = src[m.start(): src.find("\n", stmt_end) + 1 if stmt_end >= 0 else len(src)]
            following = "\n".join(src[m.end():].splitlines()[:6])
            if device_calls.search(window) or device_calls.search(following):
                line = src[: m.start()].count("\n") + 1
                pytest.fail(f"{name}:{line}: process-wide cache '{m.group(0)[:60]}'")
