"""Host sanitizer runs (no GPU): the CPU oracle and the C ABI's host-side paths
built with AddressSanitizer and UndefinedBehaviorSanitizer, each driven by a
small C++ program under tests/sanitize/ that calls every function on valid and
invalid inputs.  A sanitizer report or a failed contract check fails the test."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SAN = ["-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=all",
       "-fno-omit-frame-pointer", "-g"]
ENV = dict(os.environ, ASAN_OPTIONS="detect_leaks=0:protect_shadow_gap=0",
           UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")


def _compile(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and ("sanitize" in r.stderr or "asan" in r.stderr.lower()):
        pytest.skip("compiler without sanitizer runtimes: " + r.stderr[-300:])
    assert r.returncode == 0, r.stderr[-4000:]


def test_oracle_under_asan_and_ubsan(tmp_path):
    cxx = shutil.which("g++")
    if not cxx:
        pytest.skip("no g++")
    exe = str(tmp_path / "oracle_san")
    _compile([cxx, "-std=c++17", "-O1", "-ffp-contract=off", *SAN,
              os.path.join(ROOT, "oracle", "oracle.cpp"),
              os.path.join(HERE, "sanitize", "oracle_driver.cpp"), "-o", exe])
    p = subprocess.run([exe], capture_output=True, text=True, env=ENV, timeout=300)
    assert p.returncode == 0, (p.stdout + p.stderr)[-4000:]
    assert "ok" in p.stdout


def test_abi_host_paths_under_asan_and_ubsan(tmp_path):
    """abi.cu's host code instrumented (nvcc -Xcompiler), linked with the other
    objects of the normal build; every call in the driver returns from host checks
    or is a size query, so no device is touched."""
    from moe_expert_offload_gb300 import _build

    cxx = shutil.which("g++")
    if not cxx:
        pytest.skip("no g++")
    _build.build()
    cc = _build.nvcc()
    obj = str(tmp_path / "abi_san.o")
    _compile([cc, *_build.ARCH, "-std=c++17", "-O1", "-Xcompiler", "-fPIC",
              *[f for s in SAN for f in ("-Xcompiler", s)],
              f"-I{os.path.join(ROOT, 'include')}", "-c",
              os.path.join(_build.CSRC, "abi.cu"), "-o", obj])
    others = [os.path.join(_build.HERE, "_build", os.path.basename(s)[:-3] + ".o")
              for s in _build._sources() if not s.endswith("abi.cu")]
    assert all(os.path.exists(o) for o in others), others
    exe = str(tmp_path / "abi_san")
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(cc)), "lib64")
    _compile([cxx, "-std=c++17", "-O1", *SAN, f"-I{os.path.join(ROOT, 'include')}",
              os.path.join(HERE, "sanitize", "abi_driver.cpp"), obj, *others,
              f"-L{cuda_lib}", f"-Wl,-rpath,{cuda_lib}", "-lcudart", "-o", exe])
    p = subprocess.run([exe], capture_output=True, text=True, env=ENV, timeout=300)
    assert p.returncode == 0, (p.stdout + p.stderr)[-4000:]
    assert "ok" in p.stdout
