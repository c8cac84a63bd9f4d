"""Host code under AddressSanitizer and UndefinedBehaviorSanitizer (CPU only).

KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"),
Tests/Validation item: the PR's checks include an ASan/UBSan-clean build.  The
driver (host_sanitize_driver.cpp) is built with -fsanitize=address,undefined and
-fno-sanitize-recover, together with the oracle's C, and runs:
- the cache file's host code (csrc/cachefile.h, the part of persist.cu that
  reads untrusted headers): header parse, magic repair, torn and truncated files,
  inconsistent and random headers, the version 1 -> 2 rewrite and its failure path;
- every entry point of the oracle's C on small inputs with special values.
Any sanitizer report aborts the driver with a non-zero status.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SAN = ["-O1", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
       "-fno-omit-frame-pointer", "-fopenmp"]


def test_host_code_is_sanitizer_clean(tmp_path):
    cxx, cc = shutil.which("g++"), shutil.which("gcc")
    if cxx is None or cc is None:
        pytest.skip("no host C/C++ compiler")
    inc = ["-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(ROOT, "fp8_mla_latent_gb300", "csrc"),
           "-I" + os.path.join(ROOT, "oracle")]
    drv, orc, exe = tmp_path / "driver.o", tmp_path / "oracle.o", tmp_path / "driver"
    for cmd in ([cxx, "-std=c++17", *SAN, *inc, "-c", os.path.join(HERE, "host_sanitize_driver.cpp"),
                 "-o", str(drv)],
                [cc, "-std=c11", *SAN, *inc, "-c", os.path.join(ROOT, "oracle", "kv8_oracle.c"),
                 "-o", str(orc)],
                [cxx, *SAN, str(drv), str(orc), "-lm", "-o", str(exe)]):
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-2000:]
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0:exitcode=23",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1:exitcode=24", OMP_NUM_THREADS="2")
    work = tmp_path / "files"
    work.mkdir()
    r = subprocess.run([str(exe), str(work)], capture_output=True, text=True, env=env, timeout=600)
    report = r.stdout + r.stderr
    assert r.returncode == 0, report[-4000:]
    assert "runtime error" not in report and "AddressSanitizer" not in report, report[-4000:]
    assert "all checks passed" in r.stdout
