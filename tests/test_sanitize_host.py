"""The oracle and the library's host code (the affine packer and the Turbo4
codebook) built with AddressSanitizer and UndefinedBehaviorSanitizer and run
through every entry point on small inputs (tests/sanitize_driver.c): no
out-of-bounds access, leak, overflow or misaligned access, and the packer and
codebook agree with the oracle byte for byte under that build as well."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FLAGS = ["-O1", "-g", "-fno-omit-frame-pointer", "-fsanitize=address,undefined",
         "-fno-sanitize-recover=undefined"]


def _sanitizers_available(tmp):
    src = os.path.join(tmp, "probe.c")
    with open(src, "w") as f:
        f.write("int main(void) { return 0; }\n")
    r = subprocess.run(["gcc", *FLAGS, src, "-o", os.path.join(tmp, "probe")],
                       capture_output=True, text=True)
    return r.returncode == 0


def test_oracle_and_host_code_are_clean_under_sanitizers():
    if shutil.which("gcc") is None or shutil.which("g++") is None:
        pytest.skip("no gcc/g++")
    with tempfile.TemporaryDirectory() as tmp:
        if not _sanitizers_available(tmp):
            pytest.skip("gcc without the address/undefined sanitizer runtimes")
        inc = os.path.join(ROOT, "include")
        drv = os.path.join(tmp, "driver.o")
        host = os.path.join(tmp, "hostpack.o")
        exe = os.path.join(tmp, "sanitized")
        steps = [
            ["gcc", "-std=c11", *FLAGS, "-I", inc, "-c",
             os.path.join(ROOT, "tests", "sanitize_driver.c"), "-o", drv],
            ["g++", "-std=c++17", *FLAGS, "-I", inc, "-c",
             os.path.join(ROOT, "qwen3_gated_attention_gb300", "csrc", "hostpack.cpp"), "-o", host],
            ["g++", *FLAGS, drv, host, "-o", exe, "-lm", "-lpthread"],
        ]
        for cmd in steps:
            r = subprocess.run(cmd, capture_output=True, text=True)
            assert r.returncode == 0, f"{' '.join(cmd)}\n{r.stderr[-3000:]}"
        env = dict(os.environ)
        env["ASAN_OPTIONS"] = "detect_leaks=1:abort_on_error=0:halt_on_error=1"
        env["UBSAN_OPTIONS"] = "print_stacktrace=1:halt_on_error=1"
        r = subprocess.run([exe], capture_output=True, text=True, timeout=600, env=env)
        assert r.returncode == 0, r.stderr[-4000:]
        assert "runtime error" not in r.stderr and "AddressSanitizer" not in r.stderr, r.stderr[-4000:]
        assert "sanitized host run ok" in r.stdout
