"""Host-only code under compiler sanitizers (no GPU).

The oracle (plain C) and the library's host code (dependency builder, grouped scoreboard
tables, host-thread protocol model) are rebuilt with AddressSanitizer + UndefinedBehaviorSanitizer,
and the protocol model's threads once more with ThreadSanitizer, then driven over ragged shapes,
gated chains, several thread counts and a withheld release.  Any sanitizer report fails the test.
(The device code has no such tool on this pool; its checks are the bounded waits, the status
word and the parity tests.)
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.join(ROOT, "tests", "sanitize")
REPORT_MARKS = ("ERROR: AddressSanitizer", "runtime error:", "WARNING: ThreadSanitizer", "ERROR: LeakSanitizer")


def _build_and_run(cmd, exe, tmp_path):
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=tmp_path)
    if r.returncode != 0 and ("cannot find" in r.stderr or "unrecognized" in r.stderr):
        pytest.skip("sanitizer runtime not available: " + r.stderr.strip().splitlines()[-1])
    assert r.returncode == 0, r.stderr[-2000:]
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1", UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1",
               TSAN_OPTIONS="halt_on_error=1")
    run = subprocess.run([str(tmp_path / exe)], capture_output=True, text=True, env=env, timeout=600)
    out = run.stdout + run.stderr
    assert run.returncode == 0 and not any(m in out for m in REPORT_MARKS), out[-4000:]
    return out


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no gcc")
def test_oracle_under_asan_ubsan(tmp_path):
    cmd = ["gcc", "-std=c11", "-O1", "-g", "-fno-omit-frame-pointer", "-ffp-contract=off",
           "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined", "-pthread",
           os.path.join(HERE, "drive_oracle.c"), os.path.join(ROOT, "oracle", "oracle.c"), "-lm", "-o", "drive_oracle"]
    assert "0 failures" in _build_and_run(cmd, "drive_oracle", tmp_path)


@pytest.mark.skipif(shutil.which("g++") is None, reason="no g++")
@pytest.mark.parametrize("sanitize", ["address,undefined", "thread"])
def test_host_protocol_under_sanitizers(tmp_path, sanitize):
    extra = ["-fno-sanitize-recover=undefined"] if "undefined" in sanitize else []
    cmd = ["g++", "-std=c++17", "-O1", "-g", "-fno-omit-frame-pointer", f"-fsanitize={sanitize}", *extra, "-pthread",
           "-Wall", "-Wextra", "-Wshadow", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "drive_host.cpp"),
           os.path.join(ROOT, "mlp_latency_gb300", "csrc", "host_protocol.cpp"), "-o", "drive_host"]
    assert "0 failures" in _build_and_run(cmd, "drive_host", tmp_path)
