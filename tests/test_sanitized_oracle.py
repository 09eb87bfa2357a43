"""The CPU oracle and the record generator under AddressSanitizer and
UndefinedBehaviorSanitizer.

Both C files are compiled with -fsanitize=address,undefined (every report
fatal), and the oracle's pins (hand-worked trace, brute-force replay, closed
forms, invariants, rejections) and its property tests run in a child Python
process that loads those builds, with the sanitizer runtime preloaded.  An
out-of-bounds access, use after free or undefined operation anywhere in the
C code those tests reach fails this test.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FLAGS = ["-O1", "-g", "-fno-omit-frame-pointer", "-fsanitize=address,undefined",
         "-fno-sanitize-recover=all", "-fPIC", "-shared"]


def _runtime(name):
    p = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True)
    path = p.stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no gcc")
def test_oracle_pins_under_asan_and_ubsan(tmp_path):
    asan = _runtime("libasan.so")
    ubsan = _runtime("libubsan.so")
    if asan is None or ubsan is None:
        pytest.skip("the sanitizer runtimes are not installed")
    oracle_lib = tmp_path / "libhs_oracle_san.so"
    records_lib = tmp_path / "librecords_san.so"
    subprocess.check_call(["gcc", "-std=c11", "-Wall", *FLAGS, "-o", str(oracle_lib),
                           os.path.join(ROOT, "oracle", "hs_oracle.c")])
    subprocess.check_call(["gcc", "-std=gnu11", "-pthread", "-ffp-contract=off", *FLAGS,
                           "-o", str(records_lib), os.path.join(ROOT, "workloads", "records.c"),
                           "-lm"])
    env = dict(os.environ,
               LD_PRELOAD=f"{asan}:{ubsan}",
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=0:halt_on_error=1:exitcode=86",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1:exitcode=87",
               HS_ORACLE_LIB=str(oracle_lib), HS_RECORDS_LIB=str(records_lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "-m", "not gpu and not slow",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_properties.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert "passed" in r.stdout and "ERROR: AddressSanitizer" not in r.stderr, tail
    assert "runtime error:" not in r.stderr, tail
