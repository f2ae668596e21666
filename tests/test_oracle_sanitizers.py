"""The oracle's C under AddressSanitizer and UndefinedBehaviorSanitizer.

The same source, compiled with -fsanitize=address,undefined plus the
float-to-int overflow and float division checks (no recovery), runs the
oracle pins in a child process: an out-of-bounds access, a signed overflow,
a misaligned load, an out-of-range shift or an overflowing float-to-int
conversion fails the run.  The quantiser's saturation reading exists
precisely so that no conversion overflows, so that check holds it to it.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_oracle_pins_under_asan_and_ubsan(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    asan = subprocess.run([gcc, "-print-file-name=libasan.so"], capture_output=True,
                          text=True).stdout.strip()
    if not os.path.isabs(asan) or not os.path.exists(asan):
        pytest.skip("the gcc sanitizer runtime is not installed")
    lib = tmp_path / "libqmm_oracle_san.so"
    subprocess.run([gcc, "-O1", "-g", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", "-fno-omit-frame-pointer",
                    "-fsanitize=address,undefined,float-cast-overflow,float-divide-by-zero",
                    "-fno-sanitize-recover=all", os.path.join(ROOT, "oracle", "qmm_oracle.c"),
                    "-o", str(lib), "-lm"], check=True)
    # A sanitizer that halts the child ends it before the child's test runner
    # could show what it had captured: the child runs without output capture
    # (UBSan writes to stderr) and ASan also writes its reports to files.
    logs = tmp_path / "san"
    env = dict(os.environ, QMM_ORACLE_LIB=str(lib), LD_PRELOAD=asan,
               ASAN_OPTIONS=f"detect_leaks=0:halt_on_error=1:log_path={logs}",
               UBSAN_OPTIONS=f"halt_on_error=1:print_stacktrace=1:log_path={logs}")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "--capture=no", os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    reports = sorted(tmp_path.glob("san*"))
    text = "".join(f.read_text(errors="replace") for f in reports) + r.stderr
    assert not reports and "runtime error" not in text and "Sanitizer" not in text, text[-4000:]
    assert r.returncode == 0, (r.stdout + r.stderr)[-4000:]
