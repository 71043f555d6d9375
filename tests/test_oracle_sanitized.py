"""The oracle's C under AddressSanitizer and UndefinedBehaviorSanitizer: the
oracle pins and the acceptance-reduction checks run again, in a child
process, against a copy of dg_oracle.c built with
-fsanitize=address,undefined (no recovery from undefined behaviour) and the
sanitizer runtimes preloaded.  Any out-of-bounds access, use of freed
memory, signed overflow, bad shift or misaligned access fails the run.
Skipped where gcc has no sanitizer runtime."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _runtime(name):
    try:
        p = subprocess.run(["gcc", "-print-file-name=" + name], capture_output=True, text=True,
                           check=True).stdout.strip()
    except (OSError, subprocess.CalledProcessError):
        return None
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_oracle_pins_under_address_and_undefined_behaviour_sanitizers(tmp_path):
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if asan is None or ubsan is None:
        pytest.skip("gcc sanitizer runtimes not installed")
    lib = str(tmp_path / "liboracle_san.so")
    subprocess.run(["gcc", "-O1", "-g", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                    "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined",
                    "-fno-omit-frame-pointer", "-fPIC", "-shared", "-o", lib,
                    os.path.join(ROOT, "oracle", "dg_oracle.c"), "-lm"], check=True)
    code = ("import sys\n"
            "sys.path.insert(0, %r)\n"
            "import oracle\n"
            "oracle._LIB_PATH = %r\n"
            "import pytest\n"
            "sys.exit(pytest.main(['-q', '-x', '-p', 'no:cacheprovider', "
            "'tests/test_oracle_pins.py', 'tests/test_acceptance_reduction.py']))\n"
            % (ROOT, lib))
    env = dict(os.environ, LD_PRELOAD=asan + ":" + ubsan,
               ASAN_OPTIONS="detect_leaks=0:halt_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                         text=True, timeout=900)
    log = out.stdout[-3000:] + out.stderr[-3000:]
    assert out.returncode == 0, log
    assert "AddressSanitizer" not in log and "runtime error" not in log, log
    # the sanitized copy, not the regular build, is what ran
    assert " passed" in out.stdout, log
