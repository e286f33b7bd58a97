"""Host code under AddressSanitizer and UndefinedBehaviorSanitizer (CPU only): the C oracle
and the host structures behind the C ABI (chunked hash tree, catalogue trie), each built
with -fsanitize=address,undefined into a small driver that walks every entry point on small
and ragged inputs and the error paths. Device code is not covered here (no sanitizer runs
on the GPU pool)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SAN = os.path.join(ROOT, "tests", "sanitize")
FLAGS = ["-g", "-O1", "-fno-omit-frame-pointer", "-fsanitize=address,undefined", "-fno-sanitize-recover=all"]


def _build_run(compiler, srcs, extra, tmp_path, name, env_extra):
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not found")
    exe = str(tmp_path / name)
    res = subprocess.run([compiler, *FLAGS, *extra, "-o", exe, *srcs], capture_output=True, text=True)
    if res.returncode != 0:
        if "asan" in res.stderr or "ubsan" in res.stderr or "sanitize" in res.stderr:
            pytest.skip("compiler without sanitizer runtimes")
        raise AssertionError(res.stderr[-4000:])
    env = dict(os.environ, **env_extra)
    out = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=600)
    text = out.stdout + out.stderr
    assert out.returncode == 0, text[-4000:]
    assert "runtime error" not in text and "AddressSanitizer" not in text, text[-4000:]
    assert "ok" in out.stdout


def test_oracle_under_sanitizers(tmp_path):
    # OpenMP's worker threads keep their pools until exit: leak checks stay off here
    _build_run("gcc", [os.path.join(SAN, "oracle_san.c"), os.path.join(ROOT, "oracle", "xattn_oracle.c")],
               ["-std=c11", "-fopenmp", "-ffp-contract=off", "-lm"], tmp_path, "oracle_san",
               {"ASAN_OPTIONS": "detect_leaks=0", "UBSAN_OPTIONS": "print_stacktrace=1", "OMP_NUM_THREADS": "2"})


def test_host_structures_under_sanitizers(tmp_path):
    csrc = os.path.join(ROOT, "decode_attention_xattention_gb300", "csrc")
    _build_run("g++", [os.path.join(SAN, "host_san.cpp"), os.path.join(csrc, "cht.cpp"), os.path.join(csrc, "trie.cpp")],
               ["-std=c++17"], tmp_path, "host_san",
               {"ASAN_OPTIONS": "detect_leaks=1", "UBSAN_OPTIONS": "print_stacktrace=1"})
