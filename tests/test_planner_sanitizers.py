"""The host planner under AddressSanitizer and UndefinedBehaviorSanitizer (CPU, no GPU).

leyline_planner.cpp validates and plans caller-supplied directives before anything reaches
a device.  tests/planner_sanitize.cpp feeds it seeded random descriptors, lengths and
directives, valid and invalid, and checks every accepted plan's lengths, page counts,
segment ranges and byte accounting; built with the sanitizers, any out-of-bounds access,
signed overflow or misaligned read fails the run.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INCLUDE = "/usr/local/cuda/include"


def test_planner_fuzz_under_sanitizers(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None or not os.path.exists(os.path.join(CUDA_INCLUDE, "cuda_runtime.h")):
        pytest.skip("needs g++ and the CUDA headers")
    exe = tmp_path / "planner_sanitize"
    cmd = [gxx, "-std=c++17", "-O1", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
           "-fno-omit-frame-pointer", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(ROOT, "rope_rotation_gb300", "csrc"), "-I", CUDA_INCLUDE,
           os.path.join(ROOT, "tests", "planner_sanitize.cpp"),
           os.path.join(ROOT, "rope_rotation_gb300", "csrc", "leyline_planner.cpp"), "-o", str(exe)]
    build = subprocess.run(cmd, capture_output=True, text=True)
    if build.returncode != 0 and "sanitize" in build.stderr:
        pytest.skip("the sanitizer runtimes are not installed: " + build.stderr.strip()[-200:])
    assert build.returncode == 0, build.stderr
    for seed in (1, 2, 3):
        run = subprocess.run([str(exe), "60000", str(seed)], capture_output=True, text=True, timeout=300)
        assert run.returncode == 0, run.stdout + run.stderr
        assert "0 failed checks" in run.stdout
