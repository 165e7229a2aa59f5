"""The C ABI from plain C: tests/c_consumer.c is compiled with gcc as C99 with
warnings as errors against include/triforce_attn.h, linked against the built
library and run (it only makes calls that fail host validation, so no GPU is
needed)."""

import os
import shutil
import subprocess

import pytest

from hierarchical_speculative_decoding_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not installed")
def test_c_program_links_and_calls_the_library(tmp_path):
    lib = build.build()
    exe = tmp_path / "c_consumer"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_consumer.c"), "-o", str(exe), "-L", os.path.dirname(lib),
           "-l:" + os.path.basename(lib), "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c consumer ok" in r.stdout
