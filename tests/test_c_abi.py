"""The library used from plain C: include/attn.h compiles as C99 (-pedantic),
libattn.so links into a C program, argument validation answers before any
launch (no GPU), and a forward driven from host code through the C ABI alone
matches the oracle (GPU)."""

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from exact_attention_34_gb300 import build as eb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIBDIR = os.path.join(ROOT, "exact_attention_34_gb300")


def _compile(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not found")
def test_c99_program_links_and_validates(tmp_path):
    eb.build()
    exe = str(tmp_path / "abi_check")
    _compile(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
              os.path.join(ROOT, "tests", "c", "abi_check.c"), "-L", LIBDIR, "-lattn", f"-Wl,-rpath,{LIBDIR}",
              "-o", exe])
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout


def _bf16_to_f64(raw):
    return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.gpu
def test_forward_driven_from_c(tmp_path):
    eb.build()
    exe = str(tmp_path / "fwd_from_c")
    _compile([eb._nvcc(), "-O2", "-std=c++17", "-I", os.path.join(ROOT, "include"),
              os.path.join(ROOT, "tests", "c", "fwd_from_c.cu"), "-L", LIBDIR, "-lattn", f"-Xlinker=-rpath,{LIBDIR}",
              "-o", exe])
    r = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True)
    assert r.returncode == 0 and "OK" in r.stdout, r.stdout + r.stderr
    shape = (1, 200, 2, 64)
    q, k, v, o = (_bf16_to_f64(np.fromfile(tmp_path / f"{n}.bin", dtype=np.uint16)).reshape(shape)
                  for n in ("q", "k", "v", "o"))
    lse = np.fromfile(tmp_path / "lse.bin", dtype=np.float32).reshape(1, 2, 200)
    o_ref, lse_ref = oracle.forward(q, k, v, causal=True, scale=0.125)
    assert np.max(np.abs(o - o_ref)) <= 1e-2 * np.max(np.abs(o_ref))
    assert np.max(np.abs(lse - lse_ref)) <= 1e-2 * np.max(np.abs(lse_ref))
