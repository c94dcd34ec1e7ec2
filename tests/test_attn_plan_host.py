"""Host check of the decode-attention split plans, without a GPU.

bw_attn_plan.cuh holds the integer arithmetic by which one attention launch
splits positions 0..p of a KV head's cache over its CTAs (the workspace
kernel's splits and the cluster kernel's CTAs) and picks its launch shape.
The same header is compiled into the CUDA kernels and, here, by the host
compiler into tests/attn_plan_check.cpp. That program checks, for every
position of caches of several sizes and every launch shape, that the
shares partition 0..p in order and fit a CTA's staging, and that invalid
positions get none. The decode attention follows the W2A8 page's §六
item 2: a preallocated KV cache, one launch per step, the position read on
the device.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_gemv_bitlinear_gb300", "csrc")
SRC = os.path.join(ROOT, "tests", "attn_plan_check.cpp")


def test_attention_split_plans_partition_every_context(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "attn_plan_check")
    subprocess.run([cxx, "-std=c++17", "-O2", "-Wall", "-Wextra", "-Werror",
                    "-I", CSRC, SRC, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout
    assert r.stdout.startswith("ok "), r.stdout
