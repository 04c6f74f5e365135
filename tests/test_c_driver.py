"""The C ABI from plain C: tests/c_driver/zero1_c_driver.c includes only
zero1.h and the CUDA runtime's C header.  On CPU it must compile as strict
C99 against the header and link against the library; on a GPU its steps
(inputs drawn by its own generator and written to files) must equal the
oracle's bit for bit given the clip coefficients the library applied."""
from __future__ import annotations

import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import zero1_oracle as o
from zero_sharded_adamw_gb300 import _build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "c_driver", "zero1_c_driver.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out: str) -> str:
    lib = _build.build()
    libdir = os.path.dirname(lib)
    cmd = [shutil.which("gcc") or "gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O2",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"), SRC,
           "-L", libdir, "-lzero1", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-o", out]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def test_c_driver_builds_as_c99(tmp_path):
    exe = _compile(str(tmp_path / "drv"))
    assert os.access(exe, os.X_OK)


@pytest.mark.parametrize("std", ["-std=c99", "-std=c11"])
def test_header_is_pedantic_c(tmp_path, std):
    """zero1.h alone compiles as ISO C with every warning an error."""
    src = tmp_path / "h.c"
    src.write_text('#include "zero1.h"\nint main(void) { zero1_handle h = 0; return zero1_destroy(h); }\n')
    subprocess.run([shutil.which("gcc") or "gcc", std, "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), "-fsyntax-only", str(src)], check=True)


@pytest.mark.gpu
def test_c_driver_steps_match_the_oracle(tmp_path):
    n, world, steps = 100_003, 4, 3
    exe = _compile(str(tmp_path / "drv"))
    out = tmp_path / "out"
    out.mkdir()
    r = subprocess.run([exe, str(n), str(world), str(steps), str(out)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    rd = lambda name, dt: np.fromfile(out / name, dtype=dt)
    st = o.State(rd("master0.f32", np.float32))
    clips = rd("clip.f32", np.float32)
    hp = o.HP(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.05)
    free = o.State(rd("master0.f32", np.float32))
    for t in range(1, steps + 1):
        g = [rd(f"grads_t{t}_r{q}.bf16", np.uint16) for q in range(world)]
        reps, _, _ = o.step(st, g, hp, clip_override=np.float32(clips[t - 1]))
        _, _, c_own = o.step(free, g, hp)
        assert abs(float(clips[t - 1]) - float(c_own)) <= 1e-6 * float(c_own)
    for name, want in (("master.f32", st.master), ("m.f32", st.m), ("v.f32", st.v)):
        assert np.array_equal(rd(name, np.float32).view(np.uint32), want.view(np.uint32)), name
    for q in (0, world - 1):
        assert np.array_equal(rd(f"rep_{q}.bf16", np.uint16), reps[q])
