"""The update kernel's load-phasing rule (zero1_policy.h, host-only C++),
compiled with g++ and checked at its boundaries: which launches are phased
and at what device-wide rate."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "zero_sharded_adamw_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include "zero1_policy.h"
int main() {
    double option; int world, mv16, reread, grid, sms;
    while (std::scanf("%lf %d %d %d %d %d", &option, &world, &mv16, &reread, &grid, &sms) == 6)
        std::printf("%.1f\n", zero1::load_rate_gbs(option, world, mv16 != 0, reread != 0, grid, sms));
    return 0;
}
"""

# (option, world, moments_bf16, reread, grid, num_sms) -> rate in GB/s (0 = free-running)
CASES = [
    ((0.0, 8, 0, 0, 152, 152), 0.0),        # W = 8 scratch path: off
    ((0.0, 15, 0, 0, 152, 152), 0.0),       # below W = 16: off
    ((0.0, 16, 0, 0, 152, 152), 14000.0),   # half a tile's period
    ((0.0, 19, 0, 0, 152, 152), 14000.0),
    ((0.0, 20, 0, 0, 152, 152), 7000.0),    # a whole tile's period
    ((0.0, 64, 0, 0, 152, 152), 7000.0),
    ((0.0, 512, 0, 0, 152, 152), 7000.0),
    ((0.0, 2, 0, 1, 152, 152), 17500.0),    # gradient re-read path
    ((0.0, 1, 0, 1, 152, 152), 17500.0),
    ((0.0, 2, 0, 0, 152, 152), 0.0),        # W = 2 on the scratch path (buckets, host pieces): off
    ((0.0, 64, 1, 0, 152, 152), 0.0),       # bf16 moments: never
    ((9000.0, 64, 1, 0, 152, 152), 0.0),
    ((0.0, 64, 0, 0, 32, 152), 0.0),        # grid short of every SM: never
    ((9000.0, 64, 0, 0, 100, 152), 0.0),
    ((0.0, 64, 0, 0, 152, 0), 0.0),         # SM count unknown: never
    ((-1.0, 64, 0, 0, 152, 152), 0.0),      # option < 0: never
    ((-1.0, 2, 0, 1, 152, 152), 0.0),
    ((9000.0, 8, 0, 0, 152, 152), 9000.0),  # an explicit rate applies at any W, on either path
    ((9000.0, 2, 0, 1, 152, 152), 9000.0),
]


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    d = tmp_path_factory.mktemp("policy")
    src, exe = d / "policy_driver.cpp", d / "policy_driver"
    src.write_text(DRIVER)
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    return str(exe)


def test_load_phasing_rule(driver):
    stdin = "".join(" ".join(str(v) for v in args) + "\n" for args, _ in CASES)
    out = subprocess.run([driver], input=stdin, capture_output=True, text=True, check=True).stdout.split()
    assert len(out) == len(CASES)
    for (args, want), got in zip(CASES, out):
        assert float(got) == want, (args, got, want)
