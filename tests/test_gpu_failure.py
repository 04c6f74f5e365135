"""Failure detection on the GPU without a fault: a pipeline wait that runs
out is reported, and the device stays usable.

The update kernel's waits on its shared-memory ring are bounded (1 s of
global time).  With the test-only option inject_wait_timeout its producer
issues no loads, so every consumer and store-warp wait gives up: the kernel
returns, the sticky timeout bit is set, and zero1_get_grad_norm reports
ZERO1_ECUDA.  No trap, no bad address, no unbounded loop is involved.
Afterwards a fresh handle steps normally and matches the oracle.
"""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import workloads as WL
import zero_sharded_adamw_gb300 as z
from oracle import zero1_oracle as o
from tests.gpu_util import bits_equal, f32, u16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,world", [(100_003, 8), (70_001, 2)])     # ĝ scratch and gradient re-read
def test_wait_timeout_is_reported_and_the_device_stays_usable(n, world):
    w = WL.Workload("fail", n, world, 0.01, 2, max_norm=0.05)
    hp = z.Hparams(**w.hparams())
    g = WL.grads(w, 1, "cuda")
    reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    with z.Zero1(n, world, hp, z.Options(inject_wait_timeout=True, small_step=-1)) as bad:
        bad.set_state(WL.master(w, "cuda"))
        t0 = time.monotonic()
        bad.step(g, reps)                          # enqueues; the kernel gives up after ~1 s
        with pytest.raises(z.Zero1Error) as e:
            bad.grad_norm()
        assert e.value.code == -4 and "gave up" in str(e.value)
        assert time.monotonic() - t0 < 30
        bad.step(g, reps)                          # the bit is sticky
        with pytest.raises(z.Zero1Error):
            bad.grad_norm()

    # the context is intact: a fresh handle's step equals the oracle's
    m0 = WL.master(w, "cuda")
    with z.Zero1(n, world, hp) as good:
        good.set_state(m0)
        good.step(g, reps)
        norm, c = good.grad_norm()
        master = torch.empty(n, device="cuda")
        mm, vv = torch.empty_like(master), torch.empty_like(master)
        good.get_state(master, mm, vv)
        torch.cuda.synchronize()
    st = o.State(f32(m0))
    want_reps, _, _ = o.step(st, [u16(x) for x in g], o.HP(**w.hparams()), clip_override=np.float32(c))
    assert bits_equal(f32(master), st.master) and bits_equal(f32(mm), st.m) and bits_equal(f32(vv), st.v)
    assert all(np.array_equal(u16(r), want) for r, want in zip(reps, want_reps))
