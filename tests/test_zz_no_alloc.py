"""zero1_step_noalloc, the entry point that allocates no device memory.

It exists for callers that cannot call cudaMalloc (a framework allocator that
owns the device's memory, a plug-in with a fixed device budget, a loop that
cannot take cudaMalloc's device synchronisation): they own the fp32 master,
m and v and pass them in, and the step's scratch is a fixed array inside the
library.  This test calls it through the C ABI twice in a row (steps 1 and
2) and checks each result against the handle-based zero1_step run on the
same inputs, within the tolerance the parity tests use (1e-6 relative on the
fp32 state, 1 bf16 ulp on the replicas); with the same kernels and grid the
two should in fact agree bit for bit, which is checked as well.  Each call
is also checked directly against the CPU oracle running the same steps with
its own norm and clip coefficient, within the same tolerance.  It must pass
alone in a fresh process and after every other test, so it depends on no
state another test leaves behind.  The file sorts last so that a run that
stops at the first failure has run everything else first.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as WL
import zero_sharded_adamw_gb300 as z
from oracle import zero1_oracle as o
from tests.gpu_util import bf16_ulp, bits_equal, f32, rel_err, u16

pytestmark = pytest.mark.gpu

TOL = 1e-6


@pytest.mark.parametrize("n,world", [(1_000_003, 8), (65_541, 2), (4099, 4)])   # two kernels, re-read, one launch
def test_noalloc_matches_handle_step_on_two_calls(n, world):
    w = WL.Workload(f"noalloc_{n}_{world}", n, world, 0.02, 2, max_norm=0.5)
    hp = z.Hparams(**w.hparams())
    m0 = WL.master(w, "cuda")
    grads = {t: WL.grads(w, t, "cuda") for t in (1, 2)}

    # Existing entry point: a handle that owns its state.
    ref = []
    reps_a = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    with z.Zero1(n, world, hp) as opt:
        opt.set_state(m0)
        for t in (1, 2):
            opt.step(grads[t], reps_a)
            master = torch.empty(n, device="cuda")
            m, v = torch.empty_like(master), torch.empty_like(master)
            opt.get_state(master, m, v)
            torch.cuda.synchronize()
            ref.append((f32(master), f32(m), f32(v), [u16(r) for r in reps_a]))

    # The allocation-free entry point: caller-owned state, fixed scratch.
    master = m0.clone()
    m = torch.zeros_like(master)
    v = torch.zeros_like(master)
    reps_b = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    oracle = o.State(f32(m0))
    for t in (1, 2):
        z.zero1_step_noalloc(n, world, hp, t, grads[t], reps_b, master, m, v)
        torch.cuda.synchronize()
        got = (f32(master), f32(m), f32(v), [u16(r) for r in reps_b])
        want = ref[t - 1]
        for a, b in zip(got[:3], want[:3]):
            assert rel_err(a, b) <= TOL
            assert bits_equal(a, b)
        for ra, rb in zip(got[3], want[3]):
            assert bf16_ulp(ra, rb) <= 1
            assert np.array_equal(ra, rb)
        # the oracle, free-running on the same gradients
        reps_o, _, _ = o.step(oracle, [u16(g) for g in grads[t]], o.HP(**w.hparams()))
        for a, b in zip(got[:3], (oracle.master, oracle.m, oracle.v)):
            assert rel_err(a, b) <= TOL
        for ra, rb in zip(got[3], reps_o):
            assert bf16_ulp(ra, rb) <= 1


def test_noalloc_rejects_sizes_beyond_its_scratch():
    n, world = (1 << 22) + 1, 2
    # raw addresses: the binding cannot size-check them, so the C entry
    # point's own limit check is what answers
    g = [torch.zeros(8, dtype=torch.bfloat16, device="cuda").data_ptr()] * world
    s = torch.zeros(8, device="cuda").data_ptr()
    with pytest.raises(z.Zero1Error) as e:
        z.zero1_step_noalloc(n, world, z.Hparams(), 1, g, g, s, s, s)
    assert e.value.code == -1
    assert "4194304" in str(e.value)
