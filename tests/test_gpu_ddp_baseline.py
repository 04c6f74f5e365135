"""The DDP baseline built from the library's pieces, against the oracle:
the W bf16 gradients all-reduced (rank-ordered fp32 mean rounded to bf16,
in place), then each rank's full AdamW on its own replicated state (a
handle of world 1 per rank).  Every rank's state equals the oracle's
(all-reduce, then a one-rank step with the GPU's clip coefficient) bit for
bit, and all ranks stay identical."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as WL
import zero_sharded_adamw_gb300 as z
from oracle import zero1_oracle as o
from tests.gpu_util import bits_equal, f32, u16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,world", [(100_003, 4), (4099, 8)])
def test_ddp_baseline_matches_oracle(n, world):
    w = WL.Workload("ddp", n, world, 0.01, 3, max_norm=0.05)
    d = w.hparams()
    m0 = WL.master(w, "cuda")
    ranks = [z.Zero1(n, 1, z.Hparams(**d)) for _ in range(world)]
    for h in ranks:
        h.set_state(m0)
    reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    states = [o.State(f32(m0)) for _ in range(world)]
    try:
        for t in range(1, 4):
            grads = WL.grads(w, t, "cuda")
            host = [u16(g) for g in grads]
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            z.zero1_allreduce(n, world, z.DTYPE_BF16, z.OP_AVG, grads, grads, err)
            for q, h in enumerate(ranks):
                h.step([grads[q]], [reps[q]])
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            avg, _ = o.allreduce_rs_ag(host, average=True)
            assert all(np.array_equal(u16(grads[q]), avg[q]) for q in range(world))
            for q, h in enumerate(ranks):
                _, c = h.grad_norm()
                reps_o, _, _ = o.step(states[q], [avg[q]], o.HP(**d), clip_override=np.float32(c))
                assert np.array_equal(u16(reps[q]), reps_o[0])
        for q, h in enumerate(ranks):
            master = torch.empty(n, device="cuda")
            m, v = torch.empty_like(master), torch.empty_like(master)
            h.get_state(master, m, v)
            torch.cuda.synchronize()
            assert bits_equal(f32(master), states[q].master)
            assert bits_equal(f32(m), states[q].m) and bits_equal(f32(v), states[q].v)
            assert bits_equal(states[q].master, states[0].master)      # replicated: every rank the same
    finally:
        for h in ranks:
            h.close()
