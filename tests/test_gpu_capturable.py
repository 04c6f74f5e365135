"""Capturable steps: the step counter and learning rate on the device, the
step size and decay formed by the kernels, steps captured in CUDA graphs.

A capturable handle must give the same master, m, v and replicas, bit for
bit, as a plain handle fed the same gradients: stepped directly, across the
end of its bias-correction table, with lr changed between steps, and as a
replayed CUDA graph (one captured step replayed once per step, with lr read
from a caller's device scalar).  Both the two-kernel path and the one-launch
cluster path are covered.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads as WL
import zero_sharded_adamw_gb300 as z
from tests.gpu_util import bits_equal, f32, u16

pytestmark = pytest.mark.gpu


def _state(opt: z.Zero1, n: int):
    master = torch.empty(n, dtype=torch.float32, device="cuda")
    m, v = torch.empty_like(master), torch.empty_like(master)
    t = opt.get_state(master, m, v)
    torch.cuda.synchronize()
    return f32(master), f32(m), f32(v), t


def _same(a, b):
    assert a[3] == b[3], (a[3], b[3])
    for x, y in zip(a[:3], b[:3]):
        assert bits_equal(x, y)


SHAPES = [(100_003, 8), (4099, 4), (4096, 4), (70_001, 2)]   # two kernels (W >= 3), the one-launch cluster (ragged and 8-aligned), re-read (W <= 2)


@pytest.mark.parametrize("n,world", SHAPES)
def test_capturable_equals_plain(n, world):
    w = WL.Workload("cap", n, world, 0.01, 6, max_norm=0.05)
    hp = z.Hparams(**w.hparams())
    m0 = WL.master(w, "cuda")
    lrs = [1e-3, 1e-3, 5e-4, 2e-3, 1e-3, 7e-4]
    outs = []
    for cap in (False, True):
        reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
        with z.Zero1(n, world, hp, z.Options(capturable=cap)) as opt:
            opt.set_state(m0)
            for t in range(1, 7):
                opt.set_lr(lrs[t - 1])
                opt.step(WL.grads(w, t, "cuda"), reps)
            outs.append((_state(opt, n), [u16(r) for r in reps]))
    _same(outs[0][0], outs[1][0])
    assert all(np.array_equal(a, b) for a, b in zip(outs[0][1], outs[1][1]))


def test_capturable_across_table_end():
    """beta = (0.5, 0.6): both bias corrections reach 1.0 in double near
    t = 74, where the device table ends; steps 70..78 straddle it."""
    n, world = 5000, 4
    w = WL.Workload("tab", n, world, 0.01, 8, beta1=0.5, beta2=0.6, max_norm=0.05)
    hp = z.Hparams(**w.hparams())
    m0 = WL.master(w, "cuda")
    outs = []
    for cap in (False, True):
        reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
        with z.Zero1(n, world, hp, z.Options(capturable=cap, small_step=-1)) as opt:
            opt.set_state(m0, t=70)
            for t in range(71, 79):
                opt.step(WL.grads(w, t, "cuda"), reps)
            outs.append(_state(opt, n))
    assert outs[1][3] == 78
    _same(outs[0], outs[1])


@pytest.mark.parametrize("n,world", SHAPES)
def test_graph_replay(n, world):
    """One step captured in a CUDA graph and replayed for steps 2..7, with
    new gradients copied into the captured buffers and a cosine lr written
    to a device scalar before each replay, equals a plain handle stepping
    with set_lr."""
    steps = 7
    w = WL.Workload("graph", n, world, 0.01, steps, max_norm=0.05)
    hp = z.Hparams(**w.hparams())
    m0 = WL.master(w, "cuda")
    lr_of = lambda t: 1e-3 * (0.5 + 0.5 * math.cos(math.pi * t / steps))

    reps_ref = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    with z.Zero1(n, world, hp) as ref:
        ref.set_state(m0)
        for t in range(1, steps + 1):
            ref.set_lr(lr_of(t))
            ref.step(WL.grads(w, t, "cuda"), reps_ref)
        want = _state(ref, n)

    grads = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    lr_dev = torch.zeros(1, dtype=torch.float64, device="cuda")
    with z.Zero1(n, world, hp, z.Options(capturable=True)) as opt:
        opt.set_state(m0)
        opt.set_lr_ptr(lr_dev)
        lr_dev.fill_(lr_of(1))
        WL.grads(w, 1, "cuda", out=grads)
        opt.step(grads, reps, torch.cuda.current_stream())      # step 1, uncaptured
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            opt.step(grads, reps, torch.cuda.current_stream())  # captured, not run
        torch.cuda.synchronize()
        for t in range(2, steps + 1):
            WL.grads(w, t, "cuda", out=grads)
            lr_dev.fill_(lr_of(t))
            g.replay()
        torch.cuda.synchronize()
        got = _state(opt, n)
    _same(want, got)
    assert all(np.array_equal(u16(a), u16(b)) for a, b in zip(reps, reps_ref))


@pytest.mark.parametrize("n,world", [(100_003, 8), (4099, 4)])
@pytest.mark.parametrize("variant", ["bf16_moments", "decay_first_clip_eps"])
def test_graph_replay_variants(n, world, variant):
    """The step variants replayed from a CUDA graph equal plain steps."""
    kw = ({"moments_bf16": True} if variant == "bf16_moments"
          else {"decay_before_update": True, "clip_eps": 1e-6})
    w = WL.Workload("gv", n, world, 0.01, 5, lr=1e-2, weight_decay=0.3, max_norm=0.05)
    hp = z.Hparams(**w.hparams())
    m0 = WL.master(w, "cuda")
    dt = torch.bfloat16 if kw.get("moments_bf16") else torch.float32

    def state(opt):
        master = torch.empty(n, dtype=torch.float32, device="cuda")
        m, v = torch.empty(n, dtype=dt, device="cuda"), torch.empty(n, dtype=dt, device="cuda")
        t = opt.get_state(master, m, v)
        torch.cuda.synchronize()
        return [x.view(torch.int32 if x.dtype == torch.float32 else torch.int16).cpu() for x in (master, m, v)], t

    reps_ref = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    with z.Zero1(n, world, hp, z.Options(**kw)) as ref:
        ref.set_state(m0)
        for t in range(1, 6):
            ref.step(WL.grads(w, t, "cuda"), reps_ref)
        want = state(ref)
    grads = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    with z.Zero1(n, world, hp, z.Options(capturable=True, **kw)) as opt:
        opt.set_state(m0)
        WL.grads(w, 1, "cuda", out=grads)
        opt.step(grads, reps, torch.cuda.current_stream())
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            opt.step(grads, reps, torch.cuda.current_stream())
        for t in range(2, 6):
            WL.grads(w, t, "cuda", out=grads)
            g.replay()
        torch.cuda.synchronize()
        got = state(opt)
    assert got[1] == want[1] == 5
    assert all(torch.equal(a, b) for a, b in zip(got[0], want[0]))
    assert all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(reps, reps_ref))


def test_capturable_bucketed_equals_plain():
    n, world = 200_003, 8
    w = WL.Workload("bk", n, world, 0.01, 3, max_norm=0.05)
    hp = z.Hparams(**w.hparams())
    m0 = WL.master(w, "cuda")
    cuts = [0, 50_000, 120_000, n]
    outs = []
    for cap in (False, True):
        reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
        with z.Zero1(n, world, hp, z.Options(capturable=cap)) as opt:
            opt.set_state(m0)
            for t in range(1, 4):
                g = WL.grads(w, t, "cuda")
                z.zero1_bucket_begin(opt.handle)
                for a, b in zip(cuts[:-1], cuts[1:]):
                    z.zero1_bucket_reduce(opt.handle, a, b - a, [x[a:] for x in g])
                z.zero1_bucket_finish(opt.handle, reps)
            outs.append(_state(opt, n))
    _same(outs[0], outs[1])


def test_capturable_errors():
    with z.Zero1(64, 2) as opt:
        with pytest.raises(z.Zero1Error):
            opt.set_lr_ptr(torch.zeros(1, dtype=torch.float64, device="cuda"))
    with pytest.raises(z.Zero1Error):                  # bias correction would need ~37M table entries
        z.Zero1(64, 2, z.Hparams(beta2=0.999999), z.Options(capturable=True))
    with z.Zero1(64, 2, None, z.Options(capturable=True)) as opt:
        buf = torch.zeros(2, dtype=torch.float64, device="cuda")
        with pytest.raises(z.Zero1Error):
            opt.set_lr_ptr(buf.data_ptr() + 4)
        opt.set_lr_ptr(None)
