"""Step variants on the GPU against the oracle: torch.optim.AdamW's decay
order, a clip eps, m and v stored in bf16, and all three together.

Same protocol as test_gpu_parity: with the GPU's clip coefficient injected
the oracle's master, m, v and replicas must match bit for bit; the norm and
the coefficient within 1e-6 of the oracle's own; the free-running oracle
within 1e-6 relative (fp32 moments).  With bf16 moments a one-fp32-ulp
difference in c can flip a bf16 rounding of m or v (and so of d) at any
step, and the flips carry into later steps, so the free-running bounds are
counted in bf16 roundings: after t steps m and v lie within t * 2^-6 of the
oracle's at the array's RMS scale (each moment update rounds twice, and one
bf16 ulp is at most 2^-7 relative), and the master within 2^-5 times the
summed step sizes (two flipped roundings of |u| <= ~1 per step).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads as WL
import zero_sharded_adamw_gb300 as z
from oracle import zero1_oracle as o
from tests.gpu_util import Guarded, bits_equal, f32, rel_err, u16

pytestmark = pytest.mark.gpu


def _moments(opt: z.Zero1, n: int, bf16: bool):
    master = torch.empty(n, dtype=torch.float32, device="cuda")
    dt = torch.bfloat16 if bf16 else torch.float32
    m, v = torch.empty(n, dtype=dt, device="cuda"), torch.empty(n, dtype=dt, device="cuda")
    opt.get_state(master, m, v)
    torch.cuda.synchronize()
    conv = u16 if bf16 else f32
    return f32(master), conv(m), conv(v)


def _widen(x: np.ndarray) -> np.ndarray:
    return (x.astype(np.uint32) << 16).view(np.float32)


def run_variant(w: WL.Workload, steps: int, opts: o.Options, small_step: int = 0):
    d = w.hparams()
    step_budget = 0.0
    zopts = z.Options(opts.decay_before_update, opts.clip_eps, opts.moments_bf16, small_step=small_step)
    ohp = o.HP(**d)
    m0 = WL.master(w, "cuda")
    grads = [Guarded(w.n, torch.bfloat16) for _ in range(w.world)]
    reps = [Guarded(w.n, torch.bfloat16) for _ in range(w.world)]
    with z.Zero1(w.n, w.world, z.Hparams(**d), zopts) as opt:
        opt.set_state(m0)
        inj, free = o.state_ex(f32(m0), opts), o.state_ex(f32(m0), opts)
        for t in range(1, steps + 1):
            WL.grads(w, t, "cuda", out=[g.t for g in grads])
            opt.step([g.t for g in grads], [r.t for r in reps])
            norm_g, c_g = opt.grad_norm()
            gh = [u16(g.t) for g in grads]
            reps_i, norm_i, _ = o.step_ex(inj, gh, ohp, opts, clip_override=np.float32(c_g))
            _, _, c_f = o.step_ex(free, gh, ohp, opts)
            master, m, v = _moments(opt, w.n, opts.moments_bf16)
            assert bits_equal(master, inj.master), f"step {t}: master"
            assert np.array_equal(m.view(np.uint8), inj.m.view(np.uint8)), f"step {t}: m"
            assert np.array_equal(v.view(np.uint8), inj.v.view(np.uint8)), f"step {t}: v"
            for r in range(w.world):
                assert np.array_equal(u16(reps[r].t), reps_i[r]), f"step {t}: replica {r}"
            if math.isfinite(norm_i) and norm_i > 0:
                assert abs(norm_g - norm_i) <= 1e-6 * norm_i
                assert abs(float(c_g) - float(c_f)) <= 1e-6 * float(c_f)
            if opts.moments_bf16:
                step_budget += d["lr"] * math.sqrt(1 - d["beta2"] ** t) / (1 - d["beta1"] ** t)
                assert rel_err(_widen(m), _widen(free.m)) <= t * 2.0 ** -6
                assert rel_err(_widen(v), _widen(free.v)) <= t * 2.0 ** -6
                assert float(np.max(np.abs(master.astype(np.float64) - free.master))) <= step_budget * 2.0 ** -5
            else:
                assert rel_err(master, free.master) <= 1e-6
                assert rel_err(m, free.m) <= 1e-6 and rel_err(v, free.v) <= 1e-6
        assert all(b.intact() for b in grads + reps)


def test_decay_first():
    run_variant(WL.Workload("df", 100_003, 8, 0.01, 5, lr=1e-2, weight_decay=0.5, max_norm=0.05),
                5, o.Options(decay_before_update=True))


def test_clip_eps():
    run_variant(WL.Workload("ce", 4099, 4, 0.01, 5, max_norm=0.05), 5, o.Options(clip_eps=1e-6))


@pytest.mark.parametrize("n,world", [(1_000_003, 8), (65_541, 2), (7, 3), (4096, 1)])
def test_bf16_moments(n, world):
    run_variant(WL.Workload("mv", n, world, 0.01, 5, max_norm=0.05), 5, o.Options(moments_bf16=True))


@pytest.mark.parametrize("small_step", [1, -1])
@pytest.mark.parametrize("variant", ["decay_first", "clip_eps", "bf16_moments", "all"])
def test_variants_on_both_paths(variant, small_step):
    """Each variant at a small ragged size on the one-launch cluster path
    (small_step 1) and on the two-kernel path (-1)."""
    opts = {"decay_first": o.Options(decay_before_update=True), "clip_eps": o.Options(clip_eps=1e-6),
            "bf16_moments": o.Options(moments_bf16=True),
            "all": o.Options(decay_before_update=True, clip_eps=1e-6, moments_bf16=True)}[variant]
    w = WL.Workload("vp", 20_005, 3, 0.01, 4, lr=1e-2, weight_decay=0.5, max_norm=0.05)
    run_variant(w, 4, opts, small_step)


def test_all_variants_w64():
    run_variant(WL.Workload("all", 200_001, 64, 1e-3, 3, max_norm=0.5, rank_mean_step=1e-5),
                3, o.Options(decay_before_update=True, clip_eps=1e-6, moments_bf16=True))


def test_bf16_moments_footprint_and_checkpoint():
    """bf16 moments hold 8 bytes per padded parameter of state (fp32 master
    + bf16 m + bf16 v) and resume bit for bit from a bf16 checkpoint."""
    n, world = 30_011, 4
    w = WL.Workload("ck", n, world, 0.01, 6, max_norm=0.05)
    zo = z.Options(moments_bf16=True)
    hp = z.Hparams(**w.hparams())
    m0 = WL.master(w, "cuda")
    grads = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    reps = [torch.empty_like(grads[0]) for _ in range(world)]
    with z.Zero1(n, world, hp, zo) as a:
        _, padded, nbytes = a.layout()
        assert 8 * padded + 4 * padded <= nbytes <= 8 * padded + 4 * padded + 64 * 1024
        a.set_state(m0)
        for t in range(1, 7):
            a.step(WL.grads(w, t, "cuda", out=grads), reps)
        full = _moments(a, n, True)
    with z.Zero1(n, world, hp, zo) as b:
        b.set_state(m0)
        for t in range(1, 4):
            b.step(WL.grads(w, t, "cuda", out=grads), reps)
        mid = [torch.empty(n, device="cuda"), torch.empty(n, dtype=torch.bfloat16, device="cuda"),
               torch.empty(n, dtype=torch.bfloat16, device="cuda")]
        tsave = b.get_state(*mid)
    with z.Zero1(n, world, hp, zo) as c:
        c.set_state(*mid, t=tsave)
        for t in range(4, 7):
            c.step(WL.grads(w, t, "cuda", out=grads), reps)
        resumed = _moments(c, n, True)
    for x, y in zip(full, resumed):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_bf16_moments_range_checkpoint():
    """Per-shard save and load of bf16 moments (the range forms address m and
    v in 2-byte elements) resumes bit for bit."""
    n, world = 50_003, 4
    w = WL.Workload("ckr", n, world, 0.01, 6, max_norm=0.05)
    zo = z.Options(moments_bf16=True, small_step=-1)
    hp = z.Hparams(**w.hparams())
    m0 = WL.master(w, "cuda")
    grads = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    reps = [torch.empty_like(grads[0]) for _ in range(world)]
    with z.Zero1(n, world, hp, zo) as a:
        a.set_state(m0)
        for t in range(1, 7):
            a.step(WL.grads(w, t, "cuda", out=grads), reps)
        full = _moments(a, n, True)
    with z.Zero1(n, world, hp, zo) as b:
        b.set_state(m0)
        for t in range(1, 4):
            b.step(WL.grads(w, t, "cuda", out=grads), reps)
        s, _, _ = b.layout()
        saved = [np.zeros(n, np.float32), np.zeros(n, np.uint16), np.zeros(n, np.uint16)]
        for r in range(world):
            lo, hi = min(r * s, n), min((r + 1) * s, n)
            z.zero1_get_state_range(b.handle, lo, hi - lo, *[x[lo:] for x in saved])
        torch.cuda.synchronize()
        tsave = b.get_state()
    with z.Zero1(n, world, hp, zo) as c:
        c.set_state(np.zeros(n, np.float32), t=tsave)     # t only; every element is then loaded per shard
        for r in range(world):
            lo, hi = min(r * s, n), min((r + 1) * s, n)
            z.zero1_set_state_range(c.handle, lo, hi - lo, *[x[lo:] for x in saved])
        for t in range(4, 7):
            c.step(WL.grads(w, t, "cuda", out=grads), reps)
        resumed = _moments(c, n, True)
    for x, y in zip(full, resumed):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


@pytest.mark.parametrize("world,rate", [(2, 0.0), (16, 0.0), (24, 0.0), (64, 0.0), (128, 0.0), (8, 6500.0)])
def test_load_phasing_is_timing_only(world, rate):
    """The update kernel with phased loads (the built-in rule at W = 2 on the
    gradient re-read path and at W = 16, 24, 64 and 128 on the scratch path,
    an explicit device-wide rate at W = 8; 1M parameters, so the
    grid spans every SM) computes what the free-running kernel computes, bit
    for bit, and what the oracle computes with the step's clip coefficient
    injected, over three steps."""
    n = 1_000_003
    w = WL.Workload(f"phase_w{world}", n, world, 1e-3, 3, max_norm=0.5, rank_mean_step=1e-5)
    d = w.hparams()
    ohp = o.HP(**d)
    m0 = WL.master(w, "cuda")
    grads = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    ra = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    rb = [torch.empty_like(x) for x in ra]
    inj = o.State(f32(m0))
    with z.Zero1(n, world, z.Hparams(**d), z.Options(load_phase_gbs=rate)) as a, \
            z.Zero1(n, world, z.Hparams(**d), z.Options(load_phase_gbs=-1.0)) as b:
        a.set_state(m0)
        b.set_state(m0)
        for t in range(1, 4):
            WL.grads(w, t, "cuda", out=grads)
            a.step(grads, ra)
            b.step(grads, rb)
            norm_a, c_a = a.grad_norm()
            assert (norm_a, c_a) == b.grad_norm(), t
            reps_i, _, _ = o.step(inj, [u16(g) for g in grads], ohp, clip_override=np.float32(c_a))
            sa, sb = _moments(a, n, False), _moments(b, n, False)
            for x, y, ref in zip(sa, sb, (inj.master, inj.m, inj.v)):
                assert bits_equal(x, ref) and bits_equal(y, ref), t
            for r in range(world):
                assert np.array_equal(u16(ra[r]), reps_i[r]), (t, r)
                assert np.array_equal(u16(rb[r]), reps_i[r]), (t, r)
