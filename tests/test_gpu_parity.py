"""GPU path against the CPU oracle, through the C ABI.

Protocol per step (the oracle runs on host copies of the same seeded inputs):
  1. the GPU step runs; its norm and clip coefficient c are read back;
  2. the oracle runs the same step with c injected: master, m, v and every
     replica must match bit for bit (same fp32 operations in the same order);
  3. the GPU norm and c must match the oracle's own within 1e-6 relative;
  4. a free-running oracle (its own c) must agree with the GPU state within
     1e-6 relative (denominator floored at the array RMS, see gpu_util) and
     the replicas within 1 bf16 ulp.
Canaries around every caller buffer must survive.  Full-size workloads are
checked on the launch configuration the benchmark times: the exact norm by
streaming every gradient through the oracle, bit-exact state and replicas on
sampled windows (ends, shard boundaries, the ragged tail, random windows),
and equality of all W replicas everywhere.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads as WL
import zero_sharded_adamw_gb300 as z
from oracle import zero1_oracle as o
from tests.gpu_util import Guarded, bf16_ulp, bits_equal, f32, rel_err, u16

pytestmark = pytest.mark.gpu

TOL = 1e-6


def _hp(w: WL.Workload) -> tuple[z.Hparams, o.HP]:
    d = w.hparams()
    return z.Hparams(**d), o.HP(**d)


def _state(opt: z.Zero1, n: int):
    master = torch.empty(n, dtype=torch.float32, device="cuda")
    m, v = torch.empty_like(master), torch.empty_like(master)
    t = opt.get_state(master, m, v)
    torch.cuda.synchronize()
    return f32(master), f32(m), f32(v), t


def run_parity(w: WL.Workload, steps: int, *, lr_schedule=None, master0=None, opts=None, launches=None):
    """Run `steps` steps of workload `w` on the GPU and both oracles; assert
    the protocol above at every step.  Returns the final GPU state."""
    zhp, ohp = _hp(w)
    n = w.n
    m0 = WL.master(w, "cuda") if master0 is None else master0
    grads = [Guarded(n, torch.bfloat16) for _ in range(w.world)]
    reps = [Guarded(n, torch.bfloat16) for _ in range(w.world)]
    with z.Zero1(n, w.world, zhp, opts) as opt:
        if launches is not None:
            assert opt.launches_per_step() == launches
        opt.set_state(m0, None, None, 0)
        inj, free = o.State(f32(m0)), o.State(f32(m0))
        for t in range(1, steps + 1):
            if lr_schedule is not None:
                lr = lr_schedule(t)
                opt.set_lr(lr)
                ohp.lr = lr
            WL.grads(w, t, "cuda", out=[g.t for g in grads])
            opt.step([g.t for g in grads], [r.t for r in reps])
            norm_g, c_g = opt.grad_norm()
            gh = [u16(g.t) for g in grads]
            reps_i, norm_i, _ = o.step(inj, gh, ohp, clip_override=np.float32(c_g))
            reps_f, norm_f, c_f = o.step(free, gh, ohp)
            master, m, v, tg = _state(opt, n)
            assert tg == t
            # (2) bit-exact with the GPU's clip coefficient injected
            assert bits_equal(master, inj.master), f"step {t}: master differs"
            assert bits_equal(m, inj.m), f"step {t}: m differs"
            assert bits_equal(v, inj.v), f"step {t}: v differs"
            for r in range(w.world):
                assert np.array_equal(u16(reps[r].t), reps_i[r]), f"step {t}: replica {r} differs"
            # (3) norm and clip coefficient
            if math.isfinite(norm_i):
                assert abs(norm_g - norm_i) <= TOL * norm_i, (t, norm_g, norm_i)
                assert abs(float(c_g) - float(c_f)) <= TOL * float(c_f), (t, c_g, c_f)
            # (4) free-running oracle
            assert rel_err(master, free.master) <= TOL
            assert rel_err(m, free.m) <= TOL
            assert rel_err(v, free.v) <= TOL
            assert bf16_ulp(u16(reps[0].t), reps_f[0]) <= 1
        assert all(b.intact() for b in grads + reps), "a canary was overwritten"
        return _state(opt, n)


# ----------------------------------------------------------- small cases

def test_tiny_ten_steps():
    """W = 4, N = 4096, 10 steps with fresh gradients (clip inactive)."""
    run_parity(WL.WORKLOADS["tiny"], 10)


@pytest.mark.parametrize("path", ["one_launch", "two_kernels"])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 5, 8, 16, 64])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 63, 65, 4097, 256 * 8 * 3 + 5])
def test_shapes(n, world, path):
    """Ragged and tiny sizes, every kernel specialisation, clip active, on
    the one-launch cluster path and on the two-kernel path."""
    w = WL.Workload(f"shape_{n}_{world}", n, world, 0.05, 3, max_norm=0.01)
    small = 1 if path == "one_launch" else -1
    run_parity(w, 3, opts=z.Options(small_step=small), launches=1 if small == 1 else 2)


@pytest.mark.parametrize("n", [16_383, 16_384, 16_391, 32_768, 32_775, 65_535, 65_536])
def test_one_launch_vector_counts(n):
    """The one-launch path at the edges of 1, 2 and 4 vectors per thread
    (16,384 / 32,768 / 65,536 parameters), ragged tails included."""
    w = WL.Workload(f"small_{n}", n, 8, 0.05, 2, max_norm=0.01)
    run_parity(w, 2, opts=z.Options(small_step=1), launches=1)


def test_one_launch_selection():
    """Automatic choice: one launch while n <= 32,768 and (4W+24)*n <= 6 MiB;
    a forced one-launch handle past 65,536 parameters keeps two kernels."""
    for n, world, want in ((4096, 4, 1), (32_768, 8, 1), (16_384, 64, 1), (32_768, 64, 2), (32_769, 1, 2),
                           (65_536, 8, 2), (1_000_000, 8, 2)):
        with z.Zero1(n, world) as opt:
            assert opt.launches_per_step() == want, (n, world)
    with z.Zero1(65_537, 2, None, z.Options(small_step=1)) as opt:
        assert opt.launches_per_step() == 2
    with z.Zero1(16, 2, None, z.Options(small_step=-1)) as opt:
        assert opt.launches_per_step() == 2
    with pytest.raises(z.Zero1Error):
        z.Zero1(16, 2, None, z.Options(small_step=2))


@pytest.mark.parametrize("name,n", [("gpt2_small", 2_000_003), ("ragged_1p3b", 1_000_003),
                                    ("state_7b", 1_000_003), ("stress_w64", 200_001)])
def test_recipe_for_its_configured_steps(name, n):
    """Each large recipe (its W, gradient distribution, outliers, rank mean
    offsets and clip threshold) at a size the oracle runs in seconds, for the
    number of steps the recipe is configured with (20, 10, 5 and 5): every
    step bit-exact with the GPU's clip coefficient injected, and the GPU
    state within 1e-6 of a free-running oracle after each step."""
    w = WL.WORKLOADS[name].with_n(n)
    run_parity(w, w.steps)


def test_multi_tile_ragged_without_clipping():
    run_parity(WL.Workload("noclip", 1_000_003, 8, 1e-3, 3, max_norm=0.0), 3)


def test_lr_schedule():
    """zero1_set_lr between steps equals the oracle with the same per-step lr."""
    w = WL.Workload("sched", 50_000, 4, 0.01, 6)
    run_parity(w, 6, lr_schedule=lambda t: 1e-3 * (0.5 + 0.5 * math.cos(math.pi * t / 6)))


def test_worked_example_norm():
    """The pages' 4-rank inputs (arange(4) + rank) as gradients: the averaged
    gradient is [1.5, 2.5, 3.5, 4.5] and its norm sqrt(41)."""
    x = [torch.tensor([0.0, 1, 2, 3], device="cuda").add(r).to(torch.bfloat16) for r in range(4)]
    reps = [torch.zeros(4, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    with z.Zero1(4, 4, z.Hparams(max_norm=0.0)) as opt:
        opt.step(x, reps)
        norm, c = opt.grad_norm()
    assert abs(norm - math.sqrt(41.0)) <= 1e-15 * math.sqrt(41.0)
    assert c == 1.0


def test_bf16_master_example():
    """The pages' mixed-precision example through the library: 1000 steps of
    AdamW with beta1 = beta2 = eps = wd = 0 and lr = 1e-3 subtract fp32(1e-3)
    from a master of 1.0 each step; it ends at numpy's float32 value
    (printed as 0.0), while the replicas follow it in bf16."""
    n, world = 4096, 2
    one = torch.ones(n, dtype=torch.bfloat16, device="cuda")
    reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    hp = z.Hparams(lr=1e-3, beta1=0.0, beta2=0.0, eps=0.0, weight_decay=0.0, max_norm=0.0)
    ref = np.float32(1.0)
    for _ in range(1000):
        ref = np.float32(ref - np.float32(1e-3))
    with z.Zero1(n, world, hp) as opt:
        opt.set_state(torch.ones(n, device="cuda"))
        for _ in range(1000):
            opt.step([one] * world, reps)
        master, _, _, t = _state(opt, n)
    assert t == 1000
    assert (master == ref).all() and round(float(master[0]), 4) == 0.0
    assert np.array_equal(u16(reps[1]), o.f32_to_bf16(master))


# --------------------------------------------------- semantics and errors

@pytest.mark.parametrize("n", [30_011, 300_007])      # one-launch and two-kernel path
def test_checkpoint_resume_is_exact(n):
    """10 steps == 5 steps, save (per-rank shard ranges, to host), destroy,
    create, load, 5 steps -- bit for bit ("a checkpoint carries m, v, t")."""
    w = WL.Workload("ckpt", n, 4, 0.01, 10, max_norm=0.05)
    zhp, _ = _hp(w)
    m0 = WL.master(w, "cuda")
    grads = [torch.empty(w.n, dtype=torch.bfloat16, device="cuda") for _ in range(w.world)]
    reps_a = [torch.empty_like(grads[0]) for _ in range(w.world)]
    reps_b = [torch.empty_like(grads[0]) for _ in range(w.world)]
    with z.Zero1(w.n, w.world, zhp) as a:
        a.set_state(m0)
        for t in range(1, 11):
            a.step(WL.grads(w, t, "cuda", out=grads), reps_a)
        full = _state(a, w.n)
    b = z.Zero1(w.n, w.world, zhp)
    b.set_state(m0)
    for t in range(1, 6):
        b.step(WL.grads(w, t, "cuda", out=grads), reps_b)
    s, _, _ = b.layout()
    saved = [np.empty(w.n, np.float32) for _ in range(3)]
    for r in range(w.world):          # each rank saves its own shard
        lo, hi = min(r * s, w.n), min((r + 1) * s, w.n)
        z.zero1_get_state_range(b.handle, lo, hi - lo, *[x[lo:] for x in saved])
    torch.cuda.synchronize()
    t_saved = b.get_state()
    b.close()
    with z.Zero1(w.n, w.world, zhp) as c:
        c.set_state(*saved, t=t_saved)
        for t in range(6, 11):
            c.step(WL.grads(w, t, "cuda", out=grads), reps_b)
        resumed = _state(c, w.n)
    for x, y in zip(full[:3], resumed[:3]):
        assert bits_equal(x, y)
    assert full[3] == resumed[3] == 10
    assert all(torch.equal(x, y) for x, y in zip(reps_a, reps_b))


def test_deterministic():
    w = WL.Workload("det", 777_777, 8, 1e-3, 3, max_norm=0.01)
    zhp, _ = _hp(w)
    out = []
    for _ in range(2):
        grads = WL.grads(w, 1, "cuda")
        reps = [torch.empty_like(grads[0]) for _ in range(w.world)]
        with z.Zero1(w.n, w.world, zhp) as opt:
            opt.set_state(WL.master(w, "cuda"))
            for t in range(1, 4):
                opt.step(WL.grads(w, t, "cuda", out=grads), reps)
            out.append((opt.grad_norm(), _state(opt, w.n), u16(reps[0])))
    (n1, s1, r1), (n2, s2, r2) = out
    assert n1 == n2
    assert all(bits_equal(a, b) for a, b in zip(s1[:3], s2[:3]))
    assert np.array_equal(r1, r2)


@pytest.mark.parametrize("small_step", [1, -1])
@pytest.mark.parametrize("bad", ["inf", "nan"])
def test_nonfinite_gradient_propagates(bad, small_step):
    """An inf or NaN in one rank's gradient: the norm is not finite and the
    state follows the oracle's IEEE propagation (NaN positions match), on
    the one-launch and the two-kernel path."""
    w = WL.Workload("nf", 4099, 4, 0.01, 1)
    zhp, ohp = _hp(w)
    grads = WL.grads(w, 1, "cuda")
    grads[2][17] = float(bad)
    reps = [torch.empty_like(grads[0]) for _ in range(w.world)]
    m0 = WL.master(w, "cuda")
    with z.Zero1(w.n, w.world, zhp, z.Options(small_step=small_step)) as opt:
        opt.set_state(m0)
        opt.step(grads, reps)
        norm, c = opt.grad_norm()
        master, m, v, _ = _state(opt, w.n)
    st = o.State(f32(m0))
    reps_o, norm_o, c_o = o.step(st, [u16(g) for g in grads], ohp)
    assert not math.isfinite(norm) and not math.isfinite(norm_o)
    assert (math.isnan(norm) == math.isnan(norm_o))
    assert bits_equal(np.array([c], np.float32), np.array([c_o], np.float32)) or (math.isnan(c) and np.isnan(c_o))
    for a, b in ((master, st.master), (m, st.m), (v, st.v)):
        assert np.array_equal(np.isnan(a), np.isnan(b))
        ok = ~np.isnan(b)
        assert bits_equal(a[ok], b[ok])


def test_argument_errors():
    n, world = 1000, 4
    grads = [torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    reps = [torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    with z.Zero1(n, world) as opt:
        with pytest.raises(z.Zero1Error) as e:
            opt.step([g[1:] for g in grads], reps)          # 2-byte offset
        assert e.value.code == -2
        with pytest.raises(z.Zero1Error) as e:
            opt.step([0] + grads[1:], reps)
        assert e.value.code == -1
        assert opt.get_state() == 0                           # t unchanged by failed steps
        with pytest.raises(z.Zero1Error):
            z.zero1_get_state_range(opt.handle, n - 5, 6, np.empty(6, np.float32))
    with pytest.raises(z.Zero1Error) as e:
        z.zero1_create(n, z.ZERO1_MAX_WORLD + 1)
    assert e.value.code == -1


@pytest.mark.parametrize("small_step", [1, -1])
def test_max_world(small_step):
    """W = 512 (the runtime-W kernels with the largest pointer tables) on the
    one-launch and the two-kernel path."""
    w = WL.Workload("wmax", 1003, z.ZERO1_MAX_WORLD, 0.01, 2, max_norm=0.5)
    run_parity(w, 2, opts=z.Options(small_step=small_step), launches=1 if small_step == 1 else 2)


def test_layout_and_footprint():
    """Device footprint: 12 bytes of optimizer state per padded parameter
    (fp32 master + m + v, the pages' K = 12), plus the fp32 reduce-scatter
    scratch for W >= 3 and a few KB of partials and status."""
    for n, world in ((1_000_000, 8), (1_000_000, 2), (4096, 4)):
        with z.Zero1(n, world) as opt:
            s, padded, nbytes = opt.layout()
            assert (s, padded) == z.zero1_shard_plan(n, world)
            state = 12 * padded
            scratch = 4 * padded if world >= 3 else 0
            assert state + scratch <= nbytes <= state + scratch + 64 * 1024


def test_profile_events():
    """zero1_profile_read returns one positive (K1, K2) pair per profiled
    step, agreeing with zero1_profile_stop's sums; steps past the capacity
    are not recorded."""
    w = WL.Workload("prof", 1_000_003, 8, 0.001, 1)
    zhp, _ = _hp(w)
    g = WL.grads(w, 1, "cuda")
    reps = [torch.empty_like(g[0]) for _ in range(w.world)]
    with z.Zero1(w.n, w.world, zhp) as opt:
        opt.set_state(WL.master(w, "cuda"))
        z.zero1_profile_start(opt.handle, 3)
        for _ in range(5):
            opt.step(g, reps)
        rs, upd = z.zero1_profile_read(opt.handle, 8)
        assert len(rs) == len(upd) == 3
        assert all(x > 0 for x in rs + upd)
        assert z.zero1_profile_read(opt.handle, 2)[0] == rs[:2]
        a, b, k = z.zero1_profile_stop(opt.handle)
        assert k == 3
        assert math.isclose(a, sum(rs), rel_tol=1e-5) and math.isclose(b, sum(upd), rel_tol=1e-5)
        with pytest.raises(z.Zero1Error):
            z.zero1_profile_read(opt.handle, 1)


def test_step_host_matches_device_step():
    """The host-buffer entry point equals the device entry point."""
    w = WL.Workload("host", 100_003, 4, 0.01, 2, max_norm=0.05)
    zhp, _ = _hp(w)
    m0 = WL.master(w, "cuda")
    outs = []
    for use_host in (False, True):
        with z.Zero1(w.n, w.world, zhp) as opt:
            opt.set_state(m0)
            for t in range(1, 3):
                g = WL.grads(w, t, "cuda")
                if use_host:
                    hg = [x.cpu().pin_memory() for x in g]
                    hp_ = [torch.empty(w.n, dtype=torch.bfloat16).pin_memory() for _ in range(w.world)]
                    opt.step_host(hg, hp_)
                    reps = hp_
                else:
                    reps = [torch.empty_like(g[0]) for _ in range(w.world)]
                    opt.step(g, reps)
            outs.append(([u16(r) for r in reps], _state(opt, w.n)))
    (ra, sa), (rb, sb) = outs
    assert all(np.array_equal(a, b) for a, b in zip(ra, rb))
    assert all(bits_equal(a, b) for a, b in zip(sa[:3], sb[:3]))


def test_step_host_async_matches_step_host():
    """The pipelined host entry point gives the blocking one's results, step
    by step: four steps with a fresh output buffer set per step (each read
    after the final sync), then two with one shared set."""
    w = WL.Workload("host_async", 100_003, 4, 0.01, 2, max_norm=0.05)
    zhp, _ = _hp(w)
    m0 = WL.master(w, "cuda")
    steps = 6
    hgs = [[x.cpu().pin_memory() for x in WL.grads(w, t, "cuda")] for t in range(1, steps + 1)]
    fresh = lambda: [torch.empty(w.n, dtype=torch.bfloat16).pin_memory() for _ in range(w.world)]
    want = []
    with z.Zero1(w.n, w.world, zhp) as opt:
        opt.set_state(m0)
        for t in range(steps):
            out = fresh()
            opt.step_host(hgs[t], out)
            want.append([u16(r) for r in out])
        want_state = _state(opt, w.n)
    with z.Zero1(w.n, w.world, zhp) as opt:
        opt.set_state(m0)
        outs = [fresh() for _ in range(4)]
        for t in range(4):
            opt.step_host_async(hgs[t], outs[t])
        opt.host_sync()
        for t in range(4):
            assert all(np.array_equal(u16(a), b) for a, b in zip(outs[t], want[t])), t
        shared = fresh()
        for t in range(4, steps):
            opt.step_host_async(hgs[t], shared)
        opt.host_sync()
        assert all(np.array_equal(u16(a), b) for a, b in zip(shared, want[steps - 1]))
        got_state = _state(opt, w.n)
    assert all(bits_equal(a, b) for a, b in zip(got_state[:3], want_state[:3]))


@pytest.mark.parametrize("world", [2, 4])          # fp32 scratch kept by the handle (W >= 3) or by the host path
def test_step_host_chunked_against_oracle_and_buckets(world):
    """The host-buffer step cut into 16 chunks (the last one ragged): each
    step is bit for bit the oracle's with the step's clip coefficient
    injected, its norm within 1e-6 of the oracle's, and the result (norm
    included) is the device bucketed step's with the same cut."""
    n, chunk = 1_000_003, 65_536
    w = WL.Workload(f"host_chunks_w{world}", n, world, 0.01, 3, max_norm=0.05)
    zhp, ohp = _hp(w)
    m0 = WL.master(w, "cuda")
    cuts = [(lo, min(chunk, n - lo)) for lo in range(0, n, chunk)]
    assert len(cuts) == 16
    inj = o.State(f32(m0))
    reps_d = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    with z.Zero1(n, world, zhp, z.Options(host_chunk=chunk)) as a, z.Zero1(n, world, zhp) as b:
        a.set_state(m0)
        b.set_state(m0)
        for t in range(1, w.steps + 1):
            g = WL.grads(w, t, "cuda")
            hg = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True).copy_(x) for x in g]
            hr = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(world)]
            a.step_host(hg, hr)
            norm_a, c_a = a.grad_norm()
            z.zero1_bucket_begin(b.handle)
            for lo, cnt in cuts:
                z.zero1_bucket_reduce(b.handle, lo, cnt, [x[lo:lo + cnt] for x in g])
            z.zero1_bucket_finish(b.handle, reps_d)
            norm_b, c_b = b.grad_norm()
            assert norm_a == norm_b and c_a == c_b, (t, norm_a, norm_b)
            reps_i, norm_i, _ = o.step(inj, [u16(x) for x in g], ohp, clip_override=np.float32(c_a))
            assert abs(norm_a - norm_i) <= TOL * norm_i
            sa, sb = _state(a, n), _state(b, n)
            assert sa[3] == sb[3] == t
            for x, y, ref in zip(sa[:3], sb[:3], (inj.master, inj.m, inj.v)):
                assert bits_equal(x, ref) and bits_equal(y, ref), t
            for r in range(world):
                assert np.array_equal(u16(hr[r]), reps_i[r]), (t, r)
                assert np.array_equal(u16(reps_d[r]), reps_i[r]), (t, r)


@pytest.mark.parametrize("opts", [dict(moments_bf16=True), dict(decay_before_update=True, clip_eps=1e-6)])
def test_step_host_chunked_variants_match_buckets(opts):
    """Step variants through the chunked host path (11 chunks, the last
    ragged) equal the device bucketed step with the same cut, bit for bit,
    norm included, over three steps."""
    n, world, chunk = 700_001, 4, 65_536
    w = WL.Workload("host_var", n, world, 0.01, 3, max_norm=0.05)
    zhp, _ = _hp(w)
    m0 = WL.master(w, "cuda")
    cuts = [(lo, min(chunk, n - lo)) for lo in range(0, n, chunk)]
    mdt = torch.bfloat16 if opts.get("moments_bf16") else torch.float32
    reps_d = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    with z.Zero1(n, world, zhp, z.Options(host_chunk=chunk, **opts)) as a, \
            z.Zero1(n, world, zhp, z.Options(**opts)) as b:
        a.set_state(m0)
        b.set_state(m0)
        for t in range(1, w.steps + 1):
            g = WL.grads(w, t, "cuda")
            hg = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True).copy_(x) for x in g]
            hr = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(world)]
            a.step_host(hg, hr)
            z.zero1_bucket_begin(b.handle)
            for lo, cnt in cuts:
                z.zero1_bucket_reduce(b.handle, lo, cnt, [x[lo:lo + cnt] for x in g])
            z.zero1_bucket_finish(b.handle, reps_d)
            assert a.grad_norm() == b.grad_norm()
            sa, sb = [], []
            for opt, out in ((a, sa), (b, sb)):
                master = torch.empty(n, device="cuda")
                m, v = torch.empty(n, dtype=mdt, device="cuda"), torch.empty(n, dtype=mdt, device="cuda")
                opt.get_state(master, m, v)
                torch.cuda.synchronize()
                out += [master.view(torch.int32).cpu(), m.view(torch.int16 if mdt == torch.bfloat16 else torch.int32).cpu(),
                        v.view(torch.int16 if mdt == torch.bfloat16 else torch.int32).cpu()]
            assert all(torch.equal(x, y) for x, y in zip(sa, sb)), t
            for r in range(world):
                assert np.array_equal(u16(hr[r]), u16(reps_d[r])), (t, r)


def test_step_host_offsets_past_4_gib():
    """The host-buffer step at 2.2e9 parameters (W = 2, the default chunk):
    byte offsets into the host buffers pass 2^32.  Two steps equal the
    device bucketed step with the same cut bit for bit (state, every
    replica, norm)."""
    n, world = 2_200_000_013, 2
    free, _ = torch.cuda.mem_get_info()
    if free < 80e9:
        pytest.skip(f"needs ~80 GB of free device memory, {free / 1e9:.0f} GB free")
    w = WL.Workload("host_big", n, world, 1e-3, 2)
    zhp, _ = _hp(w)
    cuts = None
    reps_d = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    hg = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(world)]
    hr = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(world)]
    with z.Zero1(n, world, zhp) as a, z.Zero1(n, world, zhp) as b:
        m0 = WL.master(w, "cuda")
        a.set_state(m0)
        b.set_state(m0)
        del m0
        for t in range(1, w.steps + 1):
            g = WL.grads(w, t, "cuda")
            for x, y in zip(hg, g):
                x.copy_(y)
            a.step_host(hg, hr)
            if cuts is None:                        # the host path's own cut (256 MiB slots: 64M parameters at W = 2)
                chunk = (256 << 20) // (2 * world) // 2048 * 2048
                cuts = [(lo, min(chunk, n - lo)) for lo in range(0, n, chunk)]
            z.zero1_bucket_begin(b.handle)
            for lo, cnt in cuts:
                z.zero1_bucket_reduce(b.handle, lo, cnt, [x[lo:lo + cnt] for x in g])
            z.zero1_bucket_finish(b.handle, reps_d)
            del g
            assert a.grad_norm() == b.grad_norm(), t
            for r in range(world):
                assert torch.equal(hr[r].view(torch.int16), reps_d[r].view(torch.int16).cpu()), (t, r)
        for lo in (0, n // 2, n - 4096):            # state on windows, including past the 4 GiB byte offset
            xs = [np.empty(4096, np.float32) for _ in range(6)]
            z.zero1_get_state_range(a.handle, lo, 4096, *xs[:3])
            z.zero1_get_state_range(b.handle, lo, 4096, *xs[3:])
            torch.cuda.synchronize()
            assert all(bits_equal(xs[i], xs[i + 3]) for i in range(3)), lo


def test_step_host_async_chunked_pipelined():
    """Six pipelined host-buffer steps over 16 chunks (step t's downloads
    overlap step t+1's uploads) equal six blocking ones bit for bit, each
    step's replicas in its own host buffers; a device step enqueued right
    after them without zero1_host_sync is ordered after them; a capturable
    handle's device step counter advances once per step."""
    n, world, chunk, steps = 1_000_003, 4, 65_536, 6
    w = WL.Workload("host_pipe", n, world, 0.01, steps, max_norm=0.05)
    zhp, _ = _hp(w)
    m0 = WL.master(w, "cuda")
    hgs = [[torch.empty(n, dtype=torch.bfloat16, pin_memory=True).copy_(x) for x in WL.grads(w, t, "cuda")]
           for t in range(1, steps + 1)]
    g_last = WL.grads(w, steps + 1, "cuda")
    fresh = lambda: [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(world)]
    results = []
    for capturable, pipelined in ((False, False), (False, True), (True, True)):
        outs = [fresh() for _ in range(steps)]
        reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
        with z.Zero1(n, world, zhp, z.Options(host_chunk=chunk, capturable=capturable)) as opt:
            opt.set_state(m0)
            for t in range(steps):
                (opt.step_host_async if pipelined else opt.step_host)(hgs[t], outs[t])
            opt.step(g_last, reps)             # ordered after the host steps by the handle itself
            st = _state(opt, n)
            opt.host_sync()
            assert st[3] == steps + 1
            results.append(([[u16(r) for r in out] for out in outs], st, [u16(r) for r in reps]))
    (outs0, st0, reps0) = results[0]
    for outs, st, reps in results[1:]:
        for t in range(steps):
            assert all(np.array_equal(a, b) for a, b in zip(outs[t], outs0[t])), t
        assert all(bits_equal(a, b) for a, b in zip(st[:3], st0[:3]))
        assert all(np.array_equal(a, b) for a, b in zip(reps, reps0))


@pytest.mark.parametrize("n,world,chunk", [(1, 1, 0), (2047, 3, 0), (5000, 64, 2048), (130_001, 8, 0)])
def test_step_host_edge_shapes(n, world, chunk):
    """The host-buffer step at the shapes the other host tests leave out:
    one parameter on one rank, n below one chunk (the default chunk, or
    2048 parameters at W = 64, so three chunks with a ragged last one),
    W = 64.  Two steps: state and every replica bit for bit the oracle's
    with the step's clip coefficient injected, the norm within 1e-6 of the
    oracle's, and norm and replicas equal to the device bucketed step with
    the host path's cut."""
    w = WL.Workload(f"host_edge_{n}_{world}", n, world, 0.01, 2, max_norm=0.05)
    zhp, ohp = _hp(w)
    m0 = WL.master(w, "cuda")
    step = chunk or n
    cuts = [(lo, min(step, n - lo)) for lo in range(0, n, step)]
    inj = o.State(f32(m0))
    reps_d = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    with z.Zero1(n, world, zhp, z.Options(host_chunk=chunk)) as a, z.Zero1(n, world, zhp) as b:
        a.set_state(m0)
        b.set_state(m0)
        for t in range(1, w.steps + 1):
            g = WL.grads(w, t, "cuda")
            hg = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True).copy_(x) for x in g]
            hr = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(world)]
            a.step_host(hg, hr)
            norm_a, c_a = a.grad_norm()
            z.zero1_bucket_begin(b.handle)
            for lo, cnt in cuts:
                z.zero1_bucket_reduce(b.handle, lo, cnt, [x[lo:lo + cnt] for x in g])
            z.zero1_bucket_finish(b.handle, reps_d)
            assert (norm_a, c_a) == b.grad_norm(), t
            reps_i, norm_i, _ = o.step(inj, [u16(x) for x in g], ohp, clip_override=np.float32(c_a))
            assert abs(norm_a - norm_i) <= TOL * norm_i
            sa = _state(a, n)
            assert sa[3] == t
            for x, ref in zip(sa[:3], (inj.master, inj.m, inj.v)):
                assert bits_equal(x, ref), t
            for r in range(world):
                assert np.array_equal(u16(hr[r]), reps_i[r]), (t, r)
                assert np.array_equal(u16(reps_d[r]), reps_i[r]), (t, r)


# --------------------------------------------------------- full sizes

def _windows(n: int, world: int, shard: int, rng, width=4096, n_random=8):
    cuts = [(0, min(width, n)), (max(0, n - width), n)]
    for r in range(1, world):
        b = r * shard
        if b < n:
            cuts.append((max(0, b - width // 2), min(n, b + width // 2)))
    for _ in range(n_random):
        lo = int(rng.integers(0, max(1, n - width)))
        cuts.append((lo, min(n, lo + width)))
    return sorted(set(cuts))


def run_full_size(w: WL.Workload, steps: int = 1):
    """Full-size check: exact norm via the streaming oracle, bit-exact state
    and replicas on sampled windows, all replicas equal."""
    zhp, ohp = _hp(w)
    rng = np.random.default_rng(2024)
    m0 = WL.master(w, "cuda")
    with z.Zero1(w.n, w.world, zhp) as opt:
        opt.set_state(m0)
        shard, _, _ = opt.layout()
        wins = _windows(w.n, w.world, shard, rng)
        prev = {lo_hi: (f32(m0[lo_hi[0]:lo_hi[1]]), np.zeros(lo_hi[1] - lo_hi[0], np.float32),
                        np.zeros(lo_hi[1] - lo_hi[0], np.float32)) for lo_hi in wins}
        del m0
        torch.cuda.empty_cache()
        grads = [torch.empty(w.n, dtype=torch.bfloat16, device="cuda") for _ in range(w.world)]
        reps = [torch.empty(w.n, dtype=torch.bfloat16, device="cuda") for _ in range(w.world)]
        for t in range(1, steps + 1):
            WL.grads(w, t, "cuda", out=grads)
            opt.step(grads, reps)
            norm_g, c_g = opt.grad_norm()
            # exact norm: stream every gradient through the oracle in order
            acc = o.NormAccumulator()
            chunk = 1 << 25
            for lo in range(0, w.n, chunk):
                hi = min(w.n, lo + chunk)
                acc.add(o.rs_mean_range([u16(g[lo:hi]) for g in grads], w.world))
            norm_o = acc.value()
            c_o = o.clip_coef(norm_o, w.max_norm)
            assert abs(norm_g - norm_o) <= TOL * norm_o, (norm_g, norm_o)
            assert abs(float(c_g) - float(c_o)) <= TOL * float(c_o), (c_g, c_o)
            sc = o.step_scalars(ohp, w.world, t)
            for (lo, hi) in wins:
                pm, pmm, pv = (x.copy() for x in prev[(lo, hi)])
                gh = o.rs_mean_range([u16(g[lo:hi]) for g in grads], w.world)
                o.adamw_range(pm, pmm, pv, gh, np.float32(c_g), sc)
                gm, gmm, gv = (np.empty(hi - lo, np.float32) for _ in range(3))
                z.zero1_get_state_range(opt.handle, lo, hi - lo, gm, gmm, gv)
                torch.cuda.synchronize()
                assert bits_equal(gm, pm) and bits_equal(gmm, pmm) and bits_equal(gv, pv), (t, lo, hi)
                ref_b = o.f32_to_bf16(pm)
                for r in range(w.world):
                    assert np.array_equal(u16(reps[r][lo:hi]), ref_b), (t, lo, hi, r)
                prev[(lo, hi)] = (gm, gmm, gv)
            for r in range(1, w.world):
                assert torch.equal(reps[r], reps[0])
        del grads, reps
    torch.cuda.empty_cache()


def test_gpt2_small_full_size_whole_arrays():
    """GPT-2-small parameter list (124,355,328, W = 8), 2 steps, every entry
    compared with the oracle (state and all replicas)."""
    w = WL.WORKLOADS["gpt2_small"]
    st = run_parity(w, 2)
    assert st[3] == 2


def test_gpt2_small_full_size_windows():
    run_full_size(WL.WORKLOADS["gpt2_small"], steps=3)


def test_ragged_1p3b_full_size():
    run_full_size(WL.WORKLOADS["ragged_1p3b"], steps=2)


def test_stress_w64_full_size():
    run_full_size(WL.WORKLOADS["stress_w64"], steps=1)


def test_state_7b_full_size():
    free, _ = torch.cuda.mem_get_info()
    w = WL.WORKLOADS["state_7b"]
    need = (12 + 4 * w.world + 4) * w.n + (8 << 30)
    if free < need:
        pytest.skip(f"needs {need / 1e9:.0f} GB of free device memory, {free / 1e9:.0f} GB free")
    run_full_size(w, steps=2)
