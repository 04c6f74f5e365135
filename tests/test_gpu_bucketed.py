"""The ZeRO-2-style bucketed step (zero1_bucket_begin / _reduce / _finish).

Buckets arrive in backward order (last parameters first), each from its own
small gradient buffers (the full gradient is never materialised), on a side
stream.  With the GPU's clip coefficient injected the oracle's step must
match bit for bit; the norm within 1e-6 of the oracle's.  With clipping off
(c = 1 exactly on both paths) the bucketed step must equal zero1_step bit
for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as WL
import zero_sharded_adamw_gb300 as z
from oracle import zero1_oracle as o
from tests.gpu_util import bits_equal, f32, u16

pytestmark = pytest.mark.gpu


def _buckets(n: int, rng, mean: int) -> list[tuple[int, int]]:
    cuts, off = [], 0
    while off < n:
        size = int(rng.integers(1, 2 * mean)) * 8
        cuts.append((off, min(size, n - off)))
        off += size
    return cuts[::-1]                      # backward order: last layers first


def _bucketed_step(opt: z.Zero1, grads: list[torch.Tensor], reps, cuts, side: torch.cuda.Stream):
    z.zero1_bucket_begin(opt.handle)
    main = torch.cuda.current_stream()
    side.wait_stream(main)
    keep = []
    with torch.cuda.stream(side):
        for off, cnt in cuts:
            bucket = [g[off:off + cnt].clone() for g in grads]     # the rank buckets of this layer
            keep.append(bucket)
            z.zero1_bucket_reduce(opt.handle, off, cnt, bucket, side)
    main.wait_stream(side)
    z.zero1_bucket_finish(opt.handle, reps, main)
    torch.cuda.synchronize()


def _state(opt: z.Zero1, n: int):
    m = torch.empty(n, device="cuda")
    mm, vv = torch.empty_like(m), torch.empty_like(m)
    opt.get_state(m, mm, vv)
    torch.cuda.synchronize()
    return f32(m), f32(mm), f32(vv)


@pytest.mark.parametrize("n,world,mean", [(1_000_003, 8, 4000), (65_541, 2, 300), (4099, 4, 37), (200_001, 64, 2000)])
def test_bucketed_matches_oracle(n, world, mean):
    w = WL.Workload("bk", n, world, 0.02, 3, max_norm=0.05)
    d = w.hparams()
    ohp = o.HP(**d)
    rng = np.random.default_rng(n + world)
    side = torch.cuda.Stream()
    m0 = WL.master(w, "cuda")
    reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    st = o.State(f32(m0))
    with z.Zero1(n, world, z.Hparams(**d)) as opt:
        opt.set_state(m0)
        for t in range(1, 4):
            grads = WL.grads(w, t, "cuda")
            _bucketed_step(opt, grads, reps, _buckets(n, rng, mean), side)
            norm, c = opt.grad_norm()
            reps_o, norm_o, _ = o.step(st, [u16(g) for g in grads], ohp, clip_override=np.float32(c))
            assert abs(norm - norm_o) <= 1e-6 * norm_o
            master, m, v = _state(opt, n)
            assert bits_equal(master, st.master) and bits_equal(m, st.m) and bits_equal(v, st.v)
            for r in range(world):
                assert np.array_equal(u16(reps[r]), reps_o[r])
        assert opt.get_state() == 3


def test_bucketed_equals_plain_step_without_clipping():
    n, world = 777_777, 8
    w = WL.Workload("eq", n, world, 0.02, 3, max_norm=0.0)
    hp = z.Hparams(**w.hparams())
    rng = np.random.default_rng(5)
    side = torch.cuda.Stream()
    m0 = WL.master(w, "cuda")
    ra = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    rb = [torch.empty_like(ra[0]) for _ in range(world)]
    with z.Zero1(n, world, hp) as a, z.Zero1(n, world, hp) as b:
        a.set_state(m0)
        b.set_state(m0)
        for t in range(1, 4):
            grads = WL.grads(w, t, "cuda")
            a.step(grads, ra)
            _bucketed_step(b, grads, rb, _buckets(n, rng, 3000), side)
        for x, y in zip(_state(a, n), _state(b, n)):
            assert bits_equal(x, y)
        assert all(torch.equal(x, y) for x, y in zip(ra, rb))


def test_bucketed_with_bf16_moments_and_torch_order():
    n, world = 300_007, 4
    w = WL.Workload("var", n, world, 0.02, 2, max_norm=0.05)
    d = w.hparams()
    opts = o.Options(decay_before_update=True, clip_eps=1e-6, moments_bf16=True)
    rng = np.random.default_rng(9)
    side = torch.cuda.Stream()
    m0 = WL.master(w, "cuda")
    reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    st = o.state_ex(f32(m0), opts)
    with z.Zero1(n, world, z.Hparams(**d), z.Options(True, 1e-6, True)) as opt:
        opt.set_state(m0)
        for t in range(1, 3):
            grads = WL.grads(w, t, "cuda")
            _bucketed_step(opt, grads, reps, _buckets(n, rng, 1000), side)
            _, c = opt.grad_norm()
            reps_o, _, _ = o.step_ex(st, [u16(g) for g in grads], o.HP(**d), opts, clip_override=np.float32(c))
            master = torch.empty(n, device="cuda")
            m = torch.empty(n, dtype=torch.bfloat16, device="cuda")
            v = torch.empty_like(m)
            opt.get_state(master, m, v)
            torch.cuda.synchronize()
            assert bits_equal(f32(master), st.master)
            assert np.array_equal(u16(m), st.m) and np.array_equal(u16(v), st.v)
            assert np.array_equal(u16(reps[0]), reps_o[0])


def test_bucket_errors():
    n, world = 1000, 2
    g = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    with z.Zero1(n, world) as opt:
        with pytest.raises(z.Zero1Error):
            z.zero1_bucket_reduce(opt.handle, 0, n, g)            # no open step
        with pytest.raises(z.Zero1Error):
            z.zero1_bucket_finish(opt.handle, g)
        z.zero1_bucket_begin(opt.handle)
        with pytest.raises(z.Zero1Error):
            z.zero1_bucket_begin(opt.handle)                      # already open
        with pytest.raises(z.Zero1Error):
            opt.step(g, g)                                        # plain step refused while open
        with pytest.raises(z.Zero1Error):
            z.zero1_bucket_reduce(opt.handle, 4, 8, g)            # offset not a multiple of 8
        with pytest.raises(z.Zero1Error):
            z.zero1_bucket_reduce(opt.handle, 992, 16, g)         # past n
        z.zero1_bucket_reduce(opt.handle, 0, 496, g)
        z.zero1_bucket_reduce(opt.handle, 504, 496, g)            # gap at [496, 504)
        with pytest.raises(z.Zero1Error) as e:
            z.zero1_bucket_finish(opt.handle, g)
        assert "exactly once" in str(e.value)
        assert opt.get_state() == 0                               # abandoned: t unchanged
        z.zero1_bucket_begin(opt.handle)                          # a fresh step can start
        z.zero1_bucket_reduce(opt.handle, 0, 1000, g)
        z.zero1_bucket_finish(opt.handle, g)
        torch.cuda.synchronize()
        assert opt.get_state() == 1


def _bucketed_update_step(opt: z.Zero1, grads, reps, cuts, side: torch.cuda.Stream):
    """zero1_bucket_update per bucket on a side stream (clipping off), then
    zero1_bucket_finish with no replica pointers."""
    z.zero1_bucket_begin(opt.handle)
    main = torch.cuda.current_stream()
    side.wait_stream(main)
    keep = []
    with torch.cuda.stream(side):
        for off, cnt in cuts:
            bucket = [g[off:off + cnt].clone() for g in grads]
            keep.append(bucket)
            z.zero1_bucket_update(opt.handle, off, cnt, bucket, [r[off:off + cnt] for r in reps], side)
    main.wait_stream(side)
    z.zero1_bucket_finish(opt.handle, None, main)
    torch.cuda.synchronize()


@pytest.mark.parametrize("n,world,mean", [(777_777, 8, 3000), (65_541, 2, 300), (4099, 4, 37)])
def test_bucket_update_equals_plain_step_without_clipping(n, world, mean):
    """Without clipping each bucket is updated right after its reduce-scatter;
    the result equals zero1_step's bit for bit, the norm within 1e-6."""
    w = WL.Workload("upd", n, world, 0.02, 3, max_norm=0.0)
    hp = z.Hparams(**w.hparams())
    rng = np.random.default_rng(n)
    side = torch.cuda.Stream()
    m0 = WL.master(w, "cuda")
    ra = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    rb = [torch.empty_like(ra[0]) for _ in range(world)]
    with z.Zero1(n, world, hp, z.Options(small_step=-1)) as a, z.Zero1(n, world, hp) as b:
        a.set_state(m0)
        b.set_state(m0)
        for t in range(1, 4):
            grads = WL.grads(w, t, "cuda")
            a.step(grads, ra)
            _bucketed_update_step(b, grads, rb, _buckets(n, rng, mean), side)
            na, ca = a.grad_norm()
            nb, cb = b.grad_norm()
            assert ca == cb == 1.0 and abs(na - nb) <= 1e-6 * na
        assert a.get_state() == b.get_state() == 3
        for x, y in zip(_state(a, n), _state(b, n)):
            assert bits_equal(x, y)
        assert all(torch.equal(x, y) for x, y in zip(ra, rb))


def test_bucket_update_errors():
    n, world = 1000, 2
    g = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    r = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    with z.Zero1(n, world) as opt:                                # clipping on (max_norm 1.0)
        z.zero1_bucket_begin(opt.handle)
        with pytest.raises(z.Zero1Error) as e:
            z.zero1_bucket_update(opt.handle, 0, n, g, r)
        assert "clipping off" in str(e.value)
    with z.Zero1(n, world, z.Hparams(max_norm=0.0), z.Options(capturable=True)) as opt:
        z.zero1_bucket_begin(opt.handle)
        with pytest.raises(z.Zero1Error):
            z.zero1_bucket_update(opt.handle, 0, n, g, r)
    with z.Zero1(n, world, z.Hparams(max_norm=0.0)) as opt:
        z.zero1_bucket_begin(opt.handle)
        z.zero1_bucket_update(opt.handle, 0, 496, g, r)
        with pytest.raises(z.Zero1Error):
            z.zero1_bucket_reduce(opt.handle, 496, 504, [x[496:] for x in g])    # mixing the two kinds
        with pytest.raises(z.Zero1Error):
            z.zero1_bucket_update(opt.handle, 488, 16, [x[488:] for x in g], [x[488:] for x in r])   # overlap
        with pytest.raises(z.Zero1Error):
            z.zero1_bucket_update(opt.handle, 496, 13, [x[496:] for x in g], [x[496:] for x in r])   # ragged mid-way
        z.zero1_bucket_update(opt.handle, 496, 504, [x[496:] for x in g], [x[496:] for x in r])
        z.zero1_bucket_finish(opt.handle, None)
        torch.cuda.synchronize()
        assert opt.get_state() == 1


def test_bucket_reduces_on_an_sm_partition():
    """zero1_sm_partition_create splits the SMs into two green contexts; the
    bucket reduces run on the small group's stream while bf16 GEMMs (a
    backward's kind of work) run on the other group's stream, and the step
    is still the oracle's bit for bit with the GPU's clip coefficient."""
    n, world, mean = 1_000_003, 8, 4000
    w = WL.Workload("bk_part", n, world, 0.02, 2, max_norm=0.05)
    d = w.hparams()
    ohp = o.HP(**d)
    rng = np.random.default_rng(7)
    m0 = WL.master(w, "cuda")
    reps = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    st = o.State(f32(m0))
    x = torch.randn(4096, 768, device="cuda", dtype=torch.bfloat16)
    wgt = torch.randn(768, 3072, device="cuda", dtype=torch.bfloat16)
    with z.SmPartition(16) as part:
        total = torch.cuda.get_device_properties(0).multi_processor_count
        assert part.sms_a >= 16 and part.sms_a + part.sms_b <= total and part.sms_b > 0
        side = torch.cuda.ExternalStream(part.stream_a)
        other = torch.cuda.ExternalStream(part.stream_b)
        with z.Zero1(n, world, z.Hparams(**d), z.Options(bucket_ctas=part.sms_a)) as opt:
            opt.set_state(m0)
            for t in range(1, w.steps + 1):
                grads = WL.grads(w, t, "cuda")
                other.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(other):            # GEMMs beside the reduces
                    ref = x @ wgt
                    for _ in range(8):
                        y = x @ wgt
                _bucketed_step(opt, grads, reps, _buckets(n, rng, mean), side)
                torch.cuda.current_stream().wait_stream(other)
                assert torch.equal(y, ref)
                norm, c = opt.grad_norm()
                reps_o, norm_o, _ = o.step(st, [u16(g) for g in grads], ohp, clip_override=np.float32(c))
                assert abs(norm - norm_o) <= 1e-6 * norm_o
                master, m, v = _state(opt, n)
                assert bits_equal(master, st.master) and bits_equal(m, st.m) and bits_equal(v, st.v)
                for r in range(world):
                    assert np.array_equal(u16(reps[r]), reps_o[r])
        torch.cuda.synchronize()


def test_sm_partition_destroy_waits_for_queued_work():
    """zero1_sm_partition_destroy waits for the work still queued on both of
    the partition's streams before releasing its green contexts: counters
    incremented 200 times on each stream read 200 right after close(), with
    no synchronisation by the caller in between."""
    part = z.SmPartition(16)
    ys = []
    for s in (part.stream_a, part.stream_b):
        es = torch.cuda.ExternalStream(s)
        y = torch.zeros(8 << 20, device="cuda")
        es.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(es):
            for _ in range(200):
                y.add_(1.0)
        ys.append(y)
    part.close()
    part.close()                                  # a second close is a no-op
    for y in ys:
        assert bool((y == 200.0).all())
