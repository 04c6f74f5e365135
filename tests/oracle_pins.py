"""Pins that tie the CPU oracle to facts outside itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
the pages' printed values, a closed form, a library routine (numpy, torch,
torch.optim.AdamW) or brute force.  ``test_oracle_pins.py`` runs them as
tests; ``test_oracle_mutants.py`` runs all of them against copies of the
oracle with planted mistakes and requires that every mistake trips one.

Sources (page title, section):
  "Parallel training" (notes.cassieliang.com) -- sections "What one card
  holds: mixed precision and AdamW", "Training loop and checkpoint", "How
  cards talk: collective communication", "Data parallel and ZeRO".
  "Stanford CS336 Lecture 7 close reading: Parallelism (part 1)" -- 5.1, 5.2.
  "Stanford CS336 Lecture 8 close reading: Parallelism (part 2)" -- 2, 5, 7.
"""
from __future__ import annotations

import math
from pathlib import Path

import numpy as np
import torch

from oracle import zero1_oracle as o

GOLDEN = Path(__file__).parent / "golden"


def golden(name: str) -> dict[str, list[list[str]]]:
    """Parse a golden fixture: ``key value...`` lines, '#' comments."""
    out: dict[str, list[list[str]]] = {}
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        out.setdefault(key, []).append(vals)
    return out


def torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns by torch's own conversion (a library routine)."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def torch_widen(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 by torch (a library routine)."""
    return torch.from_numpy(np.ascontiguousarray(b, np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()


def rand_bf16(rng, n, sigma=1.0):
    return torch_bf16_bits((rng.standard_normal(n) * sigma).astype(np.float32))


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in units of the last place between bf16 patterns (sign-magnitude ordered)."""
    def ordered(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


# ------------------------------------------------------------ collectives

def pin_worked_example():
    """The 4-rank gloo/NCCL example: inputs arange(4)+rank, all-reduce
    [6,10,14,18], reduce-scatter rank i -> element i, all-gather the full
    vector; all-reduce and reduce-scatter + all-gather give the same bits."""
    g = golden("collectives_4rank.txt")
    world = int(g["world"][0][0])
    inputs = {int(r[0]): np.array(r[1:], dtype=np.float32) for r in g["input"]}
    x = [torch_bf16_bits(inputs[r]) for r in range(world)]
    ar = np.array(g["all_reduce"][0], dtype=np.float32)
    direct = o.allreduce_sum_direct(x)
    via, rs = o.allreduce_rs_ag(x)
    for r in range(world):
        assert np.array_equal(torch_widen(direct[r]), ar), (r, direct[r])
        assert np.array_equal(torch_widen(via[r]), ar), (r, via[r])
        assert np.array_equal(direct[r], via[r])
    s = o.shard_len(ar.size, world)
    for rank, val in g["reduce_scatter"]:
        rank = int(rank)
        assert np.array_equal(rs[rank * s:(rank + 1) * s], np.array([float(val)], np.float32))
    assert np.array_equal(torch_widen(via[0]), np.array(g["all_gather"][0], np.float32))
    # Averaging (ReduceOp.AVG in the DDP loop): the same example divided by W.
    avg, rs_avg = o.allreduce_rs_ag(x, average=True)
    assert np.array_equal(rs_avg, ar / world)
    assert np.array_equal(o.reduce_scatter_mean(x), ar / world)
    for r in range(world):
        assert np.array_equal(torch_widen(avg[r]), ar / world)


def pin_worked_example_fp32():
    """The same printed example in the page's own dtype (float32 tensors):
    the fp32 all-reduce, written directly and as reduce-scatter +
    all-gather, gives [6,10,14,18] on every rank and slice i = element i."""
    g = golden("collectives_4rank.txt")
    world = int(g["world"][0][0])
    x = [np.array(next(r[1:] for r in g["input"] if int(r[0]) == q), dtype=np.float32) for q in range(world)]
    ar = np.array(g["all_reduce"][0], dtype=np.float32)
    direct = o.allreduce_f32_direct(x)
    via, rs = o.allreduce_f32_rs_ag(x)
    for q in range(world):
        assert np.array_equal(direct[q], ar) and np.array_equal(via[q], ar)
    s = o.shard_len(ar.size, world)
    for rank, val in g["reduce_scatter"]:
        assert np.array_equal(rs[int(rank) * s:(int(rank) + 1) * s], np.array([float(val)], np.float32))
    avg = o.allreduce_f32_direct(x, average=True)
    assert all(np.array_equal(a, ar / world) for a in avg)


def pin_allreduce_f32_rank_order():
    """fp32 all-reduce = numpy's sequential float32 sum over the rank axis
    (times fp32(1/W) for the mean), ragged n; direct and RS+AG agree."""
    rng = np.random.default_rng(12)
    for world in (1, 2, 3, 4, 8, 64):
        n = 1001
        x = [(rng.standard_normal(n) * np.exp(rng.uniform(-20, 20))).astype(np.float32) for _ in range(world)]
        ref = np.cumsum(np.stack(x), axis=0, dtype=np.float32)[-1]
        for average in (False, True):
            want = ref * np.float32(1.0 / world) if average else ref
            direct = o.allreduce_f32_direct(x, average)
            via, _ = o.allreduce_f32_rs_ag(x, average)
            for q in range(world):
                assert np.array_equal(direct[q].view(np.uint32), want.view(np.uint32)), (world, average)
                assert np.array_equal(via[q].view(np.uint32), want.view(np.uint32)), (world, average)


def pin_all_gather_shards():
    """The printed example's last column: the reduce-scatter outputs [6],
    [10], [14], [18] all-gathered give [6, 10, 14, 18] on every rank; for
    random ragged shards the gather equals numpy's concatenation; and a
    reduce-scatter (sum) followed by this gather equals the all-reduce
    written directly, bit for bit."""
    g = golden("collectives_4rank.txt")
    world = int(g["world"][0][0])
    shards = [np.array([float(v)], np.float32) for _, v in sorted((int(r), v) for r, v in g["reduce_scatter"])]
    outs = o.all_gather_shards(shards, world, 1)
    want = np.array(g["all_gather"][0], np.float32)
    assert all(np.array_equal(x, want) for x in outs)
    rng = np.random.default_rng(13)
    for n, world, extra in ((1000, 3, 0), (1000, 8, 5), (17, 4, 0), (5, 8, 0)):
        s = -(-n // world) + extra
        full = rng.integers(0, 65535, n).astype(np.uint16)
        sh = [full[min(r * s, n):min((r + 1) * s, n)] for r in range(world)]
        outs = o.all_gather_shards(sh, n, s)
        assert all(np.array_equal(x, np.concatenate(sh)) for x in outs)
    x = [rand_bf16(rng, 1001, 1.0) for _ in range(5)]
    _, rs = o.allreduce_rs_ag(x)                       # fp32 reduce-scatter slices
    s = o.shard_len(1001, 5)
    b16 = o.f32_to_bf16(rs)
    gathered = o.all_gather_shards([b16[r * s:(r + 1) * s] for r in range(5)], 1001, s)
    direct = o.allreduce_sum_direct(x)
    assert all(np.array_equal(a, b) for a, b in zip(gathered, direct))


def pin_rs_rank_order():
    """The reduce-scatter sum is an fp32 left fold in rank order (numpy's
    sequential float32 cumsum) scaled by fp32(1/W); ragged n included."""
    rng = np.random.default_rng(11)
    for world in (1, 2, 3, 4, 8, 64):
        n = 1000
        scales = np.exp(rng.uniform(-12, 4, size=(world, 1)))
        grads = [rand_bf16(rng, n, 1.0) for _ in range(world)]
        grads = [torch_bf16_bits(torch_widen(g) * np.float32(scales[q, 0])) for q, g in enumerate(grads)]
        f = np.stack([torch_widen(g) for g in grads])
        ref = np.cumsum(f, axis=0, dtype=np.float32)[-1] * np.float32(1.0 / world)
        got = o.reduce_scatter_mean(grads)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), world
    # Order is visible: 2^24 + 1 rounds back to 2^24 in fp32, so the rank-order
    # mean of (2^24, 1, -2^24) is 0, not 1/3.
    big = torch_bf16_bits(np.array([2.0 ** 24], np.float32))
    one = torch_bf16_bits(np.array([1.0], np.float32))
    neg = torch_bf16_bits(np.array([-(2.0 ** 24)], np.float32))
    assert o.reduce_scatter_mean([big, one, neg])[0] == 0.0
    assert o.reduce_scatter_mean([one, big, neg])[0] == 0.0
    assert o.reduce_scatter_mean([big, neg, one])[0] == np.float32(1.0) * np.float32(1.0 / 3.0)
    # Small integers: every order is exact, the mean equals the integer mean.
    ints = [torch_bf16_bits(rng.integers(-50, 50, size=64).astype(np.float32)) for _ in range(4)]
    exact = np.sum([torch_widen(g) for g in ints], axis=0) / 4
    assert np.array_equal(o.reduce_scatter_mean(ints), exact.astype(np.float32))


def pin_shard_layout():
    """Equal chunks cover [0, n) once; the 1.3B ragged workload's chunks."""
    for n in (1, 7, 8, 9, 13, 4095, 4096, 4097, 1_300_000_005):
        for world in (1, 2, 3, 4, 8, 64):
            s = o.shard_len(n, world)
            assert s * world >= n and (s - 1) * world < n          # the smallest equal chunk
            lengths = [max(0, min((r + 1) * s, n) - min(r * s, n)) for r in range(world)]
            assert sum(lengths) == n
            assert all(length == s for length in lengths[: n // s])
    assert o.shard_len(1_300_000_005, 8) == 162_500_001


# --------------------------------------------------------------- bf16

def pin_bf16_codec():
    """Oracle fp32 <-> bf16 equals torch's conversions: ties, subnormals,
    overflow, signed zeros, infinities; NaN stays NaN."""
    rng = np.random.default_rng(3)
    vals = [rng.standard_normal(20000).astype(np.float32) * np.float32(s) for s in (1e-30, 1e-3, 1.0, 1e20)]
    b = rng.integers(0, 0xFFFF, 5000).astype(np.uint32)
    b = b[(b & 0x7F80) != 0x7F80]                                 # finite bf16 patterns
    vals.append(((b << 16) | 0x8000).view(np.float32))            # exact ties, even and odd
    vals.append(((b << 16) | 0x8001).view(np.float32))            # just above a tie
    vals.append(((b << 16) | 0x7FFF).view(np.float32))            # just below a tie
    vals.append(np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38, 3.3961e38,
                          1e-40, -1e-40, 1e-45, 2.0 ** -126, 9.2e-41], np.float32))
    x = np.concatenate(vals).astype(np.float32)
    ours, ref = o.f32_to_bf16(x), torch_bf16_bits(x)
    assert np.array_equal(ours, ref)
    nan = np.array([np.nan, -np.nan], np.float32)
    assert np.isnan(torch_widen(o.f32_to_bf16(nan))).all()
    every = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    w_ours, w_ref = o.bf16_to_f32(every), torch_widen(every)
    finite = ~np.isnan(w_ref)
    assert np.array_equal(w_ours[finite].view(np.uint32), w_ref[finite].view(np.uint32))
    assert np.isnan(w_ours[~finite]).all()


def pin_bf16_master_example():
    """The printed mixed-precision example: a bf16 weight decremented by 1e-3
    a thousand times stays 1.0; an fp32 master reaches ~0 (0.0 to 4 places);
    bf16 spacing at 1.0 is 0.0078125.  Through the optimizer: AdamW with
    beta1 = beta2 = eps = wd = 0 moves by exactly lr*sign(g), so the master
    follows numpy's float32 loop bit for bit while the replicas follow it in
    bf16."""
    g = golden("bf16_master_example.txt")
    steps, dec = int(g["steps"][0][0]), float(g["decrement"][0][0])
    w = o.f32_to_bf16(np.array([1.0], np.float32))
    d = o.f32_to_bf16(np.array([-dec], np.float32))
    for _ in range(steps):
        w = o.f32_to_bf16(o.bf16_to_f32(w) + o.bf16_to_f32(d))
    assert o.bf16_to_f32(w)[0] == float(g["bf16_weight_after"][0][0])
    spacing = float(g["bf16_spacing_near_1"][0][0])
    assert o.bf16_to_f32(np.array([0x3F81], np.uint16))[0] - 1.0 == spacing
    assert spacing == torch.finfo(torch.bfloat16).eps

    hp = o.HP(lr=dec, beta1=0.0, beta2=0.0, eps=0.0, weight_decay=0.0, max_norm=0.0)
    world = 2
    st = o.State(np.array([1.0], np.float32))
    grads = [o.f32_to_bf16(np.array([1.0], np.float32)) for _ in range(world)]
    ref = np.float32(1.0)
    for _ in range(steps):
        reps, _, _ = o.step(st, grads, hp)
        ref = np.float32(ref - np.float32(dec))
        assert st.master[0] == ref
        assert all(np.array_equal(r, torch_bf16_bits(st.master)) for r in reps)
    assert round(float(st.master[0]), 4) == float(g["fp32_master_after_rounded_4"][0][0])
    assert abs(float(st.master[0]) - 9.324634e-06) < 1e-12
    assert o.bf16_to_f32(reps[0])[0] != 1.0


# --------------------------------------------------------- norm and clip

def pin_norm():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(100_003) * 1e-3).astype(np.float32)
    ref = float(np.linalg.norm(x.astype(np.float64)))
    assert abs(o.l2_norm(x) - ref) <= 1e-13 * ref
    acc = o.NormAccumulator()
    for lo in range(0, x.size, 7919):
        acc.add(x[lo:lo + 7919])
    assert acc.value() == o.l2_norm(x)
    assert o.l2_norm(np.array([3.0, 4.0], np.float32)) == 5.0
    assert o.l2_norm(np.zeros(10, np.float32)) == 0.0
    assert math.isinf(o.l2_norm(np.array([1.0, np.inf], np.float32)))
    assert math.isnan(o.l2_norm(np.array([1.0, np.nan, np.inf], np.float32)))


def pin_clip():
    """Clip only when the norm exceeds max_norm; then the clipped vector has
    norm max_norm and the same direction."""
    assert o.clip_coef(0.5, 1.0) == np.float32(1.0)
    assert o.clip_coef(1.0, 1.0) == np.float32(1.0)
    assert o.clip_coef(4.0, 1.0) == np.float32(0.25)
    assert o.clip_coef(123.0, 0.0) == np.float32(1.0)
    assert o.clip_coef(123.0, -1.0) == np.float32(1.0)
    assert np.isnan(o.clip_coef(float("nan"), 1.0))
    assert o.clip_coef(float("inf"), 1.0) == np.float32(0.0)
    rng = np.random.default_rng(9)
    grads = [rand_bf16(rng, 4099, 0.05) for _ in range(4)]
    ghat = o.reduce_scatter_mean(grads)
    norm = o.l2_norm(ghat)
    ref = float(torch.linalg.vector_norm(torch.from_numpy(ghat.astype(np.float64))))
    assert abs(norm - ref) <= 1e-12 * ref
    for max_norm in (0.1 * norm, 0.5 * norm):
        c = o.clip_coef(norm, max_norm)
        clipped = (ghat * c).astype(np.float64)
        assert abs(np.linalg.norm(clipped) - max_norm) <= 1e-6 * max_norm
        cos = clipped @ ghat.astype(np.float64) / (np.linalg.norm(clipped) * norm)
        assert abs(cos - 1.0) < 1e-9
    # Through the step: with a huge max_norm the coefficient is exactly 1.
    st = o.State(np.zeros(4099, np.float32))
    _, n1, c1 = o.step(st, grads, o.HP(max_norm=10 * norm))
    assert c1 == np.float32(1.0) and abs(n1 - norm) <= 1e-12 * norm
    st = o.State(np.zeros(4099, np.float32))
    _, n2, c2 = o.step(st, grads, o.HP(max_norm=0.25 * norm))
    assert c2 == o.clip_coef(norm, 0.25 * norm) and c2 < 1.0


# ---------------------------------------------------------------- AdamW

def pin_adamw_first_step():
    """t = 1, eps = 0: m1/sqrt(v1) = sign(g) and the folded step size is lr,
    so p1 = (p0 - lr*sign(g)) * (1 - lr*wd) -- decay after the update."""
    rng = np.random.default_rng(21)
    n, lr, wd = 257, 0.1, 0.5
    p0 = rng.uniform(0.5, 1.0, n).astype(np.float32)
    g = rand_bf16(rng, n, 1.0)
    g[torch_widen(g) == 0] = o.f32_to_bf16(np.array([0.5], np.float32))[0]
    st = o.State(p0)
    o.step(st, [g, g], o.HP(lr=lr, beta1=0.9, beta2=0.999, eps=0.0, weight_decay=wd, max_norm=0.0))
    sgn = np.sign(torch_widen(g)).astype(np.float64)
    after = (p0.astype(np.float64) - lr * sgn) * (1.0 - lr * wd)
    before = p0.astype(np.float64) * (1.0 - lr * wd) - lr * sgn
    err = np.abs(st.master.astype(np.float64) - after)
    assert err.max() <= 4e-7, err.max()
    assert np.abs(after - before).min() > 100 * 4e-7      # the check tells the orders apart
    assert np.array_equal(st.m, (np.float32(0.1) * torch_widen(g)).astype(np.float32))


def pin_adamw_constant_gradient():
    """Constant gradient, eps = 0: m_t = (1-b1^t) g and v_t = (1-b2^t) g^2, so
    the bias-corrected update is exactly lr*sign(g) at every t."""
    rng = np.random.default_rng(22)
    n, lr = 129, 1e-2
    p = rng.uniform(0.5, 1.0, n).astype(np.float32)
    g = rand_bf16(rng, n, 0.3)
    g[torch_widen(g) == 0] = o.f32_to_bf16(np.array([0.25], np.float32))[0]
    sgn = np.sign(torch_widen(g)).astype(np.float64)
    st = o.State(p)
    hp = o.HP(lr=lr, beta1=0.9, beta2=0.95, eps=0.0, weight_decay=0.0, max_norm=0.0)
    for _ in range(10):
        before = st.master.astype(np.float64)
        o.step(st, [g, g, g], hp)
        move = before - st.master.astype(np.float64)
        assert np.abs(move - lr * sgn).max() <= 1.2e-7 + lr * 2e-6, np.abs(move - lr * sgn).max()


def pin_adamw_zero_gradient_pure_decay():
    """g = 0: m = v = 0, the Adam term is 0/eps = 0 and only the decoupled
    decay acts: p_t = p0 * (1 - lr*wd)^t (an L2 penalty added to the
    gradient would move p by ~lr instead)."""
    rng = np.random.default_rng(23)
    n, lr, wd = 64, 1e-2, 0.1
    p0 = rng.standard_normal(n).astype(np.float32)
    st = o.State(p0)
    zero = np.zeros(n, np.uint16)
    for _ in range(10):
        o.step(st, [zero, zero], o.HP(lr=lr, weight_decay=wd, max_norm=1.0))
    ref = p0.astype(np.float64) * (1.0 - lr * wd) ** 10
    assert np.abs(st.master - ref).max() <= 1e-6 * np.abs(ref).max()
    assert not st.m.any() and not st.v.any()


def _torch_adamw_run(p0, ghats, hp: o.HP):
    """float64 torch.optim.AdamW arranged to match the folded form: torch's
    eps sits outside sqrt(v/(1-b2^t)), ours outside sqrt(v), so torch gets
    eps/sqrt(1-b2^t) at step t; torch decays before its update, ours after, so
    torch runs with wd = 0 and the decay multiplies in after each step."""
    p = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    opt = torch.optim.AdamW([p], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=0.0, foreach=False)
    for t, gh in enumerate(ghats, start=1):
        p.grad = torch.tensor(gh, dtype=torch.float64)
        opt.param_groups[0]["eps"] = hp.eps / math.sqrt(1.0 - hp.beta2 ** t)
        opt.step()
        with torch.no_grad():
            p.mul_(1.0 - hp.lr * hp.weight_decay)
    s = opt.state[p]
    return p.detach().numpy(), s["exp_avg"].numpy(), s["exp_avg_sq"].numpy()


def pin_adamw_vs_torch():
    """Ten steps of the oracle's AdamW equal float64 torch.optim.AdamW (with
    the eps and decay-order adjustments) to fp32 rounding."""
    rng = np.random.default_rng(24)
    n, world = 16, 4
    hp = o.HP(lr=1e-2, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.0)
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    st = o.State(p0)
    ghats = []
    for _ in range(10):
        grads = [rand_bf16(rng, n, 1e-2) for _ in range(world)]
        ghats.append(np.mean([torch_widen(g).astype(np.float64) for g in grads], axis=0))
        o.step(st, grads, hp)
    p, m, v = _torch_adamw_run(p0, ghats, hp)
    assert np.allclose(st.master, p, rtol=1e-5, atol=1e-7 * np.abs(p).max())
    assert np.allclose(st.m, m, rtol=1e-5, atol=1e-5 * np.abs(m).max())
    assert np.allclose(st.v, v, rtol=1e-5, atol=0)
    # eps matters at this scale: the textbook placement would not match.
    assert hp.eps / math.sqrt(1 - hp.beta2 ** 10) != hp.eps


def pin_full_step_brute_force():
    """Whole steps on tiny ragged inputs (n = 13, W = 4, clipping on and off)
    against float64 library routines: torch mean of the rank gradients,
    torch.linalg.vector_norm, the clip rule, torch.optim.AdamW as above,
    torch's bf16 cast; replicas within 1 bf16 ulp, every replica equal."""
    rng = np.random.default_rng(25)
    n, world = 13, 4
    for max_norm in (0.05, 100.0):
        hp = o.HP(lr=1e-2, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=max_norm)
        p0 = (rng.standard_normal(n) * 0.5).astype(np.float32)
        st = o.State(p0)
        ghats_clipped = []
        for _ in range(5):
            grads = [rand_bf16(rng, n, 0.1) for _ in range(world)]
            mean = np.mean([torch_widen(g).astype(np.float64) for g in grads], axis=0)
            norm = float(torch.linalg.vector_norm(torch.from_numpy(mean)))
            scale = max_norm / norm if norm > max_norm else 1.0
            ghats_clipped.append(mean * scale)
            reps, onorm, oc = o.step(st, grads, hp)
            assert abs(onorm - norm) <= 1e-6 * norm
            assert abs(float(oc) - scale) <= 1e-6 * scale
            assert all(np.array_equal(r, reps[0]) for r in reps)
        p, m, v = _torch_adamw_run(p0, ghats_clipped, hp)
        assert np.allclose(st.master, p, rtol=1e-5, atol=1e-6 * np.abs(p).max())
        assert np.allclose(st.v, v, rtol=1e-4, atol=0)
        ref_b = torch_bf16_bits(p.astype(np.float32))
        assert bf16_ulp_distance(reps[0], ref_b).max() <= 1


def pin_step_ex_default_is_step():
    """The options entry with every option off is the default step, bit for bit."""
    rng = np.random.default_rng(30)
    n, world = 1001, 4
    hp = o.HP(max_norm=0.05)
    a, b = o.State((rng.standard_normal(n) * 0.02).astype(np.float32)), None
    b = a.copy()
    for _ in range(3):
        grads = [rand_bf16(rng, n, 0.01) for _ in range(world)]
        ra, na, ca = o.step(a, grads, hp)
        rb, nb, cb = o.step_ex(b, grads, hp, o.Options())
        assert na == nb and ca == cb
        assert all(np.array_equal(x, y) for x, y in zip(ra, rb))
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def pin_decay_first_vs_torch_adamw():
    """decay_before_update is torch.optim.AdamW's own order: ten steps equal
    float64 torch.optim.AdamW with weight decay on (eps scaled as before)."""
    rng = np.random.default_rng(31)
    n, world = 16, 4
    hp = o.HP(lr=1e-2, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.5, max_norm=0.0)
    p0 = rng.uniform(0.5, 1.0, n).astype(np.float32)
    st = o.state_ex(p0, o.Options(decay_before_update=True))
    p = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    opt = torch.optim.AdamW([p], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=hp.weight_decay, foreach=False)
    for t in range(1, 11):
        grads = [rand_bf16(rng, n, 1e-2) for _ in range(world)]
        o.step_ex(st, grads, hp, o.Options(decay_before_update=True))
        p.grad = torch.tensor(np.mean([torch_widen(g).astype(np.float64) for g in grads], axis=0))
        opt.param_groups[0]["eps"] = hp.eps / math.sqrt(1.0 - hp.beta2 ** t)
        opt.step()
    ref = p.detach().numpy()
    assert np.allclose(st.master, ref, rtol=2e-6, atol=0)
    # the page's order differs visibly at this lr * wd
    st2 = o.state_ex(p0, o.Options())
    rng = np.random.default_rng(31)
    for t in range(1, 11):
        o.step_ex(st2, [rand_bf16(rng, n, 1e-2) for _ in range(world)], hp, o.Options())
    assert np.abs(st2.master - ref).max() > 1e3 * 2e-6 * np.abs(ref).max()


def pin_clip_eps_vs_torch_clip_grad_norm():
    """clip_eps = 1e-6 is torch.nn.utils.clip_grad_norm_'s coefficient
    min(1, max_norm/(norm + 1e-6)); with decay first the whole step equals
    clip_grad_norm_ followed by torch.optim.AdamW (float64)."""
    for norm, mx in ((3.0, 1.0), (0.5, 1.0), (1.0, 1.0), (1.0 + 5e-7, 1.0), (1e-3, 1e-3)):
        g = torch.tensor([norm], dtype=torch.float64, requires_grad=True)
        g.grad = torch.tensor([norm], dtype=torch.float64)
        torch.nn.utils.clip_grad_norm_([g], mx)
        want = float(g.grad[0]) / norm
        assert abs(float(o.clip_coef_ex(norm, mx, 1e-6)) - want) <= 1e-7 * want, (norm, mx)
    rng = np.random.default_rng(32)
    n, world = 13, 4
    hp = o.HP(lr=1e-2, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.05)
    opts = o.Options(decay_before_update=True, clip_eps=1e-6)
    p0 = (rng.standard_normal(n) * 0.5).astype(np.float32)
    st = o.state_ex(p0, opts)
    p = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    opt = torch.optim.AdamW([p], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=hp.weight_decay, foreach=False)
    for t in range(1, 6):
        grads = [rand_bf16(rng, n, 0.1) for _ in range(world)]
        _, _, c = o.step_ex(st, grads, hp, opts)
        p.grad = torch.tensor(np.mean([torch_widen(x).astype(np.float64) for x in grads], axis=0))
        torch.nn.utils.clip_grad_norm_([p], hp.max_norm)
        opt.param_groups[0]["eps"] = hp.eps / math.sqrt(1.0 - hp.beta2 ** t)
        opt.step()
        assert c < 1.0
    assert np.allclose(st.master, p.detach().numpy(), rtol=1e-5, atol=1e-6 * np.abs(p0).max())


def pin_bf16_moments_bounds():
    """bf16 moments: stored values are bf16, v >= 0; over ten steps m and v
    stay within bf16 rounding of the fp32-moment oracle's (relative 2^-6 of
    the array scale) and the master within 1e-3 relative; with a constant
    gradient and eps = 0 every step still moves by lr*sign(g) to within the
    bf16 precision of m/sqrt(v)."""
    rng = np.random.default_rng(33)
    n, world = 4099, 4
    hp = o.HP(lr=1e-3, max_norm=0.0)
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    a, b = o.state_ex(p0, o.Options()), o.state_ex(p0, o.Options(moments_bf16=True))
    for _ in range(10):
        grads = [rand_bf16(rng, n, 1e-2) for _ in range(world)]
        o.step_ex(a, grads, hp, o.Options())
        ra, _, _ = o.step_ex(b, grads, hp, o.Options(moments_bf16=True))
    bm, bv = o.bf16_to_f32(b.m), o.bf16_to_f32(b.v)
    assert (bv >= 0).all()
    for x, ref in ((bm, a.m), (bv, a.v)):
        scale = np.sqrt(np.mean(ref.astype(np.float64) ** 2))
        assert np.abs(x - ref).max() <= 2.0 ** -6 * max(scale, 1e-30) + 2.0 ** -7 * np.abs(ref).max()
    assert np.abs(b.master - a.master).max() <= 1e-3 * np.abs(a.master).max()
    assert np.array_equal(ra[0], o.f32_to_bf16(b.master))
    # constant gradient, eps = 0
    lr = 1e-2
    hp2 = o.HP(lr=lr, beta1=0.9, beta2=0.95, eps=0.0, weight_decay=0.0, max_norm=0.0)
    p = rng.uniform(0.5, 1.0, 64).astype(np.float32)
    g = o.f32_to_bf16(np.where(rng.random(64) < 0.5, -0.25, 0.5).astype(np.float32))
    st = o.state_ex(p, o.Options(moments_bf16=True))
    sgn = np.sign(o.bf16_to_f32(g)).astype(np.float64)
    for _ in range(10):
        before = st.master.astype(np.float64)
        o.step_ex(st, [g, g], hp2, o.Options(moments_bf16=True))
        assert np.abs((before - st.master) - lr * sgn).max() <= lr * 2.0 ** -6


def pin_bf16_moments_vs_torch_inplace_ops():
    """The bf16-moment reading against the page's own in-place ops run by
    torch on bf16 tensors: m.mul_(b1).add_(g, alpha=1-b1),
    v.mul_(b2).addcmul_(g, g, value=1-b2) and denom = v.sqrt().add_(eps),
    each op computing in fp32 and rounding its result to bf16; the fp32
    master then takes p - step_size * (m / denom) and the decay, one fp32
    operation at a time.  Step by step from the oracle's state, the oracle's
    m, v and master equal torch's in at least 99.9% of the elements
    (eps = 1e-3, near sqrt(v), so that the roundings of d matter).
    Torch's kernels fuse the moments' multiply-add before the bf16
    rounding, where the reading rounds the product to fp32 first.  That
    moves a value lying at a bf16 rounding boundary by one bf16 ulp, or
    leaves a residual of the product's fp32 rounding where the two terms
    cancel exactly.  Every moment difference is within those bounds.  A
    reading without an intermediate rounding disagrees in most elements."""
    rng = np.random.default_rng(41)
    n = 20_000
    opts = o.Options(moments_bf16=True)
    hp = o.HP(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-3, weight_decay=0.1, max_norm=0.0)
    st = o.state_ex((rng.standard_normal(n) * 0.02).astype(np.float32), opts)
    as_bf16 = lambda u: torch.from_numpy(u.astype(np.uint16).view(np.int16).copy()).view(torch.bfloat16)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    for t in range(1, 7):
        g = rand_bf16(rng, n, 1e-2)
        gt = torch.from_numpy(torch_widen(g).astype(np.float32))
        m, v = as_bf16(st.m), as_bf16(st.v)
        p = torch.from_numpy(st.master.copy())
        sc = o.step_scalars(hp, 1, t)
        m.mul_(hp.beta1).add_(gt, alpha=1 - hp.beta1)
        v.mul_(hp.beta2).addcmul_(gt, gt, value=1 - hp.beta2)
        denom = v.sqrt().add_(hp.eps)
        u = m.float() / denom.float()
        p = p - torch.tensor(sc["step_size"], dtype=torch.float32) * u
        p = p * torch.tensor(sc["decay"], dtype=torch.float32)
        assert st.t == t - 1
        o.step_ex(st, [g], hp, opts)                       # W = 1, no clipping: the step sees g exactly
        gw = torch_widen(g).astype(np.float64)
        for ours, theirs, term in ((st.m, bits(m), (1 - hp.beta1) * np.abs(gw)),
                                   (st.v, bits(v), (1 - hp.beta2) * gw * gw)):
            assert np.mean(ours == theirs) >= 0.999
            a64, b64 = torch_widen(ours).astype(np.float64), torch_widen(theirs).astype(np.float64)
            tol = 2.0 ** -7 * np.maximum(np.abs(a64), np.abs(b64)) + 2.0 ** -23 * term
            assert (np.abs(a64 - b64) <= tol).all()
        assert np.mean(st.master.view(np.uint32) == p.numpy().view(np.uint32)) >= 0.999


def pin_fp32_update_vs_torch_inplace_ops():
    """The fp32 update against the page's own in-place ops run by torch on
    fp32 tensors: m.mul_(b1).add_(g, alpha=1-b1),
    v.mul_(b2).addcmul_(g, g, value=1-b2),
    p.addcdiv_(m, v.sqrt().add_(eps), value=-step_size), p.mul_(1-lr*wd),
    step by step from the oracle's own state (W = 1, no clipping, so the
    step sees g exactly).
    At the first step m = v = 0, so every op is a product with one rounding
    whatever torch fuses: there the oracle's m and v equal torch's in every
    element, which fixes the association of the second-moment term,
    ((1-b2)*g)*g, against (1-b2)*(g*g) (the two disagree in about 30% of
    bf16 gradients).  Afterwards torch's kernels fuse the multiply-add
    (one rounding of a*x + y) where the reading rounds the product first,
    so the two agree in most elements (m >= 60%, v >= 80%, master >= 90%)
    and every moment difference is within what one skipped product rounding
    and the final rounding allow: 2^-24 |product| + 2^-23 |result|.  For the
    master, torch's addcdiv scales m before dividing by d, while the reading
    takes the text's step direction m / (sqrt(v) + eps) and scales that, so
    the bound is two ulps of the scaled step, the two final roundings
    (update, then decay) and what the step's own m and v differences carry
    into step_size * m / d."""
    rng = np.random.default_rng(43)
    n = 20_000
    hp = o.HP(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.0)
    st = o.State((rng.standard_normal(n) * 0.02).astype(np.float32))
    same = lambda a, b: np.mean(a.view(np.uint32) == b.view(np.uint32))
    for t in range(1, 7):
        g = rand_bf16(rng, n, 1e-2)
        gt = torch.from_numpy(torch_widen(g).astype(np.float32))
        m, v, p = (torch.from_numpy(x.copy()) for x in (st.m, st.v, st.master))
        sc = o.step_scalars(hp, 1, t)
        m.mul_(hp.beta1).add_(gt, alpha=1 - hp.beta1)
        v.mul_(hp.beta2).addcmul_(gt, gt, value=1 - hp.beta2)
        p.addcdiv_(m, v.sqrt().add_(hp.eps), value=-float(sc["step_size"]))
        p.mul_(float(sc["decay"]))
        assert st.t == t - 1
        o.step(st, [g], hp)
        tm, tv, tp = m.numpy(), v.numpy(), p.numpy()
        if t == 1:
            assert same(st.m, tm) == 1.0 and same(st.v, tv) == 1.0
        assert same(st.m, tm) >= 0.6 and same(st.v, tv) >= 0.8 and same(st.master, tp) >= 0.9
        g64 = torch_widen(g).astype(np.float64)
        m64, v64 = tm.astype(np.float64), tv.astype(np.float64)
        d64 = np.sqrt(v64) + hp.eps
        step = float(sc["step_size"])
        # The master: torch's addcdiv forms (value * m) / d, where the reading
        # follows the text's step direction m / d and then scales it; each
        # side rounds that scaled step twice (within one ulp of it), so they
        # differ by up to two; the step direction also carries the moments'
        # differences, and two rounded ops follow (the update, the decay).
        dm = np.abs(st.m.astype(np.float64) - m64)
        dd = np.abs(st.v.astype(np.float64) - v64) / (2.0 * np.sqrt(np.maximum(v64, 1e-300)))
        carried = step * (dm / d64 + np.abs(m64) * dd / (d64 * d64))
        for ours, theirs, prod, k_prod, k_res, extra in (
                (st.m, tm, (1 - hp.beta1) * np.abs(g64), 0.5, 1, 0.0),
                (st.v, tv, (1 - hp.beta2) * g64 * g64, 0.5, 1, 0.0),
                (st.master, tp, step * np.abs(m64) / d64, 2, 2, carried)):
            a, b = ours.astype(np.float64), theirs.astype(np.float64)
            bound = 1.001 * (2.0 ** -23 * (k_prod * prod + k_res * np.maximum(np.abs(a), np.abs(b))) + extra)
            assert (np.abs(a - b) <= bound).all(), t


def pin_ddp_linearity():
    """The printed DDP check (float64): the mean of the 4 shard gradients is
    the full-batch gradient.  The oracle's reduce-scatter mean of the bf16
    shard gradients stays within bf16 rounding of it."""
    g = golden("ddp_linearity.txt")
    k, rows = int(g["shards"][0][0]), int(g["rows"][0][0])
    din, dout = int(g["in_dim"][0][0]), int(g["out_dim"][0][0])
    torch.manual_seed(int(g["seed"][0][0]))
    w1 = torch.randn(din, dout, dtype=torch.float64, requires_grad=True)
    x, y = torch.randn(rows, din, dtype=torch.float64), torch.randn(rows, dout, dtype=torch.float64)

    def loss_fn(a, b):
        return ((torch.tanh(a @ w1) - b) ** 2).mean()

    g_full, = torch.autograd.grad(loss_fn(x, y), w1)
    shards = [torch.autograd.grad(loss_fn(a, b), w1)[0] for a, b in zip(x.chunk(k), y.chunk(k))]
    assert str(torch.allclose(torch.stack(shards).mean(0), g_full)) == g["printed"][0][0]
    bf = [torch_bf16_bits(s.numpy().ravel().astype(np.float32)) for s in shards]
    got = o.reduce_scatter_mean(bf).astype(np.float64)
    bound = 2.0 ** -8 * np.mean([np.abs(s.numpy().ravel()) for s in shards], axis=0) + 1e-12
    assert (np.abs(got - g_full.numpy().ravel()) <= bound).all()


# ----------------------------------------------------------- accounting

def pin_memory_accounting():
    """16 bytes per parameter (2+2+4+4+4) and the printed 7.5B / 64-GPU
    ladder 120.0 / 31.4 / 16.6 / 1.9 GB per GPU."""
    g = golden("zero_memory_7p5b_64.txt")
    psi, world, k = float(g["psi"][0][0]), int(g["world"][0][0]), float(g["k"][0][0])
    for stage in range(4):
        gb = o.zero_bytes_per_rank(stage, psi, world, k) / 1e9
        assert round(gb, 1) == float(g[f"stage{stage}"][0][0]), (stage, gb)
    per_param = o.zero_bytes_per_rank(0, 1.0, 1, k)
    itemsizes = 2 * np.dtype(np.uint16).itemsize + 3 * np.dtype(np.float32).itemsize
    assert per_param == float(g["bytes_per_param"][0][0]) == itemsizes


def pin_ring_volume():
    g = golden("ring_volume.txt")
    b, w = float(g["ddp_7b_grad_bytes"][0][0]), int(g["ddp_7b_world"][0][0])
    assert abs(o.ring_send_bytes(b, w, "all_reduce") / 1e9 - float(g["ddp_7b_send_gb"][0][0])) < 1e-9
    q, qw = float(g["quiz_size_mb"][0][0]), int(g["quiz_world"][0][0])
    assert o.ring_send_bytes(q, qw, "all_reduce") == float(g["quiz_send_mb"][0][0])
    assert o.ring_send_bytes(q, qw, "reduce_scatter") + o.ring_send_bytes(q, qw, "all_gather") == \
        o.ring_send_bytes(q, qw, "all_reduce")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
