"""zero1_allreduce (the DDP all-reduce) against the CPU oracle through the C ABI.

The pages' worked example (4 ranks holding arange(4) + rank, all-reduce
[6, 10, 14, 18]) in both element types; random ragged shapes bit for bit
against the oracle's reduce-scatter + all-gather (which its pins tie to the
direct all-reduce); in place and out of place; canaries around every buffer;
and the pages' benchmark size (1e8 fp32 elements, world size 4) in full.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import zero_sharded_adamw_gb300 as z
from oracle import zero1_oracle as o
from tests.gpu_util import Guarded, f32, u16
from tests.oracle_pins import golden

pytestmark = pytest.mark.gpu

DT = {"bf16": (z.DTYPE_BF16, torch.bfloat16), "f32": (z.DTYPE_F32, torch.float32)}


def _host(t: torch.Tensor) -> np.ndarray:
    return u16(t) if t.dtype == torch.bfloat16 else f32(t)


def _oracle(inputs: list[np.ndarray], average: bool) -> np.ndarray:
    if inputs[0].dtype == np.uint16:
        outs, _ = o.allreduce_rs_ag(inputs, average)
    else:
        outs, _ = o.allreduce_f32_rs_ag(inputs, average)
    return outs[0]


def _run(n: int, world: int, dtype: str, op: int, inplace: bool, seed: int = 0):
    code, tdt = DT[dtype]
    g = torch.Generator(device="cuda").manual_seed(seed + 7 * n + world)
    ins = [Guarded(n, tdt) for _ in range(world)]
    for q, b in enumerate(ins):
        b.t.copy_(torch.randn(n, generator=g, device="cuda") * (q + 1) * 0.01)
    host_in = [_host(b.t) for b in ins]
    outs = ins if inplace else [Guarded(n, tdt) for _ in range(world)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    z.zero1_allreduce(n, world, code, op, [b.t for b in ins], [b.t for b in outs], err)
    torch.cuda.synchronize()
    want = _oracle(host_in, op == z.OP_AVG)
    for b in outs:
        got = _host(b.t)
        assert np.array_equal(got.view(np.uint16 if dtype == "bf16" else np.uint32),
                              want.view(np.uint16 if dtype == "bf16" else np.uint32))
    assert all(b.intact() for b in ins + outs)
    assert int(err.item()) == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_worked_example(dtype):
    """The printed 4-rank example: every rank ends with [6, 10, 14, 18]; the
    mean gives [1.5, 2.5, 3.5, 4.5]; in place as torch's all_reduce is."""
    gd = golden("collectives_4rank.txt")
    world = int(gd["world"][0][0])
    code, tdt = DT[dtype]
    ar = torch.tensor([float(v) for v in gd["all_reduce"][0]])
    for op, want in ((z.OP_SUM, ar), (z.OP_AVG, ar / world)):
        xs = [torch.tensor([float(v) for v in next(r[1:] for r in gd["input"] if int(r[0]) == q)],
                           device="cuda").to(tdt) for q in range(world)]
        z.zero1_allreduce(4, world, code, op, xs, xs)
        torch.cuda.synchronize()
        for x in xs:
            assert torch.equal(x.float().cpu(), want)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 5, 8, 9, 16, 64])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 2047, 2048, 2049, 4096 * 3 + 5, 300_007])
def test_shapes(n, world, dtype):
    for op in (z.OP_SUM, z.OP_AVG):
        _run(n, world, dtype, op, inplace=False)
    _run(n, world, dtype, z.OP_AVG, inplace=True, seed=1)


def test_many_ranks_and_tiles():
    _run(2_000_003, 512, "bf16", z.OP_AVG, inplace=False)
    _run(1_000_001, 100, "f32", z.OP_SUM, inplace=True)


def test_lecture_benchmark_size():
    """1e8 fp32 elements over 4 ranks (the lecture's benchmark), whole arrays."""
    _run(100_000_000, 4, "f32", z.OP_SUM, inplace=False)


def test_argument_errors():
    x = [torch.zeros(16, device="cuda") for _ in range(2)]
    for args, code in (((0, 2, z.DTYPE_F32, z.OP_SUM), -1), ((16, 0, z.DTYPE_F32, z.OP_SUM), -1),
                       ((16, 2, 7, z.OP_SUM), -1), ((16, 2, z.DTYPE_F32, 9), -1)):
        with pytest.raises(z.Zero1Error) as e:
            z.zero1_allreduce(*args, x, x)
        assert e.value.code == code
    with pytest.raises(z.Zero1Error) as e:
        z.zero1_allreduce(15, 2, z.DTYPE_F32, z.OP_SUM, [t[1:] for t in x], x)
    assert e.value.code == -2


def test_allreduce_sum_on_a_handle():
    """zero1_allreduce_sum takes n and W from a handle: the pages' 4-rank
    example ([0,1,2,3] + rank -> [6,10,14,18] on every rank), and equality
    with zero1_allreduce on a multi-tile ragged case, in place and not."""
    x = [torch.tensor([0.0, 1, 2, 3], device="cuda").add(r).to(torch.bfloat16) for r in range(4)]
    out = [torch.empty_like(t) for t in x]
    with z.Zero1(4, 4) as opt:
        z.zero1_allreduce_sum(opt.handle, x, out)
        torch.cuda.synchronize()
    for t in out:
        assert t.float().tolist() == [6.0, 10.0, 14.0, 18.0]
    n, world = 1_000_003, 8
    g = torch.Generator(device="cuda").manual_seed(11)
    ins = [torch.randn(n, generator=g, device="cuda").to(torch.bfloat16) for _ in range(world)]
    want = [torch.empty_like(t) for t in ins]
    z.zero1_allreduce(n, world, z.DTYPE_BF16, z.OP_SUM, ins, want)
    with z.Zero1(n, world) as opt:
        got = [torch.empty_like(t) for t in ins]
        z.zero1_allreduce_sum(opt.handle, ins, got)
        inplace = [t.clone() for t in ins]
        z.zero1_allreduce_sum(opt.handle, inplace, inplace)
        torch.cuda.synchronize()
    for a, b, c in zip(got, want, inplace):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert torch.equal(c.view(torch.int16), b.view(torch.int16))
