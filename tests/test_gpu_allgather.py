"""zero1_allgather (the ZeRO-3 / FSDP parameter all-gather) against the oracle.

The pages' example's last column ([6], [10], [14], [18] -> [6, 10, 14, 18]);
random shard lengths and ragged n, bf16 and fp32, out of place and in place
(each rank's shard inside its own output), byte for byte against the
oracle's gather, canaries around every output.
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


def _host(t):
    return u16(t) if t.dtype == torch.bfloat16 else f32(t)


def _run(n: int, world: int, shard_len: int, dtype: torch.dtype, inplace: bool):
    code = z.DTYPE_BF16 if dtype == torch.bfloat16 else z.DTYPE_F32
    g = torch.Generator(device="cuda").manual_seed(n + world)
    outs = [Guarded(n, dtype) for _ in range(world)]
    shards = []
    for r in range(world):
        lo, hi = min(r * shard_len, n), min((r + 1) * shard_len, n)
        if inplace:
            view = outs[r].t[lo:hi]
            view.copy_(torch.randn(hi - lo, generator=g, device="cuda"))
            shards.append(view if hi > lo else None)
        else:
            s = torch.randn(max(hi - lo, 1), generator=g, device="cuda").to(dtype)[: hi - lo]
            shards.append(s if hi > lo else None)
    host = [(_host(s) if s is not None else np.empty(0, dtype=np.uint16 if dtype == torch.bfloat16 else np.float32))
            for s in shards]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    z.zero1_allgather(n, world, shard_len, code, shards, [b.t for b in outs], err)
    torch.cuda.synchronize()
    want = o.all_gather_shards(host, n, shard_len)
    for b, wnt in zip(outs, want):
        assert np.array_equal(_host(b.t).view(np.uint8), wnt.view(np.uint8))
        assert b.intact()
    assert int(err.item()) == 0


def test_worked_example():
    gd = golden("collectives_4rank.txt")
    world = int(gd["world"][0][0])
    vals = [float(v) for _, v in sorted((int(r), v) for r, v in gd["reduce_scatter"])]
    # one element per rank, padded to the 8-element shard granularity
    shards = [torch.full((8,), v, device="cuda") for v in vals]
    outs = [torch.zeros(32, device="cuda") for _ in range(world)]
    z.zero1_allgather(32, world, 8, z.DTYPE_F32, shards, outs)
    torch.cuda.synchronize()
    want = torch.tensor([float(v) for v in gd["all_gather"][0]])
    for out in outs:
        assert torch.equal(out.view(world, 8)[:, 0].cpu(), want)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("world", [1, 2, 3, 8, 64])
@pytest.mark.parametrize("n", [1, 9, 4099, 65_541, 1_000_003])
def test_shapes(n, world, dtype):
    s = -(-n // world)
    for shard_len in (-(-s // 8) * 8, -(-s // 8) * 8 + 40):
        _run(n, world, shard_len, dtype, inplace=False)
    _run(n, world, -(-s // 8) * 8, dtype, inplace=True)


def test_large_layer():
    _run(39_383_808, 8, 4_922_976, torch.bfloat16, inplace=False)     # the GPT-2 embedding layer


def test_argument_errors():
    o_ = [torch.zeros(16, device="cuda") for _ in range(2)]
    with pytest.raises(z.Zero1Error) as e:
        z.zero1_allgather(16, 2, 4, z.DTYPE_F32, o_, o_)           # shard_len not a multiple of 8
    assert e.value.code == -1
    with pytest.raises(z.Zero1Error):
        z.zero1_allgather(32, 2, 8, z.DTYPE_F32, o_, o_)           # 2 * 8 < 32
