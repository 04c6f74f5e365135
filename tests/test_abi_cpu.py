"""The C-ABI library without a GPU: it builds, loads, exports every entry
point include/zero1.h declares, and its host logic (shard plan, per-step
scalars, argument checks) agrees with the oracle.  No compute call runs."""
from __future__ import annotations

import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import zero_sharded_adamw_gb300 as z
from oracle import zero1_oracle as o
from zero_sharded_adamw_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "zero1.h")


@pytest.fixture(scope="module")
def lib_path():
    return _build.build()


def declared_symbols() -> set[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(zero1_\w+)\s*\(", text, flags=re.M))


def test_exports_every_declared_symbol(lib_path):
    declared = declared_symbols()
    assert "zero1_create" in declared and "zero1_step" in declared and "zero1_destroy" in declared
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (zero1_\w+)$", out, flags=re.M))
    assert declared <= exported, declared - exported
    assert declared == set(z.EXPORTED_SYMBOLS)
    lib = C.CDLL(lib_path)
    for name in declared:
        assert getattr(lib, name)


def test_shard_plan_matches_oracle_chunks(lib_path):
    for n in (1, 7, 8, 9, 13, 4095, 4096, 4097, 124_355_328, 1_300_000_005, 7_000_000_000, 350_000_000):
        for world in (1, 2, 3, 4, 8, 64, 512):
            s, padded = z.zero1_shard_plan(n, world)
            so = o.shard_len(n, world)
            assert s % 64 == 0 and so <= s < so + 64 and padded == s * world
            assert padded - n < world * 64                      # padding below 64 per shard
            covered = sum(max(0, min((r + 1) * s, n) - min(r * s, n)) for r in range(world))
            assert covered == n


@pytest.mark.parametrize("world", [1, 2, 3, 8, 64])
@pytest.mark.parametrize("t", [1, 2, 10, 1000])
def test_step_scalars_match_oracle(lib_path, world, t):
    for hp in (dict(), dict(lr=3e-4, beta1=0.8, beta2=0.999, eps=1e-6, weight_decay=0.01),
               dict(lr=1e-3, beta1=0.0, beta2=0.0, eps=0.0, weight_decay=0.0, max_norm=0.0)):
        ours = z.zero1_step_scalars(z.Hparams(**hp), world, t)
        ref = o.step_scalars(o.HP(**hp), world, t)
        for k in ref:
            assert np.float32(ours[k]).view(np.uint32) == np.float32(ref[k]).view(np.uint32), (k, hp)


def test_argument_checks_before_any_device_call(lib_path):
    bad = [(0, 4, {}), (10, 0, {}), (10, z.ZERO1_MAX_WORLD + 1, {}), (10, 4, {"beta1": 1.0}),
           (10, 4, {"beta2": -0.1}), (10, 4, {"lr": float("nan")}), (10, 4, {"eps": -1.0}),
           (10, 4, {"weight_decay": float("inf")}), (10, 4, {"max_norm": float("nan")})]
    for n, world, hp in bad:
        with pytest.raises(z.Zero1Error) as e:
            z.zero1_create(n, world, z.Hparams(**hp))
        assert e.value.code == -1, (n, world, hp, str(e.value))
    with pytest.raises(z.Zero1Error) as e:
        z.zero1_step_scalars(z.Hparams(), 4, 0)
    assert e.value.code == -1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_create_without_device_reports_enodev(lib_path):
    with pytest.raises(z.Zero1Error) as e:
        z.zero1_create(4096, 4)
    assert e.value.code == -5


def test_unknown_handles_are_rejected_not_dereferenced(lib_path):
    bogus = 0xDEAD0000
    for call in (lambda: z.zero1_step(bogus, [16] * 4, [16] * 4),
                 lambda: z.zero1_set_lr(bogus, 1e-3),
                 lambda: z.zero1_layout(bogus),
                 lambda: z.zero1_get_state(bogus),
                 lambda: z.zero1_destroy(bogus),
                 lambda: z.zero1_step(None, [16], [16])):
        with pytest.raises(z.Zero1Error) as e:
            call()
        assert e.value.code == -1
    z.zero1_destroy(None)                      # NULL is accepted
    assert "invalid handle" in z.zero1_last_error() or z.zero1_last_error() == ""


def _declarations() -> dict[str, list[str]]:
    """Each declared entry point's parameter list, from include/zero1.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(zero1_\w+)\s*\(([^)]*)\)\s*;", text, flags=re.M | re.S):
        params = [p.strip() for p in m.group(2).replace("\n", " ").split(",")]
        out[m.group(1)] = [] if params == ["void"] or params == [""] else params
    return out


def test_binding_signatures_match_header():
    """The ctypes binding passes as many arguments as each C prototype takes,
    and pointer parameters are marshalled as pointers."""
    decls = _declarations()
    assert set(decls) == set(z.EXPORTED_SYMBOLS)
    for name, params in decls.items():
        _, args = z._SIGS[name]
        assert len(args) == len(params), (name, params, args)
        for p, a in zip(params, args):
            if "*" in p:
                assert a is C.c_void_p, (name, p)


def _struct_fields(name: str) -> list[tuple[str, str]]:
    text = open(HEADER).read()
    body = re.search(r"typedef struct(?: \w+)? \{([^}]*)\}\s*" + name + r";", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        ctype, names = decl.split(None, 1)
        for n in names.split(","):
            n = n.strip()
            fields.append((n.lstrip("*").strip(), ctype + "*" if n.startswith("*") else ctype))
    return fields


CTYPES = {"double": C.c_double, "uint32_t": C.c_uint32, "int32_t": C.c_int32, "uint64_t": C.c_uint64,
          "int": C.c_int, "void*": C.c_void_p}


@pytest.mark.parametrize("struct,binding", [("zero1_options", z._COptions), ("zero1_hparams", z._CHparams),
                                            ("zero1_sm_partition", z._CSmPartition)])
def test_structs_match_header(struct, binding):
    fields = _struct_fields(struct)
    assert [n for n, _ in fields] == [n for n, _ in binding._fields_]
    for (n, ctype), (_, bt) in zip(fields, binding._fields_):
        assert CTYPES[ctype] is bt, (struct, n, ctype, bt)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_options_checked_before_the_device(lib_path):
    """Valid options pass the checks (the call then finds no device); a wrong
    size or an out-of-range field is rejected first."""
    with pytest.raises(z.Zero1Error) as e:
        z.zero1_create_ex(4096, 4, None, z.Options(capturable=True, small_step=-1, moments_bf16=True,
                                                   load_phase_gbs=-1.0))
    assert e.value.code == -5
    lib = z._load()
    hp = z.Hparams()._c()
    h = C.c_void_p()
    for field, value in (("size", 8), ("small_step", 2), ("capturable", 3), ("inject_wait_timeout", 2),
                         ("bucket_ctas", -1), ("clip_eps", -1.0), ("load_phase_gbs", float("nan")),
                         ("load_phase_gbs", float("inf")), ("load_phase_gbs", 0.001), ("load_phase_gbs", 999.0)):
        opts = z.Options()._c()
        setattr(opts, field, value)
        assert lib.zero1_create_ex(4096, 4, C.byref(hp), C.byref(opts), C.byref(h)) == -1, field


def test_new_entry_points_reject_unknown_handles(lib_path):
    bogus = 0xDEAD0000
    for call in (lambda: z.zero1_step_host_async(bogus, [16], [16]),
                 lambda: z.zero1_host_sync(bogus),
                 lambda: z.zero1_profile_read(bogus, 4),
                 lambda: z.zero1_step_launches(bogus),
                 lambda: z.zero1_set_lr_ptr(bogus, 16),
                 lambda: z.zero1_bucket_begin(bogus),
                 lambda: z.zero1_allreduce_sum(bogus, [16], [16])):
        with pytest.raises(z.Zero1Error) as e:
            call()
        assert e.value.code == -1


def test_ptr_table_marshals_once():
    bufs = [torch.zeros(4), torch.zeros(4)]
    t = z.PtrTable(bufs)
    assert len(t) == 2
    assert [t.array[i] for i in range(2)] == [b.data_ptr() for b in bufs]
    assert z._ptrs(t) is t.array
    assert list(z._ptrs([16, None])) == [16, None]


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """Without the built library every entry point raises (no CPU fallback)."""
    monkeypatch.setattr(z, "_LIB_PATH", str(tmp_path / "libzero1.so"))
    monkeypatch.setattr(z, "_lib", None)
    for call in (lambda: z.zero1_create(4096, 4), lambda: z.zero1_shard_plan(10, 2),
                 lambda: z.Zero1(16, 2), lambda: z.zero1_last_error()):
        with pytest.raises(z.Zero1Error) as e:
            call()
        assert e.value.code == -5 and "not built" in str(e.value)


def test_binding_checks_pointer_counts_and_buffers(lib_path):
    """The binding refuses, before any C call, a pointer list whose length
    differs from the world size the C side reads, and buffers of the wrong
    type, place or size (the C side would read past the host array or hand
    the kernels addresses they cannot use)."""
    bf = lambda k: torch.zeros(k, dtype=torch.bfloat16)          # host tensors: never reach a kernel
    f32 = lambda k: torch.zeros(k, dtype=torch.float32)
    hp = z.Hparams()
    with pytest.raises(ValueError, match="3 pointers given, the call reads 4"):
        z.zero1_allreduce(16, 4, z.DTYPE_BF16, z.OP_SUM, [bf(16)] * 3, [bf(16)] * 4)
    with pytest.raises(ValueError, match="pointers given"):
        z.zero1_allgather(16, 4, 8, z.DTYPE_BF16, [0] * 4, [bf(16)] * 5)
    with pytest.raises(ValueError, match="pointers given"):
        z.zero1_step_noalloc(16, 2, hp, 1, [bf(16)], [bf(16)] * 2, f32(16), f32(16), f32(16))
    with pytest.raises(ValueError, match="CUDA tensor"):
        z.zero1_allreduce(16, 2, z.DTYPE_BF16, z.OP_SUM, [bf(16)] * 2, [bf(16)] * 2)
    with pytest.raises(ValueError, match="expected torch.float32"):
        z.zero1_step_noalloc(16, 2, hp, 1, [0, 0], [0, 0], bf(16), f32(16), f32(16))
    with pytest.raises(ValueError, match="elements, the call reads or writes 16"):
        z._check_buffer(f32(15), 16, "f32", None, "master")
    # host-buffer entry points want host memory of n entries per rank
    z._HANDLES[12345] = (16, 2, False)
    try:
        with pytest.raises(ValueError, match="pointers given"):
            z.zero1_step_host(12345, [bf(16)], [bf(16)] * 2)
        with pytest.raises(ValueError, match="elements, the call reads or writes 16"):
            z.zero1_step_host(12345, [bf(16), bf(8)], [bf(16)] * 2)
        with pytest.raises(ValueError, match="expected torch.float32"):
            z.zero1_get_state(12345, bf(16))
        with pytest.raises(ValueError, match="pointers given"):
            z.zero1_step(12345, z.PtrTable([0]), z.PtrTable([0, 0]))
    finally:
        z._HANDLES.pop(12345)
    # numpy host arrays are checked by element size and count
    with pytest.raises(ValueError, match="4-byte elements"):
        z._check_buffer(np.zeros(16, np.float32), 16, "bf16", False, "x")
    with pytest.raises(ValueError, match="host memory"):
        z._check_buffer(np.zeros(16, np.uint16), 16, "bf16", True, "x")
    z._check_buffer(np.zeros(16, np.uint16), 16, "bf16", False, "x")


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_sm_partition_errors_without_a_device(lib_path):
    with pytest.raises(z.Zero1Error) as e:
        z.zero1_sm_partition_create(0)
    assert e.value.code == -1
    with pytest.raises(z.Zero1Error) as e:
        z.zero1_sm_partition_create(16)
    assert e.value.code == -5
    z.zero1_sm_partition_destroy(z._CSmPartition())     # an empty partition is accepted
