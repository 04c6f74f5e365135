"""Python access to the CPU oracle in ``zero1_ref.c``.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this module.  It shares no code with
the CUDA library and the library never imports it.

Arrays are numpy: bf16 values travel as ``uint16`` bit patterns, fp32 state as
``float32``.  Every function is a thin ctypes marshalling layer over the C
oracle; the arithmetic lives in ``zero1_ref.c`` only.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero1_ref.c")
_LIB = os.path.join(_HERE, "libzero1_ref.so")

# -O2 without contraction, fast-math or flush-to-zero: every fp32 operation in
# the oracle is one IEEE round-to-nearest-even operation, on x86-64 and on
# aarch64 alike (gcc contracts a*b+c into an FMA by default on aarch64).
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library next to its source; return its path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


class Hparams(C.Structure):
    _fields_ = [(k, C.c_double) for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "max_norm")]


class Scalars(C.Structure):
    _fields_ = [(k, C.c_float) for k in (
        "inv_w", "beta1", "one_minus_beta1", "beta2", "one_minus_beta2", "step_size", "decay", "eps")]


class NormAcc(C.Structure):
    _fields_ = [("sum", C.c_double), ("comp", C.c_double), ("plain", C.c_double)]


def _signatures():
    P = C.c_void_p
    u64, i32, f32, f64 = C.c_uint64, C.c_int, C.c_float, C.c_double
    return {
        "zref_bf16_to_f32": (f32, [C.c_uint16]),
        "zref_f32_to_bf16": (C.c_uint16, [f32]),
        "zref_bf16_to_f32_array": (None, [P, u64, P]),
        "zref_f32_to_bf16_array": (None, [P, u64, P]),
        "zref_shard_len": (u64, [u64, i32]),
        "zref_step_scalars": (None, [P, i32, u64, P]),
        "zref_rs_mean_range": (None, [P, i32, u64, f32, P]),
        "zref_reduce_scatter_mean": (None, [P, i32, u64, P]),
        "zref_norm_acc_init": (None, [P]),
        "zref_norm_acc_add": (None, [P, P, u64]),
        "zref_norm_acc_value": (f64, [P]),
        "zref_clip_coef": (f32, [f64, f64]),
        "zref_adamw_range": (None, [P, P, P, P, u64, f32, P]),
        "zref_all_gather_bf16": (None, [P, i32, u64, P, i32]),
        "zref_step": (None, [u64, i32, P, u64, P, P, P, P, P, P, i32, f32, P, P]),
        "zref_allreduce_sum_direct": (None, [P, i32, u64, P]),
        "zref_allreduce_rs_ag": (None, [P, i32, u64, i32, P, P]),
        "zref_clip_coef_ex": (f32, [f64, f64, f64]),
        "zref_adamw_range_ex": (None, [P, P, P, P, u64, f32, P, P]),
        "zref_step_ex": (None, [u64, i32, P, P, u64, P, P, P, P, P, P, i32, f32, P, P]),
        "zref_allreduce_f32_direct": (None, [P, i32, u64, i32, P]),
        "zref_allreduce_f32_rs_ag": (None, [P, i32, u64, i32, P, P]),
        "zref_all_gather_shards": (None, [C.c_size_t, P, i32, u64, u64, P]),
        "zref_zero_bytes_per_rank": (f64, [i32, f64, i32, f64]),
        "zref_ring_send_bytes": (f64, [f64, i32, i32]),
    }


def load(path: str) -> C.CDLL:
    """Load an oracle shared library from ``path`` with its C signatures."""
    L = C.CDLL(path)
    for name, (res, args) in _signatures().items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


_lib = None


def lib() -> C.CDLL:
    """The oracle library in use (the one built from ``zero1_ref.c``)."""
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def use(L: C.CDLL | None) -> C.CDLL | None:
    """Swap the library every function below calls; return the previous one.

    The mutation tests use this to run the pins against a copy of the oracle
    with a planted mistake."""
    global _lib
    prev = _lib
    _lib = L
    return prev


# ----------------------------------------------------------------- helpers

def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _ptr_array(arrs) -> C.Array:
    return (C.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 data travels as uint16 bit patterns"
    return a


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.float32
    return a


@dataclass
class HP:
    """AdamW + clipping hyperparameters (max_norm <= 0 disables clipping)."""
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    max_norm: float = 1.0

    def c(self) -> Hparams:
        return Hparams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay, self.max_norm)


# ------------------------------------------------------------- bf16 codec

def bf16_to_f32(b) -> np.ndarray:
    b = _u16(np.asarray(b, dtype=np.uint16))
    out = np.empty(b.shape, dtype=np.float32)
    lib().zref_bf16_to_f32_array(_ptr(b), b.size, _ptr(out))
    return out


def f32_to_bf16(x) -> np.ndarray:
    x = _f32(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint16)
    lib().zref_f32_to_bf16_array(_ptr(x), x.size, _ptr(out))
    return out


# ---------------------------------------------------------------- pieces

def shard_len(n: int, world: int) -> int:
    return int(lib().zref_shard_len(n, world))


def step_scalars(hp: HP, world: int, t: int) -> dict:
    s = Scalars()
    h = hp.c()
    lib().zref_step_scalars(C.byref(h), world, t, C.byref(s))
    return {k: getattr(s, k) for k, _ in Scalars._fields_}


def reduce_scatter_mean(grads) -> np.ndarray:
    grads = [_u16(g) for g in grads]
    n = grads[0].size
    out = np.empty(n, dtype=np.float32)
    lib().zref_reduce_scatter_mean(_ptr_array(grads), len(grads), n, _ptr(out))
    return out


def rs_mean_range(grads, world: int | None = None) -> np.ndarray:
    """Element-wise rank-ordered mean of equally long bf16 windows."""
    grads = [_u16(g) for g in grads]
    w = len(grads) if world is None else world
    out = np.empty(grads[0].size, dtype=np.float32)
    lib().zref_rs_mean_range(_ptr_array(grads), len(grads), grads[0].size,
                             C.c_float(np.float32(1.0 / w)), _ptr(out))
    return out


class NormAccumulator:
    """Streaming index-order norm: add chunks in order, read the norm."""

    def __init__(self):
        self.acc = NormAcc()
        lib().zref_norm_acc_init(C.byref(self.acc))

    def add(self, x: np.ndarray) -> None:
        x = _f32(x)
        lib().zref_norm_acc_add(C.byref(self.acc), _ptr(x), x.size)

    def value(self) -> float:
        return float(lib().zref_norm_acc_value(C.byref(self.acc)))


def l2_norm(x: np.ndarray) -> float:
    a = NormAccumulator()
    a.add(x)
    return a.value()


def clip_coef(norm: float, max_norm: float) -> np.float32:
    return np.float32(lib().zref_clip_coef(norm, max_norm))


def adamw_range(master, m, v, ghat, c: float, scalars: dict) -> None:
    """In-place AdamW on fp32 arrays given the step's scalars dict."""
    arrs = [_f32(a) for a in (master, m, v, ghat)]
    for a, orig in zip(arrs[:3], (master, m, v)):
        assert a is orig or np.shares_memory(a, orig), "state must be contiguous float32"
    s = Scalars(*[scalars[k] for k, _ in Scalars._fields_])
    lib().zref_adamw_range(*[_ptr(a) for a in arrs], arrs[0].size, C.c_float(c), C.byref(s))


def all_gather_bf16(master: np.ndarray, world: int, n_replicas: int | None = None):
    master = _f32(master)
    reps = [np.empty(master.size, dtype=np.uint16) for _ in range(n_replicas or world)]
    lib().zref_all_gather_bf16(_ptr(master), world, master.size, _ptr_array(reps), len(reps))
    return reps


# ------------------------------------------------------------- full step

class State:
    """fp32 master / m / v for n parameters plus the 1-based step counter."""

    def __init__(self, master: np.ndarray, m: np.ndarray | None = None, v: np.ndarray | None = None, t: int = 0):
        self.master = np.array(master, dtype=np.float32, copy=True)
        self.m = np.zeros_like(self.master) if m is None else np.array(m, dtype=np.float32, copy=True)
        self.v = np.zeros_like(self.master) if v is None else np.array(v, dtype=np.float32, copy=True)
        self.t = int(t)

    def copy(self) -> "State":
        return State(self.master, self.m, self.v, self.t)


def step(state: State, grads, hp: HP, clip_override: float | None = None):
    """Advance ``state`` by one ZeRO-1 step; return (replicas, norm, clip)."""
    grads = [_u16(g) for g in grads]
    world, n = len(grads), grads[0].size
    assert all(g.size == n for g in grads)
    state.t += 1
    reps = [np.empty(n, dtype=np.uint16) for _ in range(world)]
    ghat = np.empty(n, dtype=np.float32)
    norm = C.c_double()
    clip = C.c_float()
    h = hp.c()
    lib().zref_step(n, world, C.byref(h), state.t, _ptr_array(grads), _ptr_array(reps),
                    _ptr(state.master), _ptr(state.m), _ptr(state.v), _ptr(ghat),
                    1 if clip_override is not None else 0,
                    C.c_float(0.0 if clip_override is None else clip_override),
                    C.byref(norm), C.byref(clip))
    return reps, float(norm.value), np.float32(clip.value)


class _COptions(C.Structure):
    _fields_ = [("decay_before_update", C.c_int), ("clip_eps", C.c_double), ("moments_bf16", C.c_int)]


@dataclass
class Options:
    """Step variants: torch's decay-first order, clip eps, bf16 moments."""
    decay_before_update: bool = False
    clip_eps: float = 0.0
    moments_bf16: bool = False

    def c(self) -> _COptions:
        return _COptions(1 if self.decay_before_update else 0, self.clip_eps, 1 if self.moments_bf16 else 0)


def state_ex(master, options: Options) -> State:
    """A fresh state (m = v = 0) whose moments have the options' storage type."""
    st = State(master)
    if options.moments_bf16:
        st.m = np.zeros(st.master.size, np.uint16)
        st.v = np.zeros(st.master.size, np.uint16)
    return st


def clip_coef_ex(norm: float, max_norm: float, clip_eps: float) -> np.float32:
    return np.float32(lib().zref_clip_coef_ex(norm, max_norm, clip_eps))


def adamw_range_ex(master, m, v, ghat, c: float, scalars: dict, options: Options) -> None:
    s = Scalars(*[scalars[k] for k, _ in Scalars._fields_])
    o = options.c()
    for a in (master, m, v, ghat):
        assert a.flags["C_CONTIGUOUS"]
    lib().zref_adamw_range_ex(_ptr(master), _ptr(m), _ptr(v), _ptr(ghat), master.size, C.c_float(c),
                              C.byref(s), C.byref(o))


def step_ex(state: State, grads, hp: HP, options: Options, clip_override: float | None = None):
    """One step with options; state.m/state.v are uint16 when moments_bf16."""
    grads = [_u16(g) for g in grads]
    world, n = len(grads), grads[0].size
    want = np.uint16 if options.moments_bf16 else np.float32
    assert state.m.dtype == want and state.v.dtype == want
    state.t += 1
    reps = [np.empty(n, dtype=np.uint16) for _ in range(world)]
    ghat = np.empty(n, dtype=np.float32)
    norm, clip = C.c_double(), C.c_float()
    h, o = hp.c(), options.c()
    lib().zref_step_ex(n, world, C.byref(h), C.byref(o), state.t, _ptr_array(grads), _ptr_array(reps),
                       _ptr(state.master), _ptr(state.m), _ptr(state.v), _ptr(ghat),
                       1 if clip_override is not None else 0,
                       C.c_float(0.0 if clip_override is None else clip_override),
                       C.byref(norm), C.byref(clip))
    return reps, float(norm.value), np.float32(clip.value)


def allreduce_sum_direct(inputs):
    inputs = [_u16(x) for x in inputs]
    outs = [np.empty(inputs[0].size, dtype=np.uint16) for _ in inputs]
    lib().zref_allreduce_sum_direct(_ptr_array(inputs), len(inputs), inputs[0].size, _ptr_array(outs))
    return outs


def allreduce_rs_ag(inputs, average: bool = False):
    inputs = [_u16(x) for x in inputs]
    n = inputs[0].size
    scratch = np.empty(n, dtype=np.float32)
    outs = [np.empty(n, dtype=np.uint16) for _ in inputs]
    lib().zref_allreduce_rs_ag(_ptr_array(inputs), len(inputs), n, 1 if average else 0,
                               _ptr(scratch), _ptr_array(outs))
    return outs, scratch


def allreduce_f32_direct(inputs, average: bool = False):
    inputs = [_f32(x) for x in inputs]
    outs = [np.empty(inputs[0].size, dtype=np.float32) for _ in inputs]
    lib().zref_allreduce_f32_direct(_ptr_array(inputs), len(inputs), inputs[0].size, 1 if average else 0,
                                    _ptr_array(outs))
    return outs


def allreduce_f32_rs_ag(inputs, average: bool = False):
    inputs = [_f32(x) for x in inputs]
    n = inputs[0].size
    scratch = np.empty(n, dtype=np.float32)
    outs = [np.empty(n, dtype=np.float32) for _ in inputs]
    lib().zref_allreduce_f32_rs_ag(_ptr_array(inputs), len(inputs), n, 1 if average else 0,
                                   _ptr(scratch), _ptr_array(outs))
    return outs, scratch


def all_gather_shards(shards, n: int, shard_len: int):
    """Rank r's shard holds elements [r*S, min((r+1)*S, n)); returns the W
    gathered n-element outputs (same dtype as the shards)."""
    shards = [np.ascontiguousarray(s) for s in shards]
    dt = shards[0].dtype
    outs = [np.empty(n, dtype=dt) for _ in shards]
    keep = [s if s.size else np.empty(1, dtype=dt) for s in shards]
    lib().zref_all_gather_shards(dt.itemsize, _ptr_array(keep), len(shards), n, shard_len, _ptr_array(outs))
    return outs


def zero_bytes_per_rank(stage: int, psi: float, world: int, k: float = 12.0) -> float:
    return float(lib().zref_zero_bytes_per_rank(stage, psi, world, k))


def ring_send_bytes(size: float, world: int, op: str) -> float:
    return float(lib().zref_ring_send_bytes(size, world, {"all_reduce": 0, "reduce_scatter": 1, "all_gather": 2}[op]))
