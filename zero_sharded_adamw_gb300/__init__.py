"""GB300 (sm_103a) ZeRO-1 data-parallel optimizer step.

A thin ctypes binding of ``libzero1.so`` (C ABI in ``include/zero1.h``): the
functions below carry the C entry points' names and only marshal arguments.
Every step of the path runs in the library's CUDA kernels; there is no
CPU fallback.  The library is built by ``__graft_entry__.build()`` (or
``python -m zero_sharded_adamw_gb300._build``); calling any entry point
without it raises ``Zero1Error``.

Pointers may be given as ints or as objects with ``data_ptr()`` (torch
tensors) or ``ctypes.data`` (numpy arrays).  Streams may be ints, objects
with ``cuda_stream`` (torch streams) or None (the legacy default stream).
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

__all__ = [
    "Zero1Error", "Zero1ArgumentError", "Hparams", "Options", "Zero1", "PtrTable",
    "zero1_create", "zero1_create_ex", "zero1_destroy", "zero1_step", "zero1_step_host",
    "zero1_step_host_async", "zero1_host_sync",
    "zero1_set_state", "zero1_get_state", "zero1_set_state_range", "zero1_get_state_range",
    "zero1_set_lr", "zero1_set_lr_ptr", "zero1_get_grad_norm",
    "zero1_layout", "zero1_bucket_begin", "zero1_bucket_reduce", "zero1_bucket_update", "zero1_bucket_finish", "zero1_profile_start", "zero1_profile_stop", "zero1_profile_read", "zero1_step_launches", "zero1_shard_plan", "zero1_step_scalars", "zero1_step_noalloc", "zero1_allreduce", "zero1_allreduce_sum", "zero1_allgather", "zero1_last_error",
    "SmPartition", "zero1_sm_partition_create", "zero1_sm_partition_destroy",
    "library_path", "EXPORTED_SYMBOLS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libzero1.so")

ZERO1_MAX_WORLD = 512
ERRORS = {-1: "ZERO1_EINVAL", -2: "ZERO1_EALIGN", -3: "ZERO1_ENOMEM", -4: "ZERO1_ECUDA", -5: "ZERO1_ENODEV"}

# Every entry point include/zero1.h declares, with its ctypes signature.
_P, _U64, _I32, _F64 = C.c_void_p, C.c_uint64, C.c_int, C.c_double
_SIGS = {
    "zero1_create": (_I32, [_U64, _I32, _P, _P]),
    "zero1_create_ex": (_I32, [_U64, _I32, _P, _P, _P]),
    "zero1_destroy": (_I32, [_P]),
    "zero1_step": (_I32, [_P, _P, _P, _P]),
    "zero1_step_host": (_I32, [_P, _P, _P, _P]),
    "zero1_step_host_async": (_I32, [_P, _P, _P, _P]),
    "zero1_host_sync": (_I32, [_P]),
    "zero1_set_state": (_I32, [_P, _P, _P, _P, _U64, _P]),
    "zero1_get_state": (_I32, [_P, _P, _P, _P, _P, _P]),
    "zero1_set_state_range": (_I32, [_P, _U64, _U64, _P, _P, _P, _P]),
    "zero1_get_state_range": (_I32, [_P, _U64, _U64, _P, _P, _P, _P]),
    "zero1_set_lr": (_I32, [_P, _F64]),
    "zero1_set_lr_ptr": (_I32, [_P, _P]),
    "zero1_get_grad_norm": (_I32, [_P, _P, _P, _P]),
    "zero1_layout": (_I32, [_P, _P, _P, _P]),
    "zero1_bucket_begin": (_I32, [_P]),
    "zero1_bucket_reduce": (_I32, [_P, _U64, _U64, _P, _P]),
    "zero1_bucket_update": (_I32, [_P, _U64, _U64, _P, _P, _P]),
    "zero1_bucket_finish": (_I32, [_P, _P, _P]),
    "zero1_profile_start": (_I32, [_P, _I32]),
    "zero1_profile_stop": (_I32, [_P, _P, _P, _P]),
    "zero1_profile_read": (_I32, [_P, _P, _P, _U64, _P]),
    "zero1_step_launches": (_I32, [_P, _P]),
    "zero1_shard_plan": (_I32, [_U64, _I32, _P, _P]),
    "zero1_step_scalars": (_I32, [_P, _I32, _U64, _P]),
    "zero1_step_noalloc": (_I32, [_U64, _I32, _P, _U64, _P, _P, _P, _P, _P, _P]),
    "zero1_allreduce": (_I32, [_U64, _I32, _I32, _I32, _P, _P, _P, _P]),
    "zero1_allreduce_sum": (_I32, [_P, _P, _P, _P]),
    "zero1_allgather": (_I32, [_U64, _I32, _U64, _I32, _P, _P, _P, _P]),
    "zero1_sm_partition_create": (_I32, [_I32, _P]),
    "zero1_sm_partition_destroy": (_I32, [_P]),
    "zero1_last_error": (C.c_char_p, []),
}
EXPORTED_SYMBOLS = tuple(_SIGS)


class Zero1Error(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{ERRORS.get(code, code)}: {message}")
        self.code = code


class Zero1ArgumentError(Zero1Error, ValueError):
    """An argument the binding refused before calling the library (a pointer
    list whose length is not the world size, a buffer of the wrong type,
    place or size): code ZERO1_EINVAL, like the library's own checks."""

    def __init__(self, message: str):
        super().__init__(-1, message)


class _CHparams(C.Structure):
    _fields_ = [(k, C.c_double) for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "max_norm")]


@dataclass
class Hparams:
    """AdamW + clipping hyperparameters; max_norm <= 0 disables clipping."""
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    max_norm: float = 1.0

    def _c(self) -> _CHparams:
        return _CHparams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay, self.max_norm)


class _COptions(C.Structure):
    _fields_ = [("size", C.c_uint32), ("decay_before_update", C.c_int32), ("clip_eps", C.c_double),
                ("moments_bf16", C.c_int32), ("bucket_ctas", C.c_int32), ("small_step", C.c_int32),
                ("capturable", C.c_int32), ("inject_wait_timeout", C.c_int32), ("host_chunk", C.c_uint64),
                ("load_phase_gbs", C.c_double)]


@dataclass
class Options:
    """Step variants: torch.optim.AdamW's decay order, a clip eps (torch's
    clip_grad_norm_ uses 1e-6), m and v stored in bf16; the bucketed step's
    CTAs per bucket; the one-launch small-n path (0 auto, 1 on, -1 off);
    capturable steps (device-side step counter and lr, for CUDA graphs);
    the host-buffer steps' chunk size; the update kernel's load phasing
    (0 = built-in rule, > 0 = device-wide rate in GB/s, < 0 = off)."""
    decay_before_update: bool = False
    clip_eps: float = 0.0
    moments_bf16: bool = False
    bucket_ctas: int = 0
    small_step: int = 0
    capturable: bool = False
    inject_wait_timeout: bool = False    # failure testing: the update kernel's waits run out
    host_chunk: int = 0                  # host-buffer steps: parameters per chunk (0 = default)
    load_phase_gbs: float = 0.0          # update-kernel load phasing: 0 built-in, > 0 rate (GB/s), < 0 off

    def _c(self) -> _COptions:
        return _COptions(C.sizeof(_COptions), 1 if self.decay_before_update else 0, self.clip_eps,
                         1 if self.moments_bf16 else 0, self.bucket_ctas, self.small_step,
                         1 if self.capturable else 0, 1 if self.inject_wait_timeout else 0, self.host_chunk,
                         self.load_phase_gbs)


_lib = None


def library_path() -> str:
    return _LIB_PATH


def _load() -> C.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise Zero1Error(-5, f"{_LIB_PATH} is not built; run "
                                 "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != 0:
        raise Zero1Error(rc, _load().zero1_last_error().decode())


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):
        return int(x.ctypes.data)
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    return int(s.cuda_stream) or None


class PtrTable:
    """A pointer array built once (W buffers' addresses), for callers that
    pass the same buffers every step: it skips the per-call marshalling.
    It keeps references to the buffers so that they outlive the table."""

    def __init__(self, xs):
        self.buffers = list(xs)
        self.array = (C.c_void_p * len(self.buffers))(*[_addr(x) for x in self.buffers])
        self._checked: set = set()       # (count, kind, on_device) already validated

    def __len__(self) -> int:
        return len(self.buffers)


# Element kinds a C entry point expects behind a pointer: torch dtype name
# and element size in bytes.
_KINDS = {"bf16": ("torch.bfloat16", 2), "f32": ("torch.float32", 4)}


def _check_buffer(x, count: int, kind: str, on_device: bool | None, what: str) -> None:
    """Raise ValueError unless buffer `x` can hold `count` elements of `kind`
    where the C side will look for them (on_device: True = CUDA memory,
    False = host memory, None = either).  Raw integer addresses and None
    pass unchecked: only objects that describe themselves can be checked."""
    if x is None or isinstance(x, int):
        return
    want, size = _KINDS[kind]
    if hasattr(x, "data_ptr") and hasattr(x, "numel"):          # torch tensor
        if str(x.dtype) != want:
            raise Zero1ArgumentError(f"{what}: expected {want}, got {x.dtype}")
        if on_device is not None and bool(x.is_cuda) != on_device:
            raise Zero1ArgumentError(f"{what}: expected a {'CUDA' if on_device else 'host'} tensor, got {x.device}")
        if not x.is_contiguous():
            raise Zero1ArgumentError(f"{what}: tensor is not contiguous")
        if x.numel() < count:
            raise Zero1ArgumentError(f"{what}: {x.numel()} elements, the call reads or writes {count}")
    elif hasattr(x, "ctypes") and hasattr(x, "nbytes"):          # numpy array (host memory)
        if on_device:
            raise Zero1ArgumentError(f"{what}: a numpy array is host memory; this argument must be device memory")
        if x.itemsize != size:
            raise Zero1ArgumentError(f"{what}: {x.itemsize}-byte elements, expected {size}-byte {kind}")
        if not x.flags["C_CONTIGUOUS"]:
            raise Zero1ArgumentError(f"{what}: array is not contiguous")
        if x.size < count:
            raise Zero1ArgumentError(f"{what}: {x.size} elements, the call reads or writes {count}")


def _ptrs(xs, world: int | None = None, count: int | None = None, kind: str | None = None,
          on_device: bool | None = True, what: str = "buffers") -> C.Array:
    """The host array of W pointers the C side reads.  With `world` it must
    hold exactly W entries (the C side reads W of them); with `count` and
    `kind` every buffer is checked to hold that many elements of that type."""
    n = len(xs)
    if world is not None and n != world:
        raise Zero1ArgumentError(f"{what}: {n} pointers given, the call reads {world}")
    if isinstance(xs, PtrTable):
        if count is not None and kind is not None:
            key = (count, kind, on_device)
            if key not in xs._checked:
                for r, x in enumerate(xs.buffers):
                    _check_buffer(x, count, kind, on_device, f"{what}[{r}]")
                xs._checked.add(key)
        return xs.array
    if count is not None and kind is not None:
        for r, x in enumerate(xs):
            _check_buffer(x, count, kind, on_device, f"{what}[{r}]")
    return (C.c_void_p * n)(*[_addr(x) for x in xs])


# (n, world, moments in bf16) of every handle this binding created, so that
# the per-call checks know the sizes the C side will use.
_HANDLES: dict[int, tuple[int, int, bool]] = {}


def _info(h) -> tuple[int | None, int | None, bool]:
    return _HANDLES.get(h, (None, None, False))


# --------------------------------------------------------- entry points

def zero1_last_error() -> str:
    return _load().zero1_last_error().decode()


def zero1_create(n: int, world: int, hp: Hparams | None = None) -> int:
    """Create a handle for n parameters over `world` emulated ranks."""
    h = C.c_void_p()
    c = (hp or Hparams())._c()
    _check(_load().zero1_create(n, world, C.byref(c), C.byref(h)))
    _HANDLES[h.value] = (n, world, False)
    return h.value


def zero1_create_ex(n: int, world: int, hp: Hparams | None = None, opts: Options | None = None) -> int:
    """Create a handle with step variants."""
    h = C.c_void_p()
    c = (hp or Hparams())._c()
    o = (opts or Options())._c()
    _check(_load().zero1_create_ex(n, world, C.byref(c), C.byref(o), C.byref(h)))
    _HANDLES[h.value] = (n, world, bool(opts and opts.moments_bf16))
    return h.value


def zero1_destroy(h: int | None) -> None:
    _check(_load().zero1_destroy(h))
    _HANDLES.pop(h, None)


def zero1_step(h: int, grad_ptrs, param_ptrs, stream=None) -> None:
    """One step: W device gradient buffers in, W device replicas out."""
    n, world, _ = _info(h)
    _check(_load().zero1_step(h, _ptrs(grad_ptrs, world, n, "bf16", True, "grads"),
                              _ptrs(param_ptrs, world, n, "bf16", True, "params"), _stream(stream)))


def zero1_step_host(h: int, host_grads, host_params, stream=None) -> None:
    """One step from host gradient buffers into host replica buffers (waits)."""
    n, world, _ = _info(h)
    _check(_load().zero1_step_host(h, _ptrs(host_grads, world, n, "bf16", False, "host_grads"),
                                   _ptrs(host_params, world, n, "bf16", False, "host_params"), _stream(stream)))


def zero1_step_host_async(h: int, host_grads, host_params, stream=None) -> None:
    """Pipelined host-buffer step; host_params are valid after zero1_host_sync."""
    n, world, _ = _info(h)
    _check(_load().zero1_step_host_async(h, _ptrs(host_grads, world, n, "bf16", False, "host_grads"),
                                         _ptrs(host_params, world, n, "bf16", False, "host_params"),
                                         _stream(stream)))


def zero1_host_sync(h: int) -> None:
    _check(_load().zero1_host_sync(h))


def _check_state(h, count, master, m, v) -> None:
    """master fp32, m and v fp32 (bf16 on a moments_bf16 handle), each able
    to hold `count` elements, in host or device memory."""
    if count is None:
        return
    mom = "bf16" if _info(h)[2] else "f32"
    _check_buffer(master, count, "f32", None, "master")
    _check_buffer(m, count, mom, None, "m")
    _check_buffer(v, count, mom, None, "v")


def zero1_set_state(h: int, master, m=None, v=None, t: int = 0, stream=None) -> None:
    _check_state(h, _info(h)[0], master, m, v)
    _check(_load().zero1_set_state(h, _addr(master), _addr(m), _addr(v), t, _stream(stream)))


def zero1_get_state(h: int, master=None, m=None, v=None, stream=None) -> int:
    _check_state(h, _info(h)[0], master, m, v)
    t = C.c_uint64()
    _check(_load().zero1_get_state(h, _addr(master), _addr(m), _addr(v), C.byref(t), _stream(stream)))
    return t.value


def zero1_set_state_range(h: int, offset: int, count: int, master, m=None, v=None, stream=None) -> None:
    _check_state(h, count, master, m, v)
    _check(_load().zero1_set_state_range(h, offset, count, _addr(master), _addr(m), _addr(v), _stream(stream)))


def zero1_get_state_range(h: int, offset: int, count: int, master=None, m=None, v=None, stream=None) -> None:
    _check_state(h, count, master, m, v)
    _check(_load().zero1_get_state_range(h, offset, count, _addr(master), _addr(m), _addr(v), _stream(stream)))


def zero1_set_lr(h: int, lr: float) -> None:
    _check(_load().zero1_set_lr(h, lr))


def zero1_set_lr_ptr(h: int, device_lr=None) -> None:
    """Capturable handles: read lr from a device float64 (None: own slot)."""
    _check(_load().zero1_set_lr_ptr(h, _addr(device_lr)))


def zero1_get_grad_norm(h: int, stream=None) -> tuple[float, float]:
    norm, clip = C.c_double(), C.c_float()
    _check(_load().zero1_get_grad_norm(h, C.byref(norm), C.byref(clip), _stream(stream)))
    return norm.value, clip.value


def zero1_layout(h: int) -> tuple[int, int, int]:
    s, p, b = C.c_uint64(), C.c_uint64(), C.c_uint64()
    _check(_load().zero1_layout(h, C.byref(s), C.byref(p), C.byref(b)))
    return s.value, p.value, b.value


def zero1_bucket_begin(h: int) -> None:
    _check(_load().zero1_bucket_begin(h))


def zero1_bucket_reduce(h: int, offset: int, count: int, grad_ptrs, stream=None) -> None:
    """Reduce-scatter one bucket: grad_ptrs[r] holds rank r's gradient for
    parameters [offset, offset+count)."""
    world = _info(h)[1]
    _check(_load().zero1_bucket_reduce(h, offset, count, _ptrs(grad_ptrs, world, count, "bf16", True, "grads"),
                                       _stream(stream)))


def zero1_bucket_update(h: int, offset: int, count: int, grad_ptrs, param_ptrs, stream=None) -> None:
    """Reduce-scatter and update one bucket (handles without clipping)."""
    world = _info(h)[1]
    _check(_load().zero1_bucket_update(h, offset, count, _ptrs(grad_ptrs, world, count, "bf16", True, "grads"),
                                       _ptrs(param_ptrs, world, count, "bf16", True, "params"), _stream(stream)))


def zero1_bucket_finish(h: int, param_ptrs, stream=None) -> None:
    n, world, _ = _info(h)
    table = None if param_ptrs is None else _ptrs(param_ptrs, world, n, "bf16", True, "params")
    _check(_load().zero1_bucket_finish(h, table, _stream(stream)))


def zero1_profile_start(h: int, capacity: int) -> None:
    _check(_load().zero1_profile_start(h, capacity))


def zero1_profile_stop(h: int) -> tuple[float, float, int]:
    """(summed reduce-scatter+norm ms, summed update+all-gather ms, steps)."""
    a, b, n = C.c_double(), C.c_double(), C.c_uint64()
    _check(_load().zero1_profile_stop(h, C.byref(a), C.byref(b), C.byref(n)))
    return a.value, b.value, n.value


def zero1_step_launches(h: int) -> int:
    """Kernel launches per zero1_step: 2, or 1 on the one-launch small-n path."""
    k = C.c_int()
    _check(_load().zero1_step_launches(h, C.byref(k)))
    return k.value


def zero1_profile_read(h: int, capacity: int) -> tuple[list[float], list[float]]:
    """Per-step (reduce-scatter+norm ms, update+all-gather ms) recorded so far."""
    a, b, n = (C.c_float * max(1, capacity))(), (C.c_float * max(1, capacity))(), C.c_uint64()
    _check(_load().zero1_profile_read(h, a, b, capacity, C.byref(n)))
    k = min(n.value, capacity)
    return list(a[:k]), list(b[:k])


def zero1_shard_plan(n: int, world: int) -> tuple[int, int]:
    """Shard length S and padded length W*S (host only, no device)."""
    s, p = C.c_uint64(), C.c_uint64()
    _check(_load().zero1_shard_plan(n, world, C.byref(s), C.byref(p)))
    return s.value, p.value


def zero1_step_scalars(hp: Hparams, world: int, t: int) -> dict:
    """The fp32 scalars step t uses (host only, no device)."""
    out = (C.c_float * 8)()
    c = hp._c()
    _check(_load().zero1_step_scalars(C.byref(c), world, t, out))
    keys = ("inv_w", "beta1", "one_minus_beta1", "beta2", "one_minus_beta2", "step_size", "decay", "eps")
    return dict(zip(keys, list(out)))


def zero1_step_noalloc(n: int, world: int, hp: Hparams, t: int, grad_ptrs, param_ptrs,
                       master, m, v, stream=None) -> None:
    """One step with caller-owned fp32 state and the library's fixed scratch
    (no device allocation; n <= 4,194,304)."""
    c = hp._c()
    grads = _ptrs(grad_ptrs, world, n, "bf16", True, "grads")
    params = _ptrs(param_ptrs, world, n, "bf16", True, "params")
    for x, name in ((master, "master"), (m, "m"), (v, "v")):
        _check_buffer(x, n, "f32", True, name)
    _check(_load().zero1_step_noalloc(n, world, C.byref(c), t, grads, params,
                                      _addr(master), _addr(m), _addr(v), _stream(stream)))


DTYPE_BF16, DTYPE_F32 = 0, 1
OP_SUM, OP_AVG = 0, 1


def zero1_allreduce(n: int, world: int, dtype: int, op: int, in_ptrs, out_ptrs, errors=None, stream=None) -> None:
    """DDP all-reduce of W device buffers (bf16 or fp32, sum or mean)."""
    kind = {DTYPE_BF16: "bf16", DTYPE_F32: "f32"}.get(dtype)
    _check(_load().zero1_allreduce(n, world, dtype, op, _ptrs(in_ptrs, world, n, kind, True, "in"),
                                   _ptrs(out_ptrs, world, n, kind, True, "out"), _addr(errors),
                                   _stream(stream)))


def zero1_allreduce_sum(h: int, in_ptrs, out_ptrs, stream=None) -> None:
    """bf16 sum all-reduce over the handle's W ranks of n elements each."""
    n, world, _ = _info(h)
    _check(_load().zero1_allreduce_sum(h, _ptrs(in_ptrs, world, n, "bf16", True, "in"),
                                       _ptrs(out_ptrs, world, n, "bf16", True, "out"), _stream(stream)))


def zero1_allgather(n: int, world: int, shard_len: int, dtype: int, shard_ptrs, out_ptrs, errors=None,
                    stream=None) -> None:
    """ZeRO-3 parameter all-gather: rank r's shard holds [r*S, min((r+1)*S, n))."""
    kind = {DTYPE_BF16: "bf16", DTYPE_F32: "f32"}.get(dtype)
    shards = _ptrs(shard_ptrs, world, None, None, True, "shards")
    if kind is not None and not isinstance(shard_ptrs, PtrTable):
        for r, x in enumerate(shard_ptrs):
            own = max(0, min(shard_len, n - r * shard_len))
            if own:
                _check_buffer(x, own, kind, True, f"shards[{r}]")
    _check(_load().zero1_allgather(n, world, shard_len, dtype, shards, _ptrs(out_ptrs, world, n, kind, True, "out"),
                                   _addr(errors), _stream(stream)))


class _CSmPartition(C.Structure):
    _fields_ = [("stream_a", C.c_void_p), ("stream_b", C.c_void_p), ("sms_a", C.c_int), ("sms_b", C.c_int),
                ("opaque", C.c_void_p)]


def zero1_sm_partition_create(sms_a: int) -> _CSmPartition:
    """Two streams on disjoint SM groups of the current device (green
    contexts): the first with at least sms_a SMs, the second with the rest."""
    part = _CSmPartition()
    _check(_load().zero1_sm_partition_create(sms_a, C.byref(part)))
    return part


def zero1_sm_partition_destroy(part: _CSmPartition) -> None:
    _check(_load().zero1_sm_partition_destroy(C.byref(part)))


class SmPartition:
    """Owning wrapper of zero1_sm_partition_create: ``stream_a`` / ``stream_b``
    are the raw cudaStream_t values (wrap them with torch.cuda.ExternalStream),
    ``sms_a`` / ``sms_b`` the SMs each group was granted."""

    def __init__(self, sms_a: int):
        self._part = zero1_sm_partition_create(sms_a)
        self.stream_a, self.stream_b = self._part.stream_a, self._part.stream_b
        self.sms_a, self.sms_b = self._part.sms_a, self._part.sms_b

    def close(self) -> None:
        """Wait for both streams' work, then release the green contexts."""
        if self._part is not None:
            part, self._part = self._part, None
            zero1_sm_partition_destroy(part)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


class Zero1:
    """Owning wrapper around a handle (closes on ``close()`` / context exit)."""

    def __init__(self, n: int, world: int, hp: Hparams | None = None, opts: Options | None = None):
        self.n, self.world, self.hp, self.opts = n, world, hp or Hparams(), opts or Options()
        self.handle = zero1_create_ex(n, world, self.hp, self.opts)

    def step(self, grads, params, stream=None) -> None:
        zero1_step(self.handle, grads, params, stream)

    def step_host(self, grads, params, stream=None) -> None:
        zero1_step_host(self.handle, grads, params, stream)

    def step_host_async(self, grads, params, stream=None) -> None:
        zero1_step_host_async(self.handle, grads, params, stream)

    def host_sync(self) -> None:
        zero1_host_sync(self.handle)

    def launches_per_step(self) -> int:
        return zero1_step_launches(self.handle)

    def set_state(self, master, m=None, v=None, t: int = 0, stream=None) -> None:
        zero1_set_state(self.handle, master, m, v, t, stream)

    def get_state(self, master=None, m=None, v=None, stream=None) -> int:
        return zero1_get_state(self.handle, master, m, v, stream)

    def set_lr(self, lr: float) -> None:
        zero1_set_lr(self.handle, lr)

    def set_lr_ptr(self, device_lr=None) -> None:
        zero1_set_lr_ptr(self.handle, device_lr)

    def grad_norm(self, stream=None) -> tuple[float, float]:
        return zero1_get_grad_norm(self.handle, stream)

    def layout(self) -> tuple[int, int, int]:
        return zero1_layout(self.handle)

    def close(self) -> None:
        if self.handle is not None:
            zero1_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
