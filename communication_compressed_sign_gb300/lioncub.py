"""ctypes binding of liblioncub.so (the C ABI in include/lioncub.h).

Argument marshalling only: every step of the method runs in the library's
CUDA kernels.  Functions keep the C names; pointers are passed as Python
ints (for example ``tensor.data_ptr()``) and streams as the raw
``cudaStream_t`` value (``torch.cuda.Stream.cuda_stream``).  A non-zero
return code raises :class:`LionCubError` with the library's message.

If the library has not been built the first call raises; there is no other
implementation to fall back on.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
# LIONCUB_LIBRARY may name another build of the same library (the tests use
# the bounds-checked build this way).
LIB_PATH = os.environ.get("LIONCUB_LIBRARY") or os.path.join(_PKG, "liblioncub.so")

# enums of include/lioncub.h
TENSOR_SYNC_M = 1
MODE_SIGN_MAJORITY = 0
MODE_L1_INTSUM = 1
FLAG_TIE_ALTERNATE = 0x100
FLAG_AVERAGE = 0x200
GRAD_BF16 = 0
GRAD_F32 = 1
OK, ERR_ARG, ERR_ALIGN, ERR_STATE, ERR_OOM, ERR_CUDA = 0, -1, -2, -3, -4, -5
MAX_WORKERS = 128
EXPORT_WIRE, EXPORT_M1, EXPORT_AGG, EXPORT_STATUS = 0, 1, 2, 3
STATUS_WAIT_TIMEOUT, STATUS_OUT_OF_BOUNDS, STATUS_GUARD = 1, 2, 4
KERNEL_COMPRESS, KERNEL_M1, KERNEL_M1_FINAL, KERNEL_REDUCE_APPLY, KERNEL_DIAGNOSE, KERNEL_COUNT = 0, 1, 2, 3, 4, 5
KERNEL_NAMES = {KERNEL_COMPRESS: "compress", KERNEL_M1: "m1_partial",
                KERNEL_M1_FINAL: "m1_finalize", KERNEL_REDUCE_APPLY: "reduce_apply",
                KERNEL_DIAGNOSE: "diagnose"}
DIAG_FIELDS = ("match", "flip", "dropped", "spurious", "ties", "max_std_m")
DIAG_BYTES = 48
QINF_FIELDS = ("match", "flip", "dropped", "spurious", "zero_codes")
QINF_BYTES = 40

# Every symbol the header declares, for load checks.
EXPORTED = (
    "lioncub_create", "lioncub_bind_state", "lioncub_step", "lioncub_step_host",
    "lioncub_set_lr", "lioncub_get_step", "lioncub_set_step", "lioncub_wire_words",
    "lioncub_debug_export", "lioncub_profile", "lioncub_profile_read",
    "lioncub_last_error", "lioncub_strerror", "lioncub_destroy", "lioncub_sign_step_noalloc",
    "lioncub_diagnose", "lioncub_host_alloc", "lioncub_host_free",
    "lioncub_dist_plan_make", "lioncub_dist_create", "lioncub_dist_bind_buffers", "lioncub_dist_compress",
    "lioncub_dist_reduce", "lioncub_dist_apply", "lioncub_diagnose_qinf",
)
# exchange buffers of the data-parallel step (LIONCUB_DIST_*)
DIST_SEND, DIST_RECV, DIST_DIR_CHUNK, DIST_DIR_ALL, DIST_AGG, DIST_SYNC_SEND, DIST_SYNC_RECV = range(7)
DIST_BUFFERS = 7
DIST_BUFFER_NAMES = ("send", "recv", "dir_chunk", "dir_all", "agg", "sync_send", "sync_recv")
NOALLOC_MAX_WORDS = 4194304


class LionCubError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{message} [{code}]")
        self.code = code


class Tensor(ctypes.Structure):
    _fields_ = [("offset", ctypes.c_int64), ("numel", ctypes.c_int64), ("flags", ctypes.c_uint32)]


class DistPlan(ctypes.Structure):
    """lioncub_dist_plan: where the exchange of one rank puts what."""
    _fields_ = [("chunk", ctypes.c_int64), ("chunk_words", ctypes.c_int64), ("dir_words", ctypes.c_int64),
                ("sync_slots", ctypes.c_int64), ("local_workers", ctypes.c_int32),
                ("first_worker", ctypes.c_int32), ("dir_bits", ctypes.c_int32), ("agg_bytes", ctypes.c_int32),
                ("bytes", ctypes.c_int64 * 7)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load liblioncub.so (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m communication_compressed_sign_gb300.build`")
        L = ctypes.CDLL(path)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        L.lioncub_create.argtypes = [ctypes.POINTER(vp), i64, i32, vp, i32, f32, f32, f32, f32, i32,
                                     i32, i32, i32]
        L.lioncub_bind_state.argtypes = [vp, vp, vp]
        L.lioncub_step.argtypes = [vp, vp, vp]
        L.lioncub_step_host.argtypes = [vp, vp, vp, vp]
        L.lioncub_set_lr.argtypes = [vp, f32]
        L.lioncub_get_step.argtypes = [vp, ctypes.POINTER(i64)]
        L.lioncub_set_step.argtypes = [vp, i64]
        L.lioncub_wire_words.argtypes = [vp]
        L.lioncub_wire_words.restype = i64
        L.lioncub_debug_export.argtypes = [vp, i32, vp, vp]
        L.lioncub_profile.argtypes = [vp, i32]
        L.lioncub_profile_read.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]
        L.lioncub_last_error.argtypes = [vp]
        L.lioncub_last_error.restype = ctypes.c_char_p
        L.lioncub_strerror.argtypes = [i32]
        L.lioncub_strerror.restype = ctypes.c_char_p
        L.lioncub_destroy.argtypes = [vp]
        L.lioncub_destroy.restype = None
        L.lioncub_sign_step_noalloc.argtypes = [i64, i32, f32, f32, f32, f32, i64, i32, vp, vp, vp, vp]
        L.lioncub_sign_step_noalloc.restype = i32
        L.lioncub_diagnose.argtypes = [vp, vp, vp, vp]
        L.lioncub_diagnose.restype = i32
        L.lioncub_diagnose_qinf.argtypes = [vp, vp, i32, ctypes.c_uint64, vp, vp]
        L.lioncub_diagnose_qinf.restype = i32
        L.lioncub_host_alloc.argtypes = [ctypes.POINTER(vp), ctypes.c_size_t]
        L.lioncub_host_alloc.restype = i32
        L.lioncub_host_free.argtypes = [vp]
        L.lioncub_host_free.restype = None
        L.lioncub_dist_plan_make.argtypes = [i64, i32, i32, i32, vp, i32, i32, i32, i32, ctypes.POINTER(DistPlan)]
        L.lioncub_dist_create.argtypes = [ctypes.POINTER(vp), i64, i32, i32, i32, vp, i32, f32, f32, f32, f32,
                                          i32, i32, i32, i32]
        L.lioncub_dist_bind_buffers.argtypes = [vp, vp]
        L.lioncub_dist_compress.argtypes = [vp, vp, vp]
        L.lioncub_dist_reduce.argtypes = [vp, vp]
        L.lioncub_dist_apply.argtypes = [vp, vp]
        for name in ("lioncub_dist_plan_make", "lioncub_dist_create", "lioncub_dist_bind_buffers",
                     "lioncub_dist_compress", "lioncub_dist_reduce", "lioncub_dist_apply"):
            getattr(L, name).restype = i32
        for name in ("lioncub_create", "lioncub_bind_state", "lioncub_step", "lioncub_step_host",
                     "lioncub_set_lr", "lioncub_get_step", "lioncub_set_step",
                     "lioncub_debug_export", "lioncub_profile", "lioncub_profile_read"):
            getattr(L, name).restype = i32
        _lib = L
        return L


def _check(rc: int, h) -> None:
    if rc != OK:
        L = load()
        msg = L.lioncub_last_error(h).decode() or L.lioncub_strerror(rc).decode()
        raise LionCubError(rc, msg)


def _ptrs(values) -> ctypes.Array:
    return (ctypes.c_void_p * len(values))(*[int(v) for v in values])


def lioncub_create(d: int, W: int, layout, beta1: float, beta2: float, lr: float, wd: float,
                   mode: int, nbits: int, grad_dtype: int, sync_interval: int) -> int:
    """layout: sequence of (offset, numel, flags), or None/empty for one tensor."""
    L = load()
    h = ctypes.c_void_p()
    if layout:
        arr = (Tensor * len(layout))(*[Tensor(int(o), int(n), int(f)) for (o, n, f) in layout])
        lp, K = ctypes.cast(arr, ctypes.c_void_p), len(layout)
    else:
        lp, K = None, 0
    rc = L.lioncub_create(ctypes.byref(h), d, W, lp, K, beta1, beta2, lr, wd, mode, nbits, grad_dtype,
                          sync_interval)
    _check(rc, None)
    return h.value


def lioncub_bind_state(h: int, theta_ptr: int, m_ptrs) -> None:
    _check(load().lioncub_bind_state(h, theta_ptr, ctypes.cast(_ptrs(m_ptrs), ctypes.c_void_p)), h)


def lioncub_step(h: int, grad_ptrs, stream: int = 0) -> None:
    _check(load().lioncub_step(h, ctypes.cast(_ptrs(grad_ptrs), ctypes.c_void_p), stream or None), h)


def lioncub_step_host(h: int, grad_host_ptrs, theta_host_out_ptr: int, stream: int = 0) -> None:
    _check(load().lioncub_step_host(h, ctypes.cast(_ptrs(grad_host_ptrs), ctypes.c_void_p),
                                    theta_host_out_ptr, stream or None), h)


def lioncub_host_alloc(nbytes: int) -> int:
    """Page-locked, device-mapped host memory for lioncub_step_host; 0 for 0 bytes."""
    p = ctypes.c_void_p()
    _check(load().lioncub_host_alloc(ctypes.byref(p), nbytes), None)
    return p.value or 0


def lioncub_host_free(ptr: int) -> None:
    load().lioncub_host_free(ptr or None)


class HostBuffer:
    """A lioncub_host_alloc block viewed as a CPU torch tensor of `numel`
    elements of `dtype`; the memory is released by close() (or when the
    object is collected).  Keep the object alive while the tensor is used."""

    def __init__(self, numel: int, dtype):
        import torch
        itemsize = torch.empty(0, dtype=dtype).element_size()
        self.nbytes = int(numel) * itemsize
        self.ptr = lioncub_host_alloc(self.nbytes)
        if self.nbytes:
            raw = (ctypes.c_char * self.nbytes).from_address(self.ptr)
            self.tensor = torch.frombuffer(raw, dtype=dtype, count=int(numel))
        else:
            self.tensor = torch.empty(0, dtype=dtype)

    def data_ptr(self) -> int:
        return self.ptr

    def close(self) -> None:
        if self.ptr:
            self.tensor = None
            lioncub_host_free(self.ptr)
            self.ptr = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def lioncub_set_lr(h: int, lr: float) -> None:
    _check(load().lioncub_set_lr(h, lr), h)


def lioncub_get_step(h: int) -> int:
    t = ctypes.c_int64()
    _check(load().lioncub_get_step(h, ctypes.byref(t)), h)
    return t.value


def lioncub_set_step(h: int, t: int) -> None:
    _check(load().lioncub_set_step(h, t), h)


def lioncub_wire_words(h: int) -> int:
    return load().lioncub_wire_words(h)


def lioncub_debug_export(h: int, what: int, dst_ptr: int, stream: int = 0) -> None:
    _check(load().lioncub_debug_export(h, what, dst_ptr, stream or None), h)


def lioncub_diagnose(h: int, grad_ptrs, out_ptr: int, stream: int = 0) -> None:
    """Fill K lioncub_diag records (48 bytes each) at device address out_ptr."""
    _check(load().lioncub_diagnose(h, ctypes.cast(_ptrs(grad_ptrs), ctypes.c_void_p), out_ptr, stream or None), h)


def lioncub_diagnose_qinf(h: int, grad_ptrs, nbits: int, seed: int, out_ptr: int, stream: int = 0) -> None:
    """Fill K lioncub_qinf_diag records (40 bytes each) at device address out_ptr."""
    _check(load().lioncub_diagnose_qinf(h, ctypes.cast(_ptrs(grad_ptrs), ctypes.c_void_p), nbits,
                                        seed & (2**64 - 1), out_ptr, stream or None), h)


def decode_qinf(raw: bytes, K: int):
    """Host bytes of K lioncub_qinf_diag records -> list of dicts."""
    import struct
    return [dict(zip(QINF_FIELDS, struct.unpack_from("<5q", raw, k * QINF_BYTES))) for k in range(K)]


def decode_diag(raw: bytes, K: int):
    """Host bytes of K lioncub_diag records -> list of dicts."""
    import struct
    out = []
    for k in range(K):
        vals = struct.unpack_from("<5qfI", raw, k * DIAG_BYTES)
        out.append(dict(zip(DIAG_FIELDS, vals[:6])))
    return out


def lioncub_profile(h: int, max_steps: int) -> None:
    _check(load().lioncub_profile(h, max_steps), h)


def lioncub_profile_read(h: int, kernel: int):
    ms = ctypes.c_double()
    n = ctypes.c_int64()
    _check(load().lioncub_profile_read(h, kernel, ctypes.byref(ms), ctypes.byref(n)), h)
    return ms.value, n.value


def lioncub_last_error(h) -> str:
    return load().lioncub_last_error(h).decode()


def lioncub_strerror(code: int) -> str:
    return load().lioncub_strerror(code).decode()


def lioncub_sign_step_noalloc(d: int, W: int, beta1: float, beta2: float, lr: float, wd: float, t: int,
                              grad_dtype: int, grad_ptrs, theta_ptr: int, m_ptrs, stream: int = 0) -> None:
    """Handle-less sign-mode step that allocates nothing (see include/lioncub.h)."""
    rc = load().lioncub_sign_step_noalloc(d, W, beta1, beta2, lr, wd, t, grad_dtype,
                                          ctypes.cast(_ptrs(grad_ptrs), ctypes.c_void_p), theta_ptr,
                                          ctypes.cast(_ptrs(m_ptrs), ctypes.c_void_p), stream or None)
    _check(rc, None)


def _layout_arg(layout):
    if layout:
        arr = (Tensor * len(layout))(*[Tensor(int(o), int(n), int(f)) for (o, n, f) in layout])
        return arr, ctypes.cast(arr, ctypes.c_void_p), len(layout)
    return None, None, 0


def lioncub_dist_plan_make(d: int, W: int, nranks: int, rank: int, layout, mode: int, nbits: int,
                           sync_interval: int) -> DistPlan:
    """The exchange plan of one rank (host arithmetic only; no device needed)."""
    keep, lp, K = _layout_arg(layout)
    plan = DistPlan()
    _check(load().lioncub_dist_plan_make(d, W, nranks, rank, lp, K, mode, nbits, sync_interval,
                                         ctypes.byref(plan)), None)
    return plan


def lioncub_dist_create(d: int, W: int, nranks: int, rank: int, layout, beta1: float, beta2: float, lr: float,
                        wd: float, mode: int, nbits: int, grad_dtype: int, sync_interval: int) -> int:
    keep, lp, K = _layout_arg(layout)
    h = ctypes.c_void_p()
    rc = load().lioncub_dist_create(ctypes.byref(h), d, W, nranks, rank, lp, K, beta1, beta2, lr, wd, mode, nbits,
                                    grad_dtype, sync_interval)
    _check(rc, None)
    return h.value


def lioncub_dist_bind_buffers(h: int, ptrs) -> None:
    """ptrs: DIST_BUFFERS device addresses (0 where the plan needs none)."""
    assert len(ptrs) == DIST_BUFFERS
    _check(load().lioncub_dist_bind_buffers(h, ctypes.cast(_ptrs([p or 0 for p in ptrs]), ctypes.c_void_p)), h)


def lioncub_dist_compress(h: int, grad_ptrs, stream: int = 0) -> None:
    _check(load().lioncub_dist_compress(h, ctypes.cast(_ptrs(grad_ptrs), ctypes.c_void_p), stream or None), h)


def lioncub_dist_reduce(h: int, stream: int = 0) -> None:
    _check(load().lioncub_dist_reduce(h, stream or None), h)


def lioncub_dist_apply(h: int, stream: int = 0) -> None:
    _check(load().lioncub_dist_apply(h, stream or None), h)


def lioncub_destroy(h: int) -> None:
    if h:
        load().lioncub_destroy(h)
