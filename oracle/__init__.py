"""CPU oracle for the compressed Lion update step (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package; the CUDA
library and its Python binding never do.  The arithmetic lives in
``lioncub_oracle.c`` (plain single-threaded C, every float operation rounded
once, M1 in fp64); this module only builds it with gcc and marshals numpy
arrays into it.

Sources: "Lion Cub: Minimizing Communication Overhead in Distributed Lion"
(machine review page, "What carries the argument", Eq. (1)) and
"Communication Efficient Distributed Training with Distributed Lion"
(summary page, "Approach").  See the C header for the per-function map.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lioncub_oracle.c")
_HDR = os.path.join(_HERE, "lioncub_oracle.h")
_LIB = os.path.join(_HERE, "liblioncub_oracle.so")

MODE_SIGN = 0
MODE_L1 = 1
GRAD_BF16 = 0
GRAD_F32 = 1
TENSOR_SYNC_M = 1
FLAG_TIE_ALTERNATE = 0x100
FLAG_AVERAGE = 0x200

_lock = threading.Lock()
_lib = None


class Diag(ctypes.Structure):
    _fields_ = [("match", ctypes.c_int64), ("flip", ctypes.c_int64), ("dropped", ctypes.c_int64),
                ("spurious", ctypes.c_int64), ("ties", ctypes.c_int64), ("max_std_m", ctypes.c_float),
                ("pad", ctypes.c_uint32)]


DIAG_FIELDS = ("match", "flip", "dropped", "spurious", "ties", "max_std_m")


class QinfDiag(ctypes.Structure):
    _fields_ = [("match", ctypes.c_int64), ("flip", ctypes.c_int64), ("dropped", ctypes.c_int64),
                ("spurious", ctypes.c_int64), ("zero_codes", ctypes.c_int64)]


QINF_FIELDS = ("match", "flip", "dropped", "spurious", "zero_codes")


class Tensor(ctypes.Structure):
    _fields_ = [("offset", ctypes.c_int64), ("numel", ctypes.c_int64), ("flags", ctypes.c_uint32)]


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library next to its source."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the oracle failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            # LIONCUB_ORACLE_LIB: a separately built copy of this source (the
            # mutation test loads deliberately broken copies through it)
            path = os.environ.get("LIONCUB_ORACLE_LIB") or build()
            L = ctypes.CDLL(path)
            f32, i64, i32, u32 = ctypes.c_float, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
            vp = ctypes.c_void_p
            L.lco_omega.argtypes = [f32]
            L.lco_omega.restype = f32
            L.lco_update_vector.argtypes = [f32, f32, f32, f32]
            L.lco_update_vector.restype = f32
            L.lco_momentum.argtypes = [f32, f32, f32, f32]
            L.lco_momentum.restype = f32
            L.lco_sign_bit.argtypes = [f32, i64]
            L.lco_sign_bit.restype = i32
            L.lco_pack_signs.argtypes = [vp, i64, i64, vp]
            L.lco_pack_signs.restype = None
            L.lco_m1.argtypes = [vp, i64]
            L.lco_m1.restype = f32
            L.lco_q1.argtypes = [vp, i64, i32, f32, vp]
            L.lco_q1.restype = None
            L.lco_pack_codes.argtypes = [vp, i64, i32, vp]
            L.lco_pack_codes.restype = None
            L.lco_vote.argtypes = [vp, i32, i64]
            L.lco_vote.restype = ctypes.c_int32
            L.lco_code_sum.argtypes = [vp, i32, i32, i64]
            L.lco_code_sum.restype = ctypes.c_int32
            L.lco_direction.argtypes = [ctypes.c_int32, i32, u32, i64]
            L.lco_direction.restype = f32
            L.lco_apply.argtypes = [f32, f32, f32, f32]
            L.lco_apply.restype = f32
            L.lco_sync_average.argtypes = [vp, i32, i64, i64]
            L.lco_sync_average.restype = None
            L.lco_step.argtypes = [i64, i32, vp, i32, f32, f32, f32, f32, i32, i32, u32, i32, i64,
                                   i32, vp, vp, vp, vp, vp, vp]
            L.lco_step.restype = i32
            L.lco_worker_std.argtypes = [vp, i32]
            L.lco_worker_std.restype = f32
            L.lco_classify.argtypes = [f32, f32]
            L.lco_classify.restype = i32
            L.lco_diagnose.argtypes = [i64, i32, vp, i32, f32, i32, i32, u32, i64, i32, vp, vp, vp]
            L.lco_diagnose.restype = i32
            u64 = ctypes.c_uint64
            L.lco_splitmix64.argtypes = [u64, u64]
            L.lco_splitmix64.restype = u64
            L.lco_qinf_uniform.argtypes = [u64, i64, i32, i64]
            L.lco_qinf_uniform.restype = f32
            L.lco_maxabs.argtypes = [vp, i64]
            L.lco_maxabs.restype = f32
            L.lco_qinf.argtypes = [vp, i64, i32, f32, u64, i64, i32, i64, vp]
            L.lco_qinf.restype = None
            L.lco_diagnose_qinf.argtypes = [i64, i32, vp, i32, f32, i32, u32, i64, u64, i64, i32, vp, vp, vp]
            L.lco_diagnose_qinf.restype = i32
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ptr_array(arrs) -> ctypes.Array:
    return (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def layout_array(layout):
    """layout: sequence of (offset, numel, flags) -> ctypes array (or None)."""
    if not layout:
        return None, 0
    arr = (Tensor * len(layout))(*[Tensor(int(o), int(n), int(f)) for (o, n, f) in layout])
    return arr, len(layout)


# ---- single-operation helpers (scalars / small vectors) -------------------

def omega(beta: float) -> float:
    return lib().lco_omega(beta)


def update_vector(m: float, g: float, beta1: float, omega1: float) -> float:
    return lib().lco_update_vector(m, g, beta1, omega1)


def momentum(m: float, g: float, beta2: float, omega2: float) -> float:
    return lib().lco_momentum(m, g, beta2, omega2)


def sign_bit(c: float, t: int) -> int:
    return lib().lco_sign_bit(c, t)


def pack_signs(c: np.ndarray, t: int) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.float32)
    out = np.zeros(max(1, (c.size + 31) // 32), dtype=np.uint32)
    lib().lco_pack_signs(_ptr(c), c.size, t, _ptr(out))
    return out[: (c.size + 31) // 32]


def m1(c: np.ndarray) -> np.float32:
    c = np.ascontiguousarray(c, dtype=np.float32)
    return np.float32(lib().lco_m1(_ptr(c) if c.size else None, c.size))


def q1(c: np.ndarray, nbits: int, m1_value=None) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.float32)
    if m1_value is None:
        m1_value = m1(c)
    out = np.zeros(max(1, c.size), dtype=np.int8)
    lib().lco_q1(_ptr(c), c.size, nbits, float(m1_value), _ptr(out))
    return out[: c.size]


def pack_codes(q: np.ndarray, nbits: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8)
    nw = (q.size * nbits + 31) // 32
    out = np.zeros(max(1, nw), dtype=np.uint32)
    lib().lco_pack_codes(_ptr(q), q.size, nbits, _ptr(out))
    return out[:nw]


def vote(words, e: int) -> int:
    words = [np.ascontiguousarray(w, dtype=np.uint32) for w in words]
    return lib().lco_vote(ctypes.cast(_ptr_array(words), ctypes.c_void_p), len(words), e)


def code_sum(words, nbits: int, e: int) -> int:
    words = [np.ascontiguousarray(w, dtype=np.uint32) for w in words]
    return lib().lco_code_sum(ctypes.cast(_ptr_array(words), ctypes.c_void_p), len(words), nbits, e)


def direction(agg: int, W: int, flags: int, t: int) -> float:
    return lib().lco_direction(agg, W, flags, t)


def apply(theta: float, u: float, lr: float, wd: float) -> float:
    return lib().lco_apply(theta, u, lr, wd)


def sync_average(ms, lo: int, hi: int) -> None:
    """Average the float32 arrays in ``ms`` over [lo, hi) in place."""
    for a in ms:
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    ptrs = _ptr_array(ms)
    lib().lco_sync_average(ctypes.cast(ptrs, ctypes.c_void_p), len(ms), lo, hi)


# ---- the full step ---------------------------------------------------------

class StepOutputs:
    def __init__(self, wire, m1, agg):
        self.wire = wire  # list of W uint32 arrays
        self.m1 = m1      # (W, K) float32 or None
        self.agg = agg    # (d,) int32


def step(*, d: int, W: int, layout, beta1: float, beta2: float, lr: float, wd: float,
         mode: int, nbits: int, flags: int, sync_interval: int, t: int,
         grads, theta: np.ndarray, m, want_outputs: bool = True) -> StepOutputs:
    """One step of the method on host arrays; theta and m are updated in place.

    grads: list of W arrays, uint16 (bf16 bit patterns) or float32.
    """
    assert len(grads) == W and len(m) == W
    g0 = grads[0]
    if g0.dtype == np.uint16:
        gdt = GRAD_BF16
    elif g0.dtype == np.float32:
        gdt = GRAD_F32
    else:
        raise TypeError("gradients must be uint16 (bf16 bits) or float32")
    for g in grads:
        assert g.dtype == g0.dtype and g.size == d and g.flags["C_CONTIGUOUS"]
    assert theta.dtype == np.float32 and theta.size == d
    for a in m:
        assert a.dtype == np.float32 and a.size == d and a.flags["C_CONTIGUOUS"]
    lay, K = layout_array(layout)
    Keff = max(K, 1)
    bits = 1 if mode == MODE_SIGN else nbits
    nwords = (d * bits + 31) // 32
    wire = m1 = agg = None
    wire_p = m1_p = agg_p = None
    if want_outputs:
        wire = [np.zeros(max(1, nwords), dtype=np.uint32) for _ in range(W)]
        wire_p = ctypes.cast(_ptr_array(wire), ctypes.c_void_p)
        agg = np.zeros(max(1, d), dtype=np.int32)
        agg_p = _ptr(agg)
        if mode == MODE_L1:
            m1 = np.zeros((W, Keff), dtype=np.float32)
            m1_p = _ptr(m1)
    gp = _ptr_array(grads)
    mp = _ptr_array(m)
    rc = lib().lco_step(d, W, ctypes.cast(lay, ctypes.c_void_p) if lay is not None else None, K,
                        beta1, beta2, lr, wd, mode, nbits, flags, sync_interval, t, gdt,
                        ctypes.cast(gp, ctypes.c_void_p), _ptr(theta), ctypes.cast(mp, ctypes.c_void_p),
                        wire_p, m1_p, agg_p)
    if rc != 0:
        raise ValueError(f"oracle step rejected its arguments (rc={rc})")
    if want_outputs:
        wire = [w[:nwords] for w in wire]
        agg = agg[:d]
    return StepOutputs(wire, m1, agg)


# ---- diagnostics -------------------------------------------------------------

def worker_std(x) -> np.float32:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return np.float32(lib().lco_worker_std(_ptr(x), x.size))


def classify(u_q: float, u_fp: float) -> int:
    return lib().lco_classify(u_q, u_fp)


def diagnose(*, d: int, W: int, layout, beta1: float, mode: int, nbits: int, flags: int, t: int,
             grads, m):
    """Per-tensor diagnostics of one step (see lioncub_oracle.h); returns a
    list of dicts with the DIAG_FIELDS keys."""
    gdt = GRAD_BF16 if grads[0].dtype == np.uint16 else GRAD_F32
    lay, K = layout_array(layout)
    out = (Diag * max(K, 1))()
    rc = lib().lco_diagnose(d, W, ctypes.cast(lay, ctypes.c_void_p) if lay is not None else None, K,
                            beta1, mode, nbits, flags, t, gdt,
                            ctypes.cast(_ptr_array(grads), ctypes.c_void_p),
                            ctypes.cast(_ptr_array(m), ctypes.c_void_p), ctypes.addressof(out))
    if rc != 0:
        raise ValueError(f"oracle diagnose rejected its arguments (rc={rc})")
    return [{f: getattr(o, f) for f in DIAG_FIELDS} for o in out]


# ---- Q_inf: max-norm scaling with stochastic rounding -------------------------

def splitmix64(seed: int, k: int) -> int:
    """Output number k of SplitMix64 started from state `seed`."""
    return int(lib().lco_splitmix64(seed & (2**64 - 1), k & (2**64 - 1)))


def qinf_uniform(seed: int, t: int, worker: int, e: int) -> float:
    return float(lib().lco_qinf_uniform(seed & (2**64 - 1), t, worker, e))


def maxabs(c: np.ndarray) -> np.float32:
    c = np.ascontiguousarray(c, dtype=np.float32)
    return np.float32(lib().lco_maxabs(_ptr(c) if c.size else None, c.size))


def qinf(c: np.ndarray, nbits: int, *, seed: int, t: int, worker: int, e_first: int = 0,
         maxabs_value=None) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.float32)
    if maxabs_value is None:
        maxabs_value = maxabs(c)
    out = np.zeros(max(1, c.size), dtype=np.int8)
    lib().lco_qinf(_ptr(c), c.size, nbits, float(maxabs_value), seed & (2**64 - 1), t, worker, e_first, _ptr(out))
    return out[: c.size]


def diagnose_qinf(*, d: int, W: int, layout, beta1: float, nbits: int, flags: int, t: int, seed: int,
                  e_base: int, grads, m):
    """Per-tensor Q_inf comparison (see lioncub_oracle.h); list of dicts with
    the QINF_FIELDS keys."""
    gdt = GRAD_BF16 if grads[0].dtype == np.uint16 else GRAD_F32
    lay, K = layout_array(layout)
    out = (QinfDiag * max(K, 1))()
    rc = lib().lco_diagnose_qinf(d, W, ctypes.cast(lay, ctypes.c_void_p) if lay is not None else None, K,
                                 beta1, nbits, flags, t, seed & (2**64 - 1), e_base, gdt,
                                 ctypes.cast(_ptr_array(grads), ctypes.c_void_p),
                                 ctypes.cast(_ptr_array(m), ctypes.c_void_p), ctypes.addressof(out))
    if rc != 0:
        raise ValueError(f"oracle Q_inf diagnose rejected its arguments (rc={rc})")
    return [{f: getattr(o, f) for f in QINF_FIELDS} for o in out]
