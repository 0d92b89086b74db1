"""Host-only checks of the C ABI library and the workload definitions.

No GPU is touched: the library is loaded, every symbol that include/lioncub.h
declares must be exported, and argument validation (which runs before any
CUDA call) must return the documented codes.  (A layout that passes
validation goes on to the device set-up, which fails without a GPU.)
"""
import ctypes
import os
import re

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lc():
    from communication_compressed_sign_gb300 import build
    build.build()
    from communication_compressed_sign_gb300 import lioncub
    lioncub.load()
    return lioncub


def _declared():
    with open(os.path.join(ROOT, "include", "lioncub.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"LIONCUB_API[^;(]*?\b(lioncub_\w+)\s*\(", text)))


def test_header_symbols_exported(lc):
    declared = _declared()
    assert len(declared) == 25
    lib = ctypes.CDLL(lc.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(lc.EXPORTED) == declared


def test_host_alloc_argument_checks(lc):
    """The page-locked allocator validates its arguments before touching
    CUDA: a NULL out pointer is ERR_ARG, zero bytes gives NULL and OK."""
    L = lc.load()
    assert L.lioncub_host_alloc(None, 64) == lc.ERR_ARG
    p = ctypes.c_void_p(1234)
    assert L.lioncub_host_alloc(ctypes.byref(p), 0) == lc.OK
    assert not p.value
    L.lioncub_host_free(None)  # a no-op


def test_create_validation_codes(lc):
    L = lc.load()
    h = ctypes.c_void_p()

    def create(d, W, layout, mode=0, nbits=1, grad=0, interval=0):
        if layout:
            arr = (lc.Tensor * len(layout))(*[lc.Tensor(*t) for t in layout])
            return L.lioncub_create(ctypes.byref(h), d, W, ctypes.cast(arr, ctypes.c_void_p), len(layout),
                                    0.9, 0.99, 1e-4, 0.1, mode, nbits, grad, interval)
        return L.lioncub_create(ctypes.byref(h), d, W, None, 0, 0.9, 0.99, 1e-4, 0.1, mode, nbits, grad,
                                interval)

    assert create(100, 0, None) == lc.ERR_ARG
    assert create(100, lc.MAX_WORKERS + 1, None) == lc.ERR_ARG
    assert create(-1, 2, None) == lc.ERR_ARG
    assert create(100, 2, None, mode=1, nbits=3) == lc.ERR_ARG
    assert "nbits" in lc.lioncub_last_error(None)
    assert create(100, 2, None, mode=7) == lc.ERR_ARG
    assert create(100, 2, None, grad=5) == lc.ERR_ARG
    assert create(100, 2, None, interval=-1) == lc.ERR_ARG
    assert create(100, 2, None, mode=1 | lc.FLAG_AVERAGE, nbits=4) == lc.ERR_ARG
    assert create(100, 2, None, mode=lc.FLAG_AVERAGE | lc.FLAG_TIE_ALTERNATE) == lc.ERR_ARG
    assert create(100, 2, None, mode=0x400) == lc.ERR_ARG
    assert create(64, 2, [(0, 40, 0), (40, 24, 0)]) == lc.ERR_ALIGN
    assert "multiple of 32" in lc.lioncub_last_error(None)
    assert create(64, 2, [(0, 32, 0), (48, 16, 0)]) == lc.ERR_ALIGN
    assert create(64, 2, [(0, 32, 0), (32, 16, 0)]) == lc.ERR_ARG      # does not reach d
    assert create(64, 2, [(0, 32, 0), (0, 32, 0)]) == lc.ERR_ARG       # overlaps
    assert create(64, 2, [(0, 64, 4)]) == lc.ERR_ARG                   # unknown tensor flag
    assert h.value is None


def _layout_expected(d, layout):
    """The documented layout contract, written independently of the library:
    tensors tile [0, d) in order, every offset a multiple of 32 (checked first
    for each tensor), non-negative sizes, known flags only."""
    nxt = 0
    for (off, n, fl) in layout:
        if off % 32:
            return "align"
        if off != nxt or n < 0:
            return "arg"
        if fl & ~1:
            return "arg"
        nxt += n
    return "ok" if nxt == d else "arg"


def test_create_layout_fuzz(lc):
    """Random layouts (ragged, overlapping, gapped, misaligned, negative,
    unknown flags) get the error the contract predicts; valid ones reach
    the device set-up (ERR_CUDA without a GPU, a handle with one)."""
    L = lc.load()
    rng = np.random.default_rng(2024)
    sizes = [0, 1, 31, 32, 33, 64, 100, 2048, 4096 + 7]
    counts = {"ok": 0, "arg": 0, "align": 0}
    for _ in range(400):
        K = int(rng.integers(1, 7))
        layout, off = [], 0
        for k in range(K):
            n = int(rng.choice(sizes))
            if k < K - 1 and rng.random() < 0.7:
                n = (n + 31) // 32 * 32  # inner tensors usually keep the next offset aligned
            o = off
            r = rng.random()
            if r < 0.05:
                o += 32            # gap
            elif r < 0.10:
                o -= 32            # overlap
            elif r < 0.15:
                o += 1             # misaligned
            if rng.random() < 0.03:
                n = -n - 1         # negative size
            fl = int(rng.choice([0, 0, 0, 1, 2]))
            layout.append((o, n, fl))
            off = o + max(n, 0)
        d = sum(max(n, 0) for (_, n, _) in layout) + (int(rng.integers(-2, 3)) if rng.random() < 0.1 else 0)
        d = max(d, 0)
        want = _layout_expected(d, layout)
        counts[want] += 1
        arr = (lc.Tensor * K)(*[lc.Tensor(*t) for t in layout])
        h = ctypes.c_void_p()
        rc = L.lioncub_create(ctypes.byref(h), d, 2, ctypes.cast(arr, ctypes.c_void_p), K, 0.9, 0.99, 1e-4,
                              0.1, 0, 1, 0, 0)
        if want == "ok":
            assert rc in (lc.OK, lc.ERR_CUDA, lc.ERR_OOM), (layout, d, rc)
            if rc == lc.OK:
                L.lioncub_destroy(h)
        else:
            assert rc == (lc.ERR_ALIGN if want == "align" else lc.ERR_ARG), (layout, d, rc, want)
            assert h.value is None
    assert min(counts.values()) >= 20, counts


def test_null_handle_paths(lc):
    L = lc.load()
    assert L.lioncub_step(None, None, None) == lc.ERR_ARG
    assert L.lioncub_bind_state(None, None, None) == lc.ERR_ARG
    assert L.lioncub_wire_words(None) == -1
    assert L.lioncub_set_lr(None, 1.0) == lc.ERR_ARG
    L.lioncub_destroy(None)
    assert lc.lioncub_strerror(lc.ERR_ALIGN) == "LIONCUB_ERR_ALIGN"
    assert lc.lioncub_strerror(-99) == "LIONCUB_ERR_UNKNOWN"


def test_binding_fails_loudly_without_library(tmp_path):
    from communication_compressed_sign_gb300 import lioncub
    saved = lioncub._lib
    lioncub._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            lioncub.load(str(tmp_path / "liblioncub.so"))
    finally:
        lioncub._lib = saved


@pytest.mark.parametrize("key,d,K", [(1, 1_048_576, 1), (2, 124_439_808, 148), (3, 354_823_168, 292),
                                     (4, 354_823_168, 292), (5, 1_416_552_448, 293),
                                     (6, 86_567_656, 152), (7, 5_543_716, 152)])
def test_workload_layouts(key, d, K):
    """Parameter counts: GPT-2 small 124,439,808 and medium 354,823,168
    (tied heads), the 1.3B layout with an untied head, ViT-B/16 86,567,656
    (1000 classes), DeiT-Tiny with a 100-class head 5,543,716."""
    wl = synth.workloads()[key]
    assert wl.d == d and len(wl.layout) == K
    off = 0
    for (_, o, n, _) in wl.layout:
        assert o == off and o % 32 == 0
        off += n
    flagged = [t[0] for t in wl.layout if t[3]]
    want = {4: ["wte"], 7: ["patch_embed.w", "patch_embed.b", "cls_token", "pos_embed", "head.w", "head.b"]}
    assert flagged == want.get(key, [])


def test_bench_byte_model():
    import bench
    W = synth.workloads()
    # sign mode: W*(G + 8 + 1/8) + W/8 + 8 bytes per parameter
    b = bench.step_bytes(W[2])
    assert abs(b / W[2].d - (8 * (2 + 8 + 1 / 8) + 8 / 8 + 8)) < 1e-3
    # L1 mode: W*(G+4) + W*(G+8+n/8) + W*n/8 + 8
    b = bench.step_bytes(W[3])
    assert abs(b / W[3].d - (8 * 6 + 8 * (2 + 8 + 0.5) + 8 * 0.5 + 8)) < 1e-3
    b = bench.step_bytes(W[5])
    assert abs(b / W[5].d - (8 * 6 + 8 * (2 + 8 + 0.25) + 8 * 0.25 + 8)) < 1e-3


def test_bench_labels_and_vision_byte_model():
    """The bench's mode and sync labels come from the workload; the byte
    model covers the D-Lion average (a sign-mode step) and L1 with sync."""
    import bench
    W = synth.workloads()
    assert bench.mode_label(W[2]) == "sign+majority"
    assert bench.mode_label(W[3]) == "L1 n=4 + int sum"
    assert bench.mode_label(W[6]) == "sign + D-Lion average"
    assert bench.sync_label(W[2]) == "none"
    assert bench.sync_label(W[4]) == "wte every step"
    assert bench.sync_label(W[7]).startswith("patch_embed.w, patch_embed.b, cls_token, pos_embed, head.w, head.b")
    b = bench.step_bytes(W[6])
    assert abs(b / W[6].d - (8 * (2 + 8 + 1 / 8) + 8 / 8 + 8)) < 1e-3
    b = bench.step_bytes(W[7])
    assert abs(b / W[7].d - (8 * 6 + 8 * (2 + 8 + 0.5) + 8 * 0.5 + 8)) < 1e-3


def test_header_constants_match_binding(lc):
    """Every LIONCUB_* enum value of the header equals the binding's constant."""
    with open(os.path.join(ROOT, "include", "lioncub.h")) as f:
        text = f.read()
    values = {}
    for body in re.findall(r"enum\s*\{(.*?)\}", text, re.S):
        body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
        for name, val in re.findall(r"(LIONCUB_\w+)\s*=\s*([-0-9xA-Fa-f]+)", body):
            values[name] = int(val, 0)
    expect = {
        "LIONCUB_TENSOR_SYNC_M": lc.TENSOR_SYNC_M, "LIONCUB_MODE_SIGN_MAJORITY": lc.MODE_SIGN_MAJORITY,
        "LIONCUB_MODE_L1_INTSUM": lc.MODE_L1_INTSUM, "LIONCUB_FLAG_TIE_ALTERNATE": lc.FLAG_TIE_ALTERNATE,
        "LIONCUB_FLAG_AVERAGE": lc.FLAG_AVERAGE, "LIONCUB_GRAD_BF16": lc.GRAD_BF16, "LIONCUB_GRAD_F32": lc.GRAD_F32,
        "LIONCUB_OK": lc.OK, "LIONCUB_ERR_ARG": lc.ERR_ARG, "LIONCUB_ERR_ALIGN": lc.ERR_ALIGN,
        "LIONCUB_ERR_STATE": lc.ERR_STATE, "LIONCUB_ERR_OOM": lc.ERR_OOM, "LIONCUB_ERR_CUDA": lc.ERR_CUDA,
        "LIONCUB_MAX_WORKERS": lc.MAX_WORKERS, "LIONCUB_EXPORT_WIRE": lc.EXPORT_WIRE,
        "LIONCUB_EXPORT_M1": lc.EXPORT_M1, "LIONCUB_EXPORT_AGG": lc.EXPORT_AGG,
        "LIONCUB_EXPORT_STATUS": lc.EXPORT_STATUS, "LIONCUB_KERNEL_COMPRESS": lc.KERNEL_COMPRESS,
        "LIONCUB_KERNEL_M1": lc.KERNEL_M1, "LIONCUB_KERNEL_M1_FINAL": lc.KERNEL_M1_FINAL,
        "LIONCUB_KERNEL_REDUCE_APPLY": lc.KERNEL_REDUCE_APPLY, "LIONCUB_KERNEL_DIAGNOSE": lc.KERNEL_DIAGNOSE,
        "LIONCUB_KERNEL_COUNT": lc.KERNEL_COUNT, "LIONCUB_NOALLOC_MAX_WORDS": lc.NOALLOC_MAX_WORDS,
        "LIONCUB_STATUS_WAIT_TIMEOUT": lc.STATUS_WAIT_TIMEOUT, "LIONCUB_STATUS_OUT_OF_BOUNDS": lc.STATUS_OUT_OF_BOUNDS,
        "LIONCUB_STATUS_GUARD": lc.STATUS_GUARD,
        "LIONCUB_DIST_SEND": lc.DIST_SEND, "LIONCUB_DIST_RECV": lc.DIST_RECV,
        "LIONCUB_DIST_DIR_CHUNK": lc.DIST_DIR_CHUNK, "LIONCUB_DIST_DIR_ALL": lc.DIST_DIR_ALL,
        "LIONCUB_DIST_AGG": lc.DIST_AGG, "LIONCUB_DIST_SYNC_SEND": lc.DIST_SYNC_SEND,
        "LIONCUB_DIST_SYNC_RECV": lc.DIST_SYNC_RECV, "LIONCUB_DIST_BUFFERS": lc.DIST_BUFFERS,
    }
    assert set(values) == set(expect), set(values) ^ set(expect)
    for name, v in expect.items():
        assert values[name] == v, name
    # struct layouts the binding assumes
    assert ctypes.sizeof(lc.Tensor) == 24
    assert lc.DIAG_BYTES == 48
    assert ctypes.sizeof(lc.DistPlan) == 104


def test_dist_calls_check_their_handle(lc):
    """The data-parallel calls refuse a NULL handle and bad plans without
    touching CUDA; a plan is host arithmetic and needs no device."""
    L = lc.load()
    assert L.lioncub_dist_compress(None, None, None) == lc.ERR_ARG
    assert L.lioncub_dist_reduce(None, None) == lc.ERR_ARG
    assert L.lioncub_dist_apply(None, None) == lc.ERR_ARG
    assert L.lioncub_dist_bind_buffers(None, None) == lc.ERR_ARG
    assert L.lioncub_dist_plan_make(100, 4, 2, 0, None, 0, 0, 1, 0, None) == lc.ERR_ARG
    p = lc.lioncub_dist_plan_make(1 << 20, 8, 4, 3, None, lc.MODE_L1_INTSUM, 4, 0)
    assert (p.local_workers, p.first_worker, p.agg_bytes) == (2, 6, 1)  # 8 * 7 = 56 fits int8
    assert p.bytes[lc.DIST_AGG] == 1 << 20 and p.bytes[lc.DIST_SEND] == 0
    p = lc.lioncub_dist_plan_make(1 << 20, 32, 4, 3, None, lc.MODE_L1_INTSUM, 4, 0)
    assert p.agg_bytes == 4  # 32 * 7 = 224 does not
