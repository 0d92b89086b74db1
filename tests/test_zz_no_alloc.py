"""The allocation-free sign-mode entry point against the handle-based one and
against the oracle.

lioncub_sign_step_noalloc exists for callers that cannot allocate device
memory when they run a step (an allocator that owns all device memory, code
that must avoid the synchronization cudaMalloc can cause, plug-ins that only
allocate at initialisation).  It keeps its packed sign words in a fixed 16 MiB
array of the library's static device memory.  Here it must produce exactly
the theta and momenta of lioncub_step (sign mode is bit-exact) on four calls
in a row, reusing the shared array; on the small sizes it must also equal
the CPU oracle bit for bit.  A block of gradients is zero on every worker at
every step, so the momenta stay 0 there and the update vector is an exact
zero at both step parities: the alternating-zero rule ("Lion Cub", "What
carries the argument") sends +1 on even steps and -1 on odd ones, which the
handle path's exported words and theta's closed form show.  A d == 0 call
is the set-up call a caller makes while it initialises; sizes beyond the
array are refused.

The file is named to be collected last, so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ZERO_BLOCK = 64  # elements [0, 64) of every worker's gradient are 0 at every step
STEPS = 4


@pytest.fixture(scope="module")
def lc():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from communication_compressed_sign_gb300 import lioncub
    lioncub.load()
    return lioncub


def _workload(d, W, grad, seed):
    dist = ("normal", 1e-3) if grad == "f32" else ("t", 3.0, 1e-3, 0.0, 1.0)
    return synth.Workload(0, "noalloc", W, synth.flat_layout(d), grad, dist, 0, 1, STEPS, seed=seed)


def _zero_mask(d):
    mask = torch.zeros(d, dtype=torch.bool)
    mask[:ZERO_BLOCK] = True
    mask[::7] = True
    return mask


def _host_bits(g, grad):
    x = g.cpu()
    return x.view(torch.int16).numpy().view(np.uint16).copy() if grad == "bf16" else x.numpy().copy()


@pytest.mark.parametrize("d,W,grad", [(1_000_003, 8, "bf16"), (16_777_216, 8, "bf16"), (70_001, 5, "f32"),
                                      (33, 1, "bf16")])
def test_noalloc_matches_handle_path(lc, d, W, grad):
    import oracle

    dev = torch.device("cuda", 0)
    wl = _workload(d, W, grad, seed=d % 1000)
    with_oracle = d <= 100_000
    theta_a = torch.empty(d, dtype=torch.float32, device=dev)
    synth.fill_theta_(theta_a, wl)
    m_a = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
    theta_b = theta_a.clone()
    m_b = [x.clone() for x in m_a]
    theta_o = theta_a.cpu().numpy().copy() if with_oracle else None
    m_o = [np.zeros(d, np.float32) for _ in range(W)] if with_oracle else None
    gdt = synth.grad_dtype(wl)
    gcode = lc.GRAD_F32 if grad == "f32" else lc.GRAD_BF16
    grads = [torch.empty(d, dtype=gdt, device=dev) for _ in range(W)]
    zero = _zero_mask(d).to(dev)
    nwords = (d + 31) // 32
    wire = torch.empty((W, nwords), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream

    h = lc.lioncub_create(d, W, None, wl.beta1, wl.beta2, wl.lr, wl.wd, lc.MODE_SIGN_MAJORITY, 1, gcode, 0)
    try:
        lc.lioncub_bind_state(h, theta_a.data_ptr(), [x.data_ptr() for x in m_a])
        for t in range(STEPS):  # consecutive calls share (and reuse) the static array
            for i in range(W):
                synth.fill_grad_(grads[i], wl, t, i)
                grads[i][zero] = 0
            gp = [g.data_ptr() for g in grads]
            theta_prev = theta_b[:ZERO_BLOCK].cpu().numpy().copy()
            lc.lioncub_step(h, gp, stream)
            lc.lioncub_debug_export(h, lc.EXPORT_WIRE, wire.data_ptr(), stream)
            lc.lioncub_sign_step_noalloc(d, W, wl.beta1, wl.beta2, wl.lr, wl.wd, t, gcode, gp,
                                         theta_b.data_ptr(), [x.data_ptr() for x in m_b], stream)
            torch.cuda.synchronize()
            assert lc.lioncub_last_error(None) == ""
            assert torch.equal(theta_a.view(torch.int32), theta_b.view(torch.int32)), t
            for x, y in zip(m_a, m_b):
                assert torch.equal(x.view(torch.int32), y.view(torch.int32)), t

            # the exact-zero block: every worker sends +1 on even steps, -1 on odd ones
            zero_word = 0xFFFFFFFF if t % 2 == 0 else 0
            words = wire[:, 0].cpu().numpy().view(np.uint32)
            if d >= 32:
                assert (words == zero_word).all(), (t, words)
            u = 1.0 if t % 2 == 0 else -1.0
            want = np.array([oracle.apply(float(x), u, wl.lr, wl.wd) for x in theta_prev[:min(d, ZERO_BLOCK)]],
                            np.float32)
            got = theta_b[:min(d, ZERO_BLOCK)].cpu().numpy()
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), t
            for x in m_b:
                assert not x[zero].any()

            if with_oracle:
                g_o = [_host_bits(g, grad) for g in grads]
                out = oracle.step(d=d, W=W, layout=None, beta1=wl.beta1, beta2=wl.beta2, lr=wl.lr, wd=wl.wd,
                                  mode=0, nbits=1, flags=0, sync_interval=0, t=t, grads=g_o, theta=theta_o,
                                  m=m_o)
                wire_h = wire.cpu().numpy().view(np.uint32)
                for i in range(W):
                    assert np.array_equal(wire_h[i], out.wire[i]), (t, i, int((wire_h[i] != out.wire[i]).sum()))
                assert np.array_equal(theta_b.cpu().numpy().view(np.uint32), theta_o.view(np.uint32)), t
                for i in range(W):
                    assert np.array_equal(m_b[i].cpu().numpy().view(np.uint32), m_o[i].view(np.uint32)), (t, i)
    finally:
        lc.lioncub_destroy(h)


def test_noalloc_setup_call(lc):
    """A d == 0 call with valid pointers does the per-device set-up, launches
    nothing and succeeds; a later call then runs as usual."""
    dev = torch.device("cuda", 0)
    buf = torch.zeros(64, dtype=torch.float32, device=dev)
    before = buf.clone()
    lc.lioncub_sign_step_noalloc(0, 4, 0.9, 0.99, 1e-4, 0.1, 0, lc.GRAD_F32, [buf.data_ptr()] * 4,
                                 buf.data_ptr(), [buf.data_ptr()] * 4)
    torch.cuda.synchronize()
    assert torch.equal(buf, before)
    assert lc.lioncub_last_error(None) == ""


def test_noalloc_rejects_oversize(lc):
    dev = torch.device("cuda", 0)
    buf = torch.zeros(64, dtype=torch.float32, device=dev)
    too_big = 16_777_216 + 1  # W = 8: 8 * 524,292 words > 4,194,304
    with pytest.raises(lc.LionCubError) as e:
        lc.lioncub_sign_step_noalloc(too_big, 8, 0.9, 0.99, 1e-4, 0.1, 0, lc.GRAD_BF16, [buf.data_ptr()] * 8,
                                     buf.data_ptr(), [buf.data_ptr()] * 8)
    assert e.value.code == lc.ERR_ARG
    assert "LIONCUB_NOALLOC_MAX_WORDS" in str(e.value)
    # a later successful call clears the message
    lc.lioncub_sign_step_noalloc(0, 8, 0.9, 0.99, 1e-4, 0.1, 0, lc.GRAD_BF16, [buf.data_ptr()] * 8,
                                 buf.data_ptr(), [buf.data_ptr()] * 8)
    assert lc.lioncub_last_error(None) == ""


def test_noalloc_under_bounds_checks():
    """The same cases on the bounds-checked build: its kernels record any
    out-of-range index in a static status word, which each call reads back
    first, so the final set-up call fails if any earlier kernel set it."""
    if os.environ.get("LIONCUB_LIBRARY"):
        pytest.skip("already running on another build of the library")
    from communication_compressed_sign_gb300 import build
    import __graft_entry__
    __graft_entry__.build()
    lib = build.build(bounds_check=True)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.abspath(__file__), "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider", "-k", "not under_bounds_checks"],
                       cwd=ROOT, env={**os.environ, "LIONCUB_LIBRARY": lib}, capture_output=True, text=True,
                       timeout=900)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
