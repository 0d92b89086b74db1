"""The allocation-free sign-mode entry point against the handle-based one.

lioncub_sign_step_noalloc exists for callers that cannot allocate device
memory when they run a step (an allocator that owns all device memory, code
that must avoid the synchronization cudaMalloc can cause, plug-ins that only
allocate at initialisation).  It keeps its packed sign words in a fixed 16 MiB
array of the library's static device memory.  Here it must produce exactly
the theta and momenta of lioncub_step (sign mode is bit-exact) on two calls
in a row, reusing the shared array, and refuse sizes beyond the array.

The file is named to be collected last, so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lc():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from communication_compressed_sign_gb300 import lioncub
    lioncub.load()
    return lioncub


def _state(d, W, seed):
    dev = torch.device("cuda", 0)
    wl = synth.Workload(0, "noalloc", W, synth.flat_layout(d), "bf16", ("t", 3.0, 1e-3, 0.0, 1.0), 0, 1, 2,
                        seed=seed)
    theta = torch.empty(d, dtype=torch.float32, device=dev)
    synth.fill_theta_(theta, wl)
    m = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
    return wl, theta, m


@pytest.mark.parametrize("d,W,grad", [(1_000_003, 8, "bf16"), (16_777_216, 8, "bf16"), (70_001, 5, "f32"),
                                      (33, 1, "bf16")])
def test_noalloc_matches_handle_path(lc, d, W, grad):
    dev = torch.device("cuda", 0)
    wl, theta_a, m_a = _state(d, W, seed=d % 1000)
    wl.grad = grad
    if grad == "f32":
        wl.dist = ("normal", 1e-3)
    theta_b = theta_a.clone()
    m_b = [x.clone() for x in m_a]
    gdt = synth.grad_dtype(wl)
    gcode = lc.GRAD_F32 if grad == "f32" else lc.GRAD_BF16
    grads = [torch.empty(d, dtype=gdt, device=dev) for _ in range(W)]
    stream = torch.cuda.current_stream().cuda_stream

    h = lc.lioncub_create(d, W, None, wl.beta1, wl.beta2, wl.lr, wl.wd, lc.MODE_SIGN_MAJORITY, 1, gcode, 0)
    try:
        lc.lioncub_bind_state(h, theta_a.data_ptr(), [x.data_ptr() for x in m_a])
        for t in range(2):  # two calls in a row share the static array
            for i in range(W):
                synth.fill_grad_(grads[i], wl, t, i)
                if t == 1:
                    grads[i][::7] = 0  # exact zeros exercise the step-parity bit
            gp = [g.data_ptr() for g in grads]
            lc.lioncub_step(h, gp, stream)
            lc.lioncub_sign_step_noalloc(d, W, wl.beta1, wl.beta2, wl.lr, wl.wd, t, gcode, gp,
                                         theta_b.data_ptr(), [x.data_ptr() for x in m_b], stream)
            torch.cuda.synchronize()
            assert torch.equal(theta_a.view(torch.int32), theta_b.view(torch.int32)), t
            for x, y in zip(m_a, m_b):
                assert torch.equal(x.view(torch.int32), y.view(torch.int32)), t
    finally:
        lc.lioncub_destroy(h)


def test_noalloc_rejects_oversize(lc):
    dev = torch.device("cuda", 0)
    buf = torch.zeros(64, dtype=torch.float32, device=dev)
    too_big = 16_777_216 + 1  # W = 8: 8 * 524,292 words > 4,194,304
    with pytest.raises(lc.LionCubError) as e:
        lc.lioncub_sign_step_noalloc(too_big, 8, 0.9, 0.99, 1e-4, 0.1, 0, lc.GRAD_BF16, [buf.data_ptr()] * 8,
                                     buf.data_ptr(), [buf.data_ptr()] * 8)
    assert e.value.code == lc.ERR_ARG
    assert "LIONCUB_NOALLOC_MAX_WORDS" in str(e.value)
