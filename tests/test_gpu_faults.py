"""Fault handling of the C ABI on the GPU, with every fault made on the host.

Allocation and launch failures come from the library's fault-injection
environment variables (LIONCUB_FAIL_ALLOC / LIONCUB_FAIL_LAUNCH): the failing
call is never made, an error code is returned in its place.  A corrupted
guard band is planted by a host-issued memset at creation
(LIONCUB_POISON_GUARD).  The one device wait (the staged reduce's bounded
wait for its bulk copies) is made to give up early by LIONCUB_WAIT_POLLS,
which replaces it with a few non-blocking polls; the block still drains its
copies with the normal bounded wait before it leaves.  Nothing here faults,
traps or hangs the device.

Checked: every allocation of lioncub_create can fail cleanly (ERR_OOM, no
leak, the library still usable); a failed staging allocation of the
host-buffer step leaves the handle usable and a retry computes the same
result; a launch that fails before the compress kernel leaves theta and m
untouched, so a retry is bit-exact with a run that never failed; a failure
of the last launch keeps the step counter and theta; the guard-band check
reports a planted overrun through the status word; a wait that runs out is
reported through the status word and leaves the device usable.
"""
import pytest

import synth
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    yield
    torch.cuda.empty_cache()


from communication_compressed_sign_gb300 import lioncub as lc  # noqa: E402

# device allocations lioncub_create makes: wire, tile table, tile ranges,
# tensor sizes, status word; L1 mode adds M1 partials, M1 and 1/M1
CREATE_ALLOCS = {0: 5, 1: 8}


def _wl(d, W, mode, nbits, grad="bf16"):
    dist = ("t", 3.0, 1e-3, 0.0, 1.0) if grad == "bf16" else ("normal", 1e-3)
    return synth.Workload(0, "faults", W, synth.flat_layout(d), grad, dist, mode, nbits, 4)


def _create(wl):
    return lc.lioncub_create(wl.d, wl.W, None, wl.beta1, wl.beta2, wl.lr, wl.wd, wl.mode, wl.nbits,
                             lc.GRAD_F32 if wl.grad == "f32" else lc.GRAD_BF16, wl.sync_interval)


class _State:
    """theta, W momenta and W gradient buffers on the device for workload wl."""

    def __init__(self, wl):
        dev = torch.device("cuda", 0)
        self.wl = wl
        self.theta = torch.empty(wl.d, dtype=torch.float32, device=dev)
        synth.fill_theta_(self.theta, wl)
        self.m = [torch.zeros(wl.d, dtype=torch.float32, device=dev) for _ in range(wl.W)]
        self.g = [torch.empty(wl.d, dtype=synth.grad_dtype(wl), device=dev) for _ in range(wl.W)]

    def fill(self, t):
        for i, x in enumerate(self.g):
            synth.fill_grad_(x, self.wl, t, i)

    def bind(self, h):
        lc.lioncub_bind_state(h, self.theta.data_ptr(), [x.data_ptr() for x in self.m])

    def step(self, h):
        lc.lioncub_step(h, [x.data_ptr() for x in self.g], torch.cuda.current_stream().cuda_stream)

    def snapshot(self):
        torch.cuda.synchronize()
        return self.theta.clone(), [x.clone() for x in self.m]


def _equal_bits(a, b):
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def _status(h):
    out = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    lc.lioncub_debug_export(h, lc.EXPORT_STATUS, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return int(out.item())


def _clean_run(wl, steps):
    st = _State(wl)
    h = _create(wl)
    try:
        st.bind(h)
        for t in range(steps):
            st.fill(t)
            st.step(h)
        assert _status(h) == 0
    finally:
        lc.lioncub_destroy(h)
    return st.snapshot()


# ---------------------------------------------------------------------------
# allocation failures
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode,nbits", [(0, 1), (1, 4)])
def test_every_create_allocation_can_fail_cleanly(monkeypatch, mode, nbits):
    """The k-th allocation of lioncub_create fails for every k: ERR_OOM, the
    message names the set-up, and repeating it leaks no device memory."""
    wl = _wl(1 << 22, 8, mode, nbits)  # wire 4 MB (sign) / 16 MB (n = 4)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for k in range(1, CREATE_ALLOCS[mode] + 1):
        monkeypatch.setenv("LIONCUB_FAIL_ALLOC", str(k))
        for _ in range(16):
            with pytest.raises(lc.LionCubError) as e:
                _create(wl)
            assert e.value.code == lc.ERR_OOM, k
            assert "device set-up failed" in str(e.value)
    # one past the last allocation: creation succeeds
    monkeypatch.setenv("LIONCUB_FAIL_ALLOC", str(CREATE_ALLOCS[mode] + 1))
    lc.lioncub_destroy(_create(wl))
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free0 - free1 < (8 << 20), f"{(free0 - free1) >> 20} MiB not returned"
    # and the library computes correctly afterwards
    monkeypatch.delenv("LIONCUB_FAIL_ALLOC")
    parity.run_parity(_wl(6000, 3, mode, nbits), parity.tensor_pieces(synth.flat_layout(6000), {"flat"}), 3)


@pytest.mark.parametrize("extra", [1, 2])
def test_staging_allocation_failure(monkeypatch, extra):
    """extra = 1: the first staging buffer of lioncub_step_host cannot be
    allocated -> ERR_OOM, the step counter stays, and the next call (which
    allocates again) succeeds.  extra = 2: only the second buffer fails, so
    uploads run single-buffered.  Either way the results equal device steps."""
    wl = _wl(70000, 4, 0, 1)
    steps = 4
    ref_theta, ref_m = _clean_run(wl, steps)

    monkeypatch.setenv("LIONCUB_FAIL_ALLOC", str(CREATE_ALLOCS[0] + extra))
    st = _State(wl)
    h = _create(wl)
    monkeypatch.delenv("LIONCUB_FAIL_ALLOC")
    try:
        st.bind(h)
        host_g = [torch.empty(wl.d, dtype=synth.grad_dtype(wl)).pin_memory() for _ in range(wl.W)]
        theta_out = torch.empty(wl.d, dtype=torch.float32).pin_memory()
        stream = torch.cuda.current_stream().cuda_stream
        for t in range(steps):
            st.fill(t)
            for i in range(wl.W):
                host_g[i].copy_(st.g[i])
            ptrs = [x.data_ptr() for x in host_g]
            if t == 0 and extra == 1:
                with pytest.raises(lc.LionCubError) as e:
                    lc.lioncub_step_host(h, ptrs, theta_out.data_ptr(), stream)
                assert e.value.code == lc.ERR_OOM
                assert lc.lioncub_get_step(h) == 0
            lc.lioncub_step_host(h, ptrs, theta_out.data_ptr(), stream)
            torch.cuda.synchronize()
        assert lc.lioncub_get_step(h) == steps
        assert _status(h) == 0
    finally:
        lc.lioncub_destroy(h)
    theta, m = st.snapshot()
    assert _equal_bits(theta, ref_theta)
    assert _equal_bits(theta_out, ref_theta.cpu())
    for x, y in zip(m, ref_m):
        assert _equal_bits(x, y)


# ---------------------------------------------------------------------------
# launch failures
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode,nbits,k,kernel", [
    (0, 1, 1, "compress"),
    (1, 4, 1, "m1_partial"), (1, 4, 2, "m1_finalize"), (1, 4, 3, "compress"),
])
def test_launch_failure_before_state_changes(monkeypatch, mode, nbits, k, kernel):
    """A launch that fails at or before the compress kernel changes neither
    theta nor m: the step reports ERR_CUDA naming the kernel, the counter
    stays, and retrying continues exactly as if nothing had failed."""
    wl = _wl(9000, 5, mode, nbits)
    steps = 3
    ref_theta, ref_m = _clean_run(wl, steps)

    monkeypatch.setenv("LIONCUB_FAIL_LAUNCH", str(k))
    st = _State(wl)
    h = _create(wl)
    monkeypatch.delenv("LIONCUB_FAIL_LAUNCH")
    try:
        st.bind(h)
        before = st.snapshot()
        st.fill(0)
        with pytest.raises(lc.LionCubError) as e:
            st.step(h)
        assert e.value.code == lc.ERR_CUDA
        assert f"{kernel} launch" in str(e.value)
        assert lc.lioncub_get_step(h) == 0
        after = st.snapshot()
        assert _equal_bits(after[0], before[0])
        for x, y in zip(after[1], before[1]):
            assert _equal_bits(x, y)
        for t in range(steps):
            st.fill(t)
            st.step(h)
        assert lc.lioncub_get_step(h) == steps
        assert _status(h) == 0
    finally:
        lc.lioncub_destroy(h)
    theta, m = st.snapshot()
    assert _equal_bits(theta, ref_theta)
    for x, y in zip(m, ref_m):
        assert _equal_bits(x, y)


@pytest.mark.parametrize("mode,nbits,k", [(0, 1, 2), (1, 2, 4)])
def test_launch_failure_of_the_apply(monkeypatch, mode, nbits, k):
    """The reduce/apply launch fails: ERR_CUDA, the counter stays and theta is
    untouched (m has moved, as the header states); the handle keeps working."""
    wl = _wl(9000, 4, mode, nbits)
    monkeypatch.setenv("LIONCUB_FAIL_LAUNCH", str(k))
    st = _State(wl)
    h = _create(wl)
    monkeypatch.delenv("LIONCUB_FAIL_LAUNCH")
    try:
        st.bind(h)
        theta0 = st.snapshot()[0]
        st.fill(0)
        with pytest.raises(lc.LionCubError) as e:
            st.step(h)
        assert e.value.code == lc.ERR_CUDA and "reduce_apply launch" in str(e.value)
        assert lc.lioncub_get_step(h) == 0
        assert _equal_bits(st.snapshot()[0], theta0)
        st.step(h)
        assert lc.lioncub_get_step(h) == 1
        assert _status(h) == 0
        assert not _equal_bits(st.snapshot()[0], theta0)
    finally:
        lc.lioncub_destroy(h)


# ---------------------------------------------------------------------------
# guard bands around the library's scratch
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode,nbits", [(0, 1), (1, 8)])
def test_guard_check_reports_a_planted_overrun(monkeypatch, mode, nbits):
    """With one guard byte overwritten at creation, the status export reports
    LIONCUB_STATUS_GUARD (and nothing else); the same steps on an unpoisoned
    handle report 0."""
    wl = _wl(5000, 3, mode, nbits)
    for poison in (False, True):
        if poison:
            monkeypatch.setenv("LIONCUB_POISON_GUARD", "1")
        st = _State(wl)
        h = _create(wl)
        monkeypatch.delenv("LIONCUB_POISON_GUARD", raising=False)
        try:
            st.bind(h)
            for t in range(2):
                st.fill(t)
                st.step(h)
            assert _status(h) == (lc.STATUS_GUARD if poison else 0)
        finally:
            lc.lioncub_destroy(h)


# ---------------------------------------------------------------------------
# the bounded device wait
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode,nbits", [(0, 1), (1, 4)])
def test_wait_timeout_is_reported(monkeypatch, mode, nbits):
    """The staged reduce's wait for its bulk copies is made to run out
    (LIONCUB_WAIT_POLLS=1: one non-blocking poll right after the copies are
    issued, long before they can land): the step still returns and the device
    stays usable, the blocks that gave up drain their copies and leave, and
    the status word reports LIONCUB_STATUS_WAIT_TIMEOUT.  A handle created
    without the hook then matches the oracle."""
    wl = _wl(1 << 20, 8, mode, nbits)  # 256 staged blocks
    monkeypatch.setenv("LIONCUB_WAIT_POLLS", "1")
    st = _State(wl)
    h = _create(wl)
    monkeypatch.delenv("LIONCUB_WAIT_POLLS")
    try:
        st.bind(h)
        theta0, m0 = st.snapshot()
        st.fill(0)
        st.step(h)  # returns; the kernel's blocks give up and drain
        assert lc.lioncub_get_step(h) == 1
        theta1, m1 = st.snapshot()
        status = _status(h)
        assert status & lc.STATUS_WAIT_TIMEOUT, status
        assert status & ~lc.STATUS_WAIT_TIMEOUT == 0, status
        assert not _equal_bits(m1[0], m0[0])  # the compress pass ran before the reduce gave up
        # theta is invalid for this step: blocks that gave up left their part unchanged
        assert int((theta1.view(torch.int32) == theta0.view(torch.int32)).sum()) > 0
    finally:
        lc.lioncub_destroy(h)
    torch.cuda.synchronize()
    parity.run_parity(_wl(70_001, 8, mode, nbits), parity.tensor_pieces(synth.flat_layout(70_001), {"flat"}), 2)
