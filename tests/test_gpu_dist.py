"""The data-parallel exchange's kernels on one GPU, against the single-GPU step.

N ranks are emulated in one process on one GPU: N handles from
``lioncub_dist_create`` (rank r holding workers r*W/N .. (r+1)*W/N - 1, its
own theta and its workers' momenta) and N sets of exchange buffers.  The
collectives between the three launches of a step are done by plain device
copies in the test (the all-to-all moves segment r of every rank's send
buffer to rank r; the allgathers concatenate in rank order; the allreduce
adds the int8/int32 code sums).  Every launch is enqueued on one stream, one
after the other: no kernel waits for another rank's.

After every step each emulated rank's theta, and the momenta of its workers,
must equal those of ``lioncub_step`` over all W workers on one GPU, bit for
bit -- in sign mode (majority, tie alternation, the D-Lion average), in L1
mode with 2-, 4- and 8-bit codes, with and without momentum sync -- which
the single-GPU parity tests tie to the oracle.  Two more tests run
``DistLionCub`` itself: through a real NCCL process group of one rank, and at
N = 2 and 4 as processes sharing this GPU through a gloo group.
"""
import os
import socket

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


SMALL = [("emb", 0, 4096, synth.SYNC_M), ("w", 4096, 4992, 0), ("x", 9088, 32, 0), ("head", 9120, 2048, synth.SYNC_M),
         ("b", 11168, 45, 0)]


def _bits(x):
    return x.view(torch.int32)


def _run(lc, wl, N, steps, zero_every=11):
    """wl's steps on one handle and on N emulated ranks; compares after each step."""
    from communication_compressed_sign_gb300 import dist as cdist

    dev = torch.device("cuda", 0)
    d, W = wl.d, wl.W
    lay = synth.abi_layout(wl.layout)
    gcode = lc.GRAD_F32 if wl.grad == "f32" else lc.GRAD_BF16
    mode = wl.mode | wl.flags
    s = torch.cuda.current_stream()
    sp = s.cuda_stream

    theta0 = torch.empty(d, dtype=torch.float32, device=dev)
    synth.fill_theta_(theta0, wl)
    grads = [torch.empty(d, dtype=synth.grad_dtype(wl), device=dev) for _ in range(W)]

    theta_ref = theta0.clone()
    m_ref = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
    h_ref = lc.lioncub_create(d, W, lay, wl.beta1, wl.beta2, wl.lr, wl.wd, mode, wl.nbits, gcode, wl.sync_interval)
    hs = []
    try:
        lc.lioncub_bind_state(h_ref, theta_ref.data_ptr(), [x.data_ptr() for x in m_ref])
        plans, bufs, thetas, ms = [], [], [], []
        for r in range(N):
            plan = lc.lioncub_dist_plan_make(d, W, N, r, lay, mode, wl.nbits, wl.sync_interval)
            h = lc.lioncub_dist_create(d, W, N, r, lay, wl.beta1, wl.beta2, wl.lr, wl.wd, mode, wl.nbits, gcode,
                                       wl.sync_interval)
            hs.append(h)
            b = cdist.allocate_buffers(plan, dev)
            lc.lioncub_dist_bind_buffers(h, [x.data_ptr() if x is not None else 0 for x in b])
            th = theta0.clone()
            mm = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(plan.local_workers)]
            lc.lioncub_bind_state(h, th.data_ptr(), [x.data_ptr() for x in mm])
            plans.append(plan), bufs.append(b), thetas.append(th), ms.append(mm)
        Wl = plans[0].local_workers
        sign = wl.mode == 0

        for t in range(steps):
            for j in range(W):
                synth.fill_grad_(grads[j], wl, t, j)
                if zero_every:
                    grads[j][::zero_every] = 0
                    grads[j][64:96] = 0
            lc.lioncub_step(h_ref, [g.data_ptr() for g in grads], sp)
            sync = cdist.is_sync_step(t, wl.sync_interval, plans[0])
            for r in range(N):
                lc.lioncub_dist_compress(hs[r], [g.data_ptr() for g in grads[r * Wl:(r + 1) * Wl]], sp)
            if sign:  # all-to-all: segment r of every send buffer to rank r
                for r in range(N):
                    recv = bufs[r][lc.DIST_RECV].view(N, -1)
                    for src in range(N):
                        recv[src].copy_(bufs[src][lc.DIST_SEND].view(N, -1)[r])
            if sync:
                gathered = torch.cat([bufs[q][lc.DIST_SYNC_SEND] for q in range(N)])
                for r in range(N):
                    bufs[r][lc.DIST_SYNC_RECV].copy_(gathered)
            for r in range(N):
                lc.lioncub_dist_reduce(hs[r], sp)
            if sign:
                gathered = torch.cat([bufs[q][lc.DIST_DIR_CHUNK] for q in range(N)])
                for r in range(N):
                    bufs[r][lc.DIST_DIR_ALL].copy_(gathered)
            else:
                total = sum(bufs[q][lc.DIST_AGG].to(torch.int32) for q in range(N))
                for r in range(N):
                    bufs[r][lc.DIST_AGG].copy_(total.to(bufs[r][lc.DIST_AGG].dtype))
            for r in range(N):
                lc.lioncub_dist_apply(hs[r], sp)
            torch.cuda.synchronize()
            for r in range(N):
                assert torch.equal(_bits(thetas[r]), _bits(theta_ref)), \
                    (wl.name, N, t, r, int((thetas[r] != theta_ref).sum()))
                for i in range(Wl):
                    assert torch.equal(_bits(ms[r][i]), _bits(m_ref[r * Wl + i])), (wl.name, N, t, r, i)
                assert lc.lioncub_get_step(hs[r]) == t + 1
        status = torch.full((1,), -1, dtype=torch.int32, device=dev)
        for h in hs + [h_ref]:
            lc.lioncub_debug_export(h, lc.EXPORT_STATUS, status.data_ptr(), sp)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
    finally:
        for h in hs:
            lc.lioncub_destroy(h)
        lc.lioncub_destroy(h_ref)


def _small(name, W, mode, nbits, flags=0, sync=0, grad="f32", layout=None, d=None):
    dist = ("normal", 1e-3) if grad == "f32" else ("t", 3.0, 1e-3, 0.0, 1.0)
    lay = layout if layout is not None else (SMALL if d is None else synth.flat_layout(d))
    return synth.Workload(0, name, W, lay, grad, dist, mode, nbits, 4, sync_interval=sync, flags=flags)


@pytest.mark.parametrize("N", [2, 4])
@pytest.mark.parametrize("case", [
    ("sign", 4, 0, 1, 0, 1, "f32"),
    ("sign_bf16_sync2", 8, 0, 1, 0, 2, "bf16"),
    ("tie_alternate", 4, 0, 1, 0x100, 0, "f32"),
    ("average_sync1", 8, 0, 1, 0x200, 1, "bf16"),
    ("l1n2_sync1", 4, 1, 2, 0, 1, "f32"),
    ("l1n4", 8, 1, 4, 0, 0, "bf16"),
    ("l1n8_int32_sums", 4, 1, 8, 0, 3, "f32"),
])
def test_emulated_ranks_small(lc, case, N):
    name, W, mode, nbits, flags, sync, grad = case
    _run(lc, _small(name, W, mode, nbits, flags, sync, grad), N, 4)


@pytest.mark.parametrize("d,W,N", [(1_000_003, 8, 8), (33, 4, 4), (4096 * 3 + 1, 6, 3)])
def test_emulated_ranks_flat(lc, d, W, N):
    _run(lc, _small(f"flat{d}", W, 0, 1, d=d, grad="bf16"), N, 3)


@pytest.mark.parametrize("key,N", [(7, 2), (7, 8), (6, 4), (2, 8), (3, 2)])
def test_emulated_ranks_workloads(lc, key, N):
    """The pages' layouts: DeiT-Tiny (4-bit codes, embedding and head momenta
    synchronized), ViT-B/16 (D-Lion average), GPT-2 small (signs) and GPT-2
    medium (4-bit codes, 0.1 % outliers), W = 8 workers split over N ranks."""
    wl = synth.workloads()[key]
    _run(lc, wl, N, 3, zero_every=0)


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


@pytest.mark.parametrize("mode,nbits,sync", [(0, 1, 1), (1, 4, 1)])
def test_nccl_single_rank_group(lc, mode, nbits, sync):
    """DistLionCub through torch.distributed with NCCL (one rank, this GPU):
    the real collective calls on the step's stream; results equal lioncub_step."""
    import torch.distributed as dist
    from communication_compressed_sign_gb300.dist import DistLionCub

    if dist.is_initialized():
        pytest.skip("a process group already exists in this process")
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dev = torch.device("cuda", 0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1,
                            device_id=dev)
    try:
        wl = _small("nccl", 4, mode, nbits, sync=sync, grad="bf16")
        d, W = wl.d, wl.W
        lay = synth.abi_layout(wl.layout)
        theta0 = torch.empty(d, dtype=torch.float32, device=dev)
        synth.fill_theta_(theta0, wl)
        opt = DistLionCub(d, W, lay, beta1=wl.beta1, beta2=wl.beta2, lr=wl.lr, wd=wl.wd, mode=mode, nbits=nbits,
                          grad_dtype=lc.GRAD_BF16, sync_interval=sync, device=dev)
        theta = theta0.clone()
        m = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
        opt.bind(theta, m)
        theta_ref = theta0.clone()
        m_ref = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
        h = lc.lioncub_create(d, W, lay, wl.beta1, wl.beta2, wl.lr, wl.wd, mode, nbits, lc.GRAD_BF16, sync)
        grads = [torch.empty(d, dtype=torch.bfloat16, device=dev) for _ in range(W)]
        try:
            lc.lioncub_bind_state(h, theta_ref.data_ptr(), [x.data_ptr() for x in m_ref])
            for t in range(4):
                for j in range(W):
                    synth.fill_grad_(grads[j], wl, t, j)
                opt.step(grads)
                lc.lioncub_step(h, [g.data_ptr() for g in grads], torch.cuda.current_stream().cuda_stream)
                torch.cuda.synchronize()
                assert torch.equal(_bits(theta), _bits(theta_ref)), t
                for x, y in zip(m, m_ref):
                    assert torch.equal(_bits(x), _bits(y)), t
            assert opt.t == 4
        finally:
            lc.lioncub_destroy(h)
            opt.close()
    finally:
        dist.destroy_process_group()


def test_exchange_call_order_and_handles(lc):
    """The three exchange calls run in order only (ERR_STATE otherwise, the
    step counter unchanged), need their buffers bound, and a data-parallel
    handle refuses the single-GPU step, host step and diagnostics."""
    from communication_compressed_sign_gb300 import dist as cdist

    dev = torch.device("cuda", 0)
    d, W, N = 10_000, 4, 2
    h = lc.lioncub_dist_create(d, W, N, 1, None, 0.9, 0.99, 1e-4, 0.1, 0, 1, lc.GRAD_BF16, 0)
    try:
        theta = torch.zeros(d, dtype=torch.float32, device=dev)
        m = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W // N)]
        g = [torch.zeros(d, dtype=torch.bfloat16, device=dev) for _ in range(W // N)]
        lc.lioncub_bind_state(h, theta.data_ptr(), [x.data_ptr() for x in m])
        with pytest.raises(lc.LionCubError) as e:  # buffers not bound yet
            lc.lioncub_dist_compress(h, [x.data_ptr() for x in g])
        assert e.value.code == lc.ERR_STATE
        plan = lc.lioncub_dist_plan_make(d, W, N, 1, None, 0, 1, 0)
        bufs = cdist.allocate_buffers(plan, dev)
        ptrs = [b.data_ptr() if b is not None else 0 for b in bufs]
        missing = list(ptrs)
        missing[lc.DIST_RECV] = 0
        with pytest.raises(lc.LionCubError) as e:
            lc.lioncub_dist_bind_buffers(h, missing)
        assert e.value.code == lc.ERR_ARG
        misaligned = list(ptrs)
        misaligned[lc.DIST_SEND] += 4
        with pytest.raises(lc.LionCubError) as e:
            lc.lioncub_dist_bind_buffers(h, misaligned)
        assert e.value.code == lc.ERR_ALIGN
        lc.lioncub_dist_bind_buffers(h, ptrs)
        for call in (lambda: lc.lioncub_dist_reduce(h), lambda: lc.lioncub_dist_apply(h)):
            with pytest.raises(lc.LionCubError) as e:
                call()
            assert e.value.code == lc.ERR_STATE and "out of order" in str(e.value)
        lc.lioncub_dist_compress(h, [x.data_ptr() for x in g])
        with pytest.raises(lc.LionCubError) as e:
            lc.lioncub_dist_compress(h, [x.data_ptr() for x in g])
        assert e.value.code == lc.ERR_STATE
        lc.lioncub_dist_reduce(h)
        assert lc.lioncub_get_step(h) == 0
        lc.lioncub_dist_apply(h)
        assert lc.lioncub_get_step(h) == 1
        torch.cuda.synchronize()
        host = torch.zeros(d, dtype=torch.float32)
        for call in (lambda: lc.lioncub_step(h, [x.data_ptr() for x in g]),
                     lambda: lc.lioncub_step_host(h, [x.data_ptr() for x in g], host.data_ptr()),
                     lambda: lc.lioncub_diagnose(h, [x.data_ptr() for x in g], theta.data_ptr()),
                     lambda: lc.lioncub_diagnose_qinf(h, [x.data_ptr() for x in g], 4, 0, theta.data_ptr())):
            with pytest.raises(lc.LionCubError) as e:
                call()
            assert e.value.code == lc.ERR_STATE
    finally:
        lc.lioncub_destroy(h)
    # and a single-GPU handle refuses the exchange calls
    h = lc.lioncub_create(d, W, None, 0.9, 0.99, 1e-4, 0.1, 0, 1, lc.GRAD_BF16, 0)
    try:
        with pytest.raises(lc.LionCubError) as e:
            lc.lioncub_dist_bind_buffers(h, [0] * lc.DIST_BUFFERS)
        assert e.value.code == lc.ERR_STATE
    finally:
        lc.lioncub_destroy(h)


def _gloo_rank(rank, nranks, port, case, q):
    try:
        import synth as sy
        import torch.distributed as dist
        from communication_compressed_sign_gb300 import lioncub
        from communication_compressed_sign_gb300.dist import DistLionCub
        lioncub.load()
        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=nranks)
        name, W, mode, nbits, flags, sync, grad = case
        dist_ = ("normal", 1e-3) if grad == "f32" else ("t", 3.0, 1e-3, 0.0, 1.0)
        wl = sy.Workload(0, name, W, SMALL, grad, dist_, mode, nbits, 4, sync_interval=sync, flags=flags)
        d, lay = wl.d, sy.abi_layout(wl.layout)
        gcode = lioncub.GRAD_F32 if grad == "f32" else lioncub.GRAD_BF16
        theta0 = torch.empty(d, dtype=torch.float32, device=dev)
        sy.fill_theta_(theta0, wl)
        opt = DistLionCub(d, W, lay, beta1=wl.beta1, beta2=wl.beta2, lr=wl.lr, wd=wl.wd, mode=mode | flags,
                          nbits=nbits, grad_dtype=gcode, sync_interval=sync, device=dev)
        Wl, first = opt.plan.local_workers, opt.plan.first_worker
        theta = theta0.clone()
        m = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(Wl)]
        opt.bind(theta, m)
        theta_ref = theta0.clone()
        m_ref = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
        h = lioncub.lioncub_create(d, W, lay, wl.beta1, wl.beta2, wl.lr, wl.wd, mode | flags, nbits, gcode, sync)
        grads = [torch.empty(d, dtype=sy.grad_dtype(wl), device=dev) for _ in range(W)]
        try:
            lioncub.lioncub_bind_state(h, theta_ref.data_ptr(), [x.data_ptr() for x in m_ref])
            for t in range(4):
                for j in range(W):
                    sy.fill_grad_(grads[j], wl, t, j)
                    grads[j][::11] = 0
                opt.step(grads[first:first + Wl])
                lioncub.lioncub_step(h, [g.data_ptr() for g in grads], torch.cuda.current_stream().cuda_stream)
                torch.cuda.synchronize()
                assert torch.equal(_bits(theta), _bits(theta_ref)), (name, rank, t)
                for i in range(Wl):
                    assert torch.equal(_bits(m[i]), _bits(m_ref[first + i])), (name, rank, t, i)
        finally:
            lioncub.lioncub_destroy(h)
            opt.close()
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except BaseException:
        import traceback
        q.put((rank, traceback.format_exc()))


@pytest.mark.parametrize("case,nranks", [(("sign_sync1", 4, 0, 1, 0, 1, "bf16"), 2),
                                         (("l1n4_sync2", 4, 1, 4, 0, 2, "f32"), 2),
                                         (("average", 4, 0, 1, 0x200, 0, "bf16"), 2),
                                         (("sign_w8_sync1", 8, 0, 1, 0, 1, "bf16"), 4),
                                         (("l1n2", 8, 1, 2, 0, 0, "bf16"), 4)])
def test_processes_through_torch_distributed(lc, case, nranks):
    """DistLionCub with 2 or 4 ranks as processes that share this GPU, the
    collectives through a gloo group (which moves CUDA tensors through the
    host, so no kernel ever waits for another process): the product's own
    collective calls between the library's launches equal lioncub_step over
    all W workers bit for bit."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gloo_rank, args=(r, nranks, port, case, q)) for r in range(nranks)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in range(nranks))
    for p in procs:
        p.join(timeout=60)
    bad = {r: m for r, m in res.items() if m != "ok"}
    assert not bad, "\n".join(f"rank {r}:\n{m}" for r, m in bad.items())
