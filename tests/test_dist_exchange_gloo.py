"""The data-parallel exchange on gloo process groups of 2 and 4 ranks (CPU).

Each rank holds W/N workers and a copy of theta.  Its part of the step is
computed with the oracle's functions, laid out in the exchange buffers
exactly where the library's plan puts it (``lioncub_dist_plan_make``, a host
function of the CUDA library: chunk ownership, row layout, direction fields,
code-sum width, sync slots), and moved with the same collective calls the
GPU path issues (``dist.exchange_after_compress`` / ``exchange_after_reduce``)
over gloo:

  sign mode   the rank's packed words, chunk-major -> all-to-all -> the
              chunk owner's vote of every worker's words -> 2-bit directions
              (or the vote sums, for the average) -> allgather -> theta;
  L1 mode     the code sum of the rank's workers -> allreduce -> theta;
  sync steps  the new momenta of flagged tensors -> allgather -> the average
              in worker order on every rank.

After several steps every rank's theta and its workers' momenta must equal a
single-process oracle run of all W workers bit for bit, and the words each
chunk owner received must be every worker's words for its chunk.  This is
the bookkeeping of the multi-GPU path ("Lion Cub" page, quoted body text on
the implementation: AlltoAll for 1-bit, AllReduce for wider codes); the same
collectives run on the GPU with NCCL.
"""
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402

LAYOUT = [(0, 4096, 1), (4096, 5000 // 32 * 32, 0), (4096 + 4992, 32, 0), (4096 + 5024, 2048, 1),
          (4096 + 5024 + 2048, 45, 0)]
D_LAYOUT = 4096 + 5024 + 2048 + 45

CASES = {
    # name: (d, layout, W, nranks, mode, nbits, flags, sync_interval, grad)
    "sign_w4_n2_sync1": (D_LAYOUT, LAYOUT, 4, 2, 0, 1, 0, 1, "f32"),
    "sign_w4_n4_sync2_bf16": (D_LAYOUT, LAYOUT, 4, 4, 0, 1, 0, 2, "bf16"),
    "sign_w6_n2_tie_alternate": (D_LAYOUT, LAYOUT, 6, 2, 0, 1, 0x100, 0, "f32"),
    "sign_w4_n2_average": (D_LAYOUT, LAYOUT, 4, 2, 0, 1, 0x200, 1, "f32"),
    "sign_small_d_empty_chunks": (1000, None, 4, 4, 0, 1, 0, 0, "f32"),
    "l1n2_w4_n2_sync1": (D_LAYOUT, LAYOUT, 4, 2, 1, 2, 0, 1, "f32"),
    "l1n4_w4_n4_bf16": (D_LAYOUT, LAYOUT, 4, 4, 1, 4, 0, 0, "bf16"),
    "l1n8_w2_n2_int32_sums": (D_LAYOUT, LAYOUT, 2, 2, 1, 8, 0, 3, "f32"),
}
STEPS = 4
BETA1, BETA2, LR, WD = 0.9, 0.99, 1e-4, 0.1


def _grads(d, W, t, grad):
    """Worker gradients of step t: N(0, 1e-3^2) with exact zeros (every 11th
    element, and a whole 32-element block) so the alternating rule shows."""
    out = []
    for i in range(W):
        rng = np.random.default_rng(1000 * t + i)
        g = (rng.standard_normal(d) * 1e-3).astype(np.float32)
        g[::11] = 0.0
        g[64:96] = 0.0
        if grad == "bf16":
            bits = g.view(np.uint32)
            bits = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)  # round to nearest even
            out.append(bits)
        else:
            out.append(g)
    return out


def _unpack2(words, n):
    e = np.arange(n)
    f = (words[e // 16].astype(np.int64) >> (2 * (e % 16))) & 3
    return np.where(f >= 2, f - 4, f)


def _rank_main(rank, nranks, port, name, q):
    try:
        _run_rank(rank, nranks, port, name)
        q.put((rank, "ok"))
    except BaseException as exc:  # report to the parent
        import traceback
        q.put((rank, traceback.format_exc()))
        raise SystemExit(1) from exc


def _run_rank(rank, nranks, port, name):
    import torch.distributed as dist
    from communication_compressed_sign_gb300 import dist as cdist
    from communication_compressed_sign_gb300 import lioncub as lc

    d, layout, W, N, mode, nbits, flags, sync_interval, grad = CASES[name]
    assert N == nranks
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=nranks)
    try:
        plan = lc.lioncub_dist_plan_make(d, W, N, rank, layout, mode | flags, nbits, sync_interval)
        Wl = plan.local_workers
        first = plan.first_worker
        assert Wl == W // N and first == rank * Wl
        sign = mode == 0
        if sign:
            assert plan.chunk % 4096 == 0 and plan.chunk * N >= d and plan.chunk_words == plan.chunk // 32
            assert plan.bytes[lc.DIST_SEND] == N * Wl * plan.chunk_words * 4
            assert plan.bytes[lc.DIST_RECV] == W * plan.chunk_words * 4
            assert plan.dir_bits == (8 if flags & 0x200 else 2)
            assert plan.bytes[lc.DIST_DIR_ALL] == N * plan.bytes[lc.DIST_DIR_CHUNK]
        else:
            qmax = (1 << (nbits - 1)) - 1
            assert plan.agg_bytes == (1 if W * qmax <= 127 else 4)
            assert plan.bytes[lc.DIST_AGG] >= d * plan.agg_bytes
        flagged = [(o, n) for (o, n, f) in (layout or []) if f & 1] if sync_interval > 0 else []
        slots = sum((n + 2047) // 2048 * 2048 for (_, n) in flagged)
        assert plan.sync_slots == slots
        assert plan.bytes[lc.DIST_SYNC_RECV] == W * slots * 4

        lay = [(o, n, f) for (o, n, f) in layout] if layout else None
        rng = np.random.default_rng(7)
        theta0 = rng.uniform(-0.05, 0.05, d).astype(np.float32)
        theta = theta0.copy()               # this rank's copy
        m_loc = [np.zeros(d, np.float32) for _ in range(Wl)]
        theta_ref = theta0.copy()           # single-process run of all W workers
        m_ref = [np.zeros(d, np.float32) for _ in range(W)]
        bufs = cdist.allocate_buffers(plan, "cpu")
        cw = plan.chunk_words

        for t in range(STEPS):
            g_all = _grads(d, W, t, grad)
            ref = oracle.step(d=d, W=W, layout=lay, beta1=BETA1, beta2=BETA2, lr=LR, wd=WD, mode=mode, nbits=nbits,
                              flags=flags, sync_interval=sync_interval, t=t, grads=g_all, theta=theta_ref, m=m_ref)
            g_loc = g_all[first:first + Wl]
            sync = cdist.is_sync_step(t, sync_interval, plan)

            # -- compress (the rank's workers; their momenta move, theta is not used)
            scratch = theta.copy()
            m_new = [x.copy() for x in m_loc]
            out = oracle.step(d=d, W=Wl, layout=lay, beta1=BETA1, beta2=BETA2, lr=LR, wd=WD, mode=mode, nbits=nbits,
                              flags=flags, sync_interval=0, t=t, grads=g_loc, theta=scratch, m=m_new)
            if sign:
                send = bufs[lc.DIST_SEND].numpy().view(np.uint32).reshape(N, Wl, cw)
                send[:] = 0
                for c in range(N):
                    for i in range(Wl):
                        piece = out.wire[i][c * cw:(c + 1) * cw]
                        send[c, i, :piece.size] = piece
            if sync:
                ss = bufs[lc.DIST_SYNC_SEND].numpy().reshape(Wl, slots)
                base = 0
                for (o, n) in flagged:
                    for i in range(Wl):
                        ss[i, base:base + n] = m_new[i][o:o + n]
                    base += (n + 2047) // 2048 * 2048
            cdist.exchange_after_compress(bufs, mode, sync)

            # -- reduce
            if sign:
                recv = bufs[lc.DIST_RECV].numpy().view(np.uint32).reshape(W, cw)
                c0 = rank * plan.chunk
                L = max(0, min(d - c0, plan.chunk))
                for j in range(W):  # the owner received every worker's words of its chunk
                    want = ref.wire[j][c0 // 32:(c0 + L + 31) // 32]
                    assert np.array_equal(recv[j, :want.size], want), (name, t, j)
                rows = [np.ascontiguousarray(recv[j]) for j in range(W)]
                dc = bufs[lc.DIST_DIR_CHUNK].numpy().view(np.uint32)
                dc[:] = 0
                if plan.dir_bits == 2:
                    for e in range(L):
                        u = int(oracle.direction(oracle.vote(rows, e), W, flags, t))
                        dc[e // 16] |= np.uint32((u & 3) << (2 * (e % 16)))
                else:
                    db = dc.view(np.int8)
                    for e in range(L):
                        db[e] = oracle.vote(rows, e)
            else:
                agg = bufs[lc.DIST_AGG].numpy()
                agg[:] = 0
                for e in range(d):
                    agg[e] = oracle.code_sum(out.wire, nbits, e)
            cdist.exchange_after_reduce(bufs, mode)

            # -- apply
            if sign:
                da = bufs[lc.DIST_DIR_ALL].numpy().view(np.uint32)
                if plan.dir_bits == 2:
                    u_all = _unpack2(da, d).astype(np.float64)
                else:
                    sums = da.view(np.int8)[:d]
                    u_all = np.array([oracle.direction(int(s), W, flags, t) for s in sums])
                if not flags & 0x100:  # (with tie alternation a tied vote moves theta too)
                    assert np.array_equal(np.sign(ref.agg), np.sign(u_all).astype(int)), (name, t)
            else:
                sums = bufs[lc.DIST_AGG].numpy()[:d].astype(np.int64)
                assert np.array_equal(sums, ref.agg), (name, t)
                u_all = np.array([oracle.direction(int(s), W, flags, t) for s in sums])
            for e in range(d):
                theta[e] = oracle.apply(float(theta[e]), float(u_all[e]), LR, WD)
            if sync:
                sr = bufs[lc.DIST_SYNC_RECV].numpy().reshape(W, slots)
                rows = [np.ascontiguousarray(sr[j]) for j in range(W)]
                base = 0
                for (o, n) in flagged:
                    oracle.sync_average(rows, base, base + n)
                    for i in range(Wl):
                        m_new[i][o:o + n] = rows[0][base:base + n]
                    base += (n + 2047) // 2048 * 2048
            m_loc = m_new

            assert np.array_equal(theta.view(np.uint32), theta_ref.view(np.uint32)), \
                (name, rank, t, int((theta != theta_ref).sum()))
            for i in range(Wl):
                assert np.array_equal(m_loc[i].view(np.uint32), m_ref[first + i].view(np.uint32)), (name, rank, t, i)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("name", sorted(CASES))
def test_exchange_equals_single_process_oracle(name):
    import multiprocessing as mp
    import __graft_entry__  # noqa: F401  (puts the repository root on sys.path)
    from communication_compressed_sign_gb300 import build
    build.build()
    oracle.build()
    nranks = CASES[name][3]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, nranks, port, name, q)) for r in range(nranks)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(nranks):
        r, msg = q.get(timeout=300)
        results[r] = msg
    for p in procs:
        p.join(timeout=60)
    bad = {r: m for r, m in results.items() if m != "ok"}
    assert not bad, "\n".join(f"rank {r}:\n{m}" for r, m in bad.items())
    assert all(p.exitcode == 0 for p in procs)


def test_plan_rejects_bad_partitions():
    from communication_compressed_sign_gb300 import build
    from communication_compressed_sign_gb300 import lioncub as lc
    build.build()
    for (W, N, rank, mode) in ((6, 4, 0, 0), (4, 5, 0, 0), (4, 2, 2, 0), (128, 2, 0, 0x200)):
        with pytest.raises(lc.LionCubError) as e:
            lc.lioncub_dist_plan_make(10_000, W, N, rank, None, mode, 1, 0)
        assert e.value.code == lc.ERR_ARG
    # one rank: the whole vector is its chunk
    p = lc.lioncub_dist_plan_make(10_000, 8, 1, 0, None, 0, 1, 0)
    assert p.chunk == 12_288 and p.local_workers == 8 and p.first_worker == 0
