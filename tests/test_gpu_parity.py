"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

The five workloads run at their full sizes, in the launch configuration the
benchmark times; the oracle checks pieces of them (see tests/parity.py).
Small cases cover ragged sizes, many worker counts, both gradient dtypes,
every code width, the tie and average rules, the sync interval, exact zeros,
the host-buffer entry point, determinism, checkpoint/resume and the error
paths.  Sign mode must be bit-exact; L1 mode within the tolerances stated in
tests/parity.py.
"""
import dataclasses

import numpy as np
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

WL = synth.workloads()


def _names(wl, *names):
    return parity.tensor_pieces(wl.layout, set(names))


# ---------------------------------------------------------------------------
# the five workloads, full size
# ---------------------------------------------------------------------------

def test_workload1_flat_1m_full():
    wl = WL[1]
    rep = parity.run_parity(wl, parity.tensor_pieces(wl.layout, {"flat"}), wl.steps)
    assert rep.elements == 1_048_576


def test_workload2_gpt2_small_sign():
    wl = WL[2]
    pieces = sorted(parity.chunk_pieces(wl.layout, "wte", 8, 4096, seed=2)
                    + _names(wl, "h11.attn.c_proj.w", "h11.ln_2.w", "h11.ln_2.b", "h11.mlp.c_fc.b",
                             "ln_f.w", "ln_f.b"), key=lambda p: p.src)
    parity.run_parity(wl, pieces, wl.steps)


def test_workload3_gpt2_medium_l1_n4():
    wl = WL[3]
    pieces = _names(wl, "wpe", "h0.ln_1.w", "h0.attn.c_attn.b", "h7.attn.c_proj.w", "h23.mlp.c_proj.b",
                    "ln_f.w", "ln_f.b")
    rep = parity.run_parity(wl, pieces, wl.steps)
    print(rep)


@pytest.mark.parametrize("interval,beta2", [(1, 0.99), (10, 0.95)])
def test_workload4_gpt2_medium_w16_sync(interval, beta2):
    """As configured (sync every step), and with the pages' periodic setting:
    beta2 = 0.95 and the embedding's momentum synchronized every 10 steps."""
    wl = dataclasses.replace(WL[4], sync_interval=interval, beta2=beta2)
    pieces = sorted(parity.chunk_pieces(wl.layout, "wte", 16, 2048, seed=4)
                    + _names(wl, "wpe", "h3.attn.c_proj.w", "ln_f.b"), key=lambda p: p.src)
    assert any(p.flags for p in pieces)
    parity.run_parity(wl, pieces, wl.steps)


def test_workload5_xl_l1_n2():
    wl = WL[5]
    pieces = _names(wl, "wpe", "h0.ln_1.w", "h12.attn.c_proj.w", "ln_f.w", "ln_f.b")
    rep = parity.run_parity(wl, pieces, wl.steps)
    print(rep)


def test_workload6_vit_b16_dlion_average():
    """ViT-B/16 (86,567,656 parameters, ImageNet head) with the D-Lion
    average aggregation: patch projection, position embedding, one block's
    attention and MLP weights, the head and its ragged 1000-element bias."""
    wl = WL[6]
    assert wl.flags == lc.FLAG_AVERAGE
    pieces = _names(wl, "patch_embed.w", "cls_token", "pos_embed", "blocks5.attn.qkv.w", "blocks5.mlp.fc2.w",
                    "norm.b", "head.w", "head.b")
    parity.run_parity(wl, pieces, wl.steps)


def test_workload7_deit_tiny_l1_embedding_head_sync():
    """DeiT-Tiny with a 100-class head, 4-bit codes, the input embedding
    (patch projection, class token, position embedding) and the head's
    momentum synchronized every step: every tensor, whole."""
    wl = WL[7]
    parity.run_parity(wl, parity.tensor_pieces(wl.layout, {n for (n, _, _, _) in wl.layout}), wl.steps)


@pytest.mark.parametrize("key,names,steps", [
    (3, ("wte",), 2),
    (4, ("wte",), 3),
    (5, ("wte", "head", "h0.mlp.c_fc.w"), 2),
])
def test_largest_tensors_whole(key, names, steps):
    """The largest tensors of the 350M and 1.3B workloads, whole, at full
    size and in the benchmark's launch configuration: every element's wire
    field, aggregate, theta and momentum against the oracle (51.5M to 222.6M
    parameters, 8 or 16 workers; the momentum-synchronized embedding of the
    16-worker workload included)."""
    wl = WL[key]
    pieces = _names(wl, *names)
    assert sum(p.n for p in pieces) >= 51_000_000
    rep = parity.run_parity(wl, pieces, steps)
    print(rep)


# ---------------------------------------------------------------------------
# small cases
# ---------------------------------------------------------------------------

def _small(d, W, grad="bf16", mode=0, nbits=1, layout=None, sync_interval=0, dist=None, seed=0):
    layout = layout if layout is not None else synth.flat_layout(d)
    if dist is None:
        dist = ("t", 3.0, 1e-3, 0.0, 1.0) if grad == "bf16" else ("normal", 1e-3)
    return synth.Workload(0, "small", W, layout, grad, dist, mode, nbits, 6, sync_interval=sync_interval,
                          seed=seed)


SMALL = [
    # d, W, grad, mode, nbits
    (1, 1, "f32", 0, 1), (31, 2, "bf16", 0, 1), (33, 3, "f32", 0, 1), (2047, 5, "bf16", 0, 1),
    (2048, 16, "bf16", 0, 1), (2049, 4, "f32", 0, 1), (6005, 7, "bf16", 0, 1), (40000, 128, "bf16", 0, 1),
    (1, 1, "bf16", 1, 2), (33, 2, "f32", 1, 4), (2047, 3, "bf16", 1, 8), (2049, 5, "bf16", 1, 2),
    (6005, 16, "f32", 1, 4), (100003, 8, "bf16", 1, 4), (4099, 128, "bf16", 1, 8), (70001, 2, "bf16", 1, 2),
]


@pytest.mark.parametrize("d,W,grad,mode,nbits", SMALL)
def test_small_ragged(d, W, grad, mode, nbits):
    wl = _small(d, W, grad, mode, nbits, seed=d + W)
    parity.run_parity(wl, parity.tensor_pieces(wl.layout, {"flat"}), 6)


def _multi_layout(sync=True):
    sizes = [("emb", 320), ("w1", 2048 * 3), ("empty", 0), ("b1", 32), ("w2", 4096 + 64), ("tail", 45)]
    out, off = [], 0
    for name, n in sizes:
        out.append((name, off, n, synth.SYNC_M if (sync and name == "emb") else 0))
        off += n
    return out


@pytest.mark.parametrize("mode,nbits", [(0, 1), (1, 2), (1, 4), (1, 8)])
@pytest.mark.parametrize("interval", [1, 3])
def test_multi_tensor_sync(mode, nbits, interval):
    layout = _multi_layout()
    wl = _small(synth.layout_total(layout), 6, "bf16", mode, nbits, layout=layout, sync_interval=interval)
    pieces = parity.tensor_pieces(layout, {n for (n, _, _, _) in layout})
    parity.run_parity(wl, pieces, 7)


@pytest.mark.parametrize("mode,nbits", [(0, 1), (1, 8)])
def test_many_small_tensors(mode, nbits):
    """2,000 tensors of 32 to 4,128 elements (every tile boundary case: one
    partial tile, exactly one tile, several tiles plus a ragged one), a
    ragged last tensor, a tenth of them momentum-synchronized every second
    step: the per-tensor tile table, the (worker, tensor) M1 combine and
    the split between plain and synchronized tiles at scale."""
    rng = np.random.default_rng(77 + nbits)
    sizes = [int(x) * 32 for x in rng.integers(1, 130, 1999)] + [45]
    layout, off = [], 0
    for k, n in enumerate(sizes):
        layout.append((f"t{k}", off, n, synth.SYNC_M if rng.random() < 0.1 else 0))
        off += n
    wl = _small(off, 5, "bf16", mode, nbits, layout=layout, sync_interval=2, seed=nbits)
    parity.run_parity(wl, parity.tensor_pieces(layout, {n for (n, _, _, _) in layout}), 4)


@pytest.mark.parametrize("flags", [lc.FLAG_TIE_ALTERNATE, lc.FLAG_AVERAGE])
@pytest.mark.parametrize("W", [2, 4, 9])
def test_tie_and_average_rules(flags, W):
    wl = _small(5000, W, "bf16", 0, 1, seed=W)
    parity.run_parity(wl, parity.tensor_pieces(wl.layout, {"flat"}), 5, mode_flags=flags)


def test_tie_alternate_in_l1_mode():
    wl = _small(5000, 4, "bf16", 1, 2)
    parity.run_parity(wl, parity.tensor_pieces(wl.layout, {"flat"}), 4, mode_flags=lc.FLAG_TIE_ALTERNATE)


def _zero_pattern(t, i, g):
    # every third element zero on even workers, every fifth on odd ones
    g[:: 3 if i % 2 == 0 else 5] = 0


def test_exact_zero_update_vectors():
    """Zero gradients with m = 0 give c == 0 exactly, so the alternating rule
    decides those bits (and, where every worker is zero, the vote)."""
    wl = _small(4096 + 17, 4, "bf16", 0, 1, dist=("t", 3.0, 0.0, 0.0, 1.0))  # scale 0: all-zero gradients
    parity.run_parity(wl, parity.tensor_pieces(wl.layout, {"flat"}), 4)
    wl = _small(4096 + 17, 4, "bf16", 1, 4, dist=("t", 3.0, 0.0, 0.0, 1.0))
    parity.run_parity(wl, parity.tensor_pieces(wl.layout, {"flat"}), 3)
    for mode, nbits in ((0, 1), (1, 2)):
        wl = _small(9000 + 5, 6, "f32", mode, nbits)
        parity.run_parity(wl, parity.tensor_pieces(wl.layout, {"flat"}), 5, grad_hook=_zero_pattern)


@pytest.mark.parametrize("mode,nbits,interval", [(0, 1, 0), (1, 4, 3)])
def test_host_steps_pipelined_back_to_back(mode, nbits, interval):
    """Eight lioncub_step_host calls issued back to back with no host
    synchronization, each from its own set of page-locked gradient buffers:
    uploads run ahead into the two staging buffers while earlier steps
    compute, so any missing ordering between an upload and the step that
    last read its staging buffer would change the result.  theta (device and
    host copy) and every momentum must equal eight device-buffer steps on
    the same gradients, bit for bit."""
    dev = torch.device("cuda", 0)
    layout = [("a", 0, 3 << 20, synth.SYNC_M if interval else 0), ("b", 3 << 20, (1 << 20) + 77, 0)]
    wl = _small(synth.layout_total(layout), 4, "bf16", mode, nbits, layout=layout, sync_interval=interval)
    K = 8
    grads = [[torch.empty(wl.d, dtype=torch.bfloat16, device=dev) for _ in range(wl.W)] for _ in range(K)]
    for t in range(K):
        for i in range(wl.W):
            synth.fill_grad_(grads[t][i], wl, t, i)
    host = [[lc.HostBuffer(wl.d, torch.bfloat16) for _ in range(wl.W)] for _ in range(K)]
    for t in range(K):
        for i in range(wl.W):
            host[t][i].tensor.copy_(grads[t][i])
    theta_out = lc.HostBuffer(wl.d, torch.float32)

    def run(use_host):
        theta = torch.empty(wl.d, dtype=torch.float32, device=dev)
        synth.fill_theta_(theta, wl)
        m = [torch.zeros(wl.d, dtype=torch.float32, device=dev) for _ in range(wl.W)]
        h = lc.lioncub_create(wl.d, wl.W, synth.abi_layout(layout), wl.beta1, wl.beta2, wl.lr, wl.wd, mode, nbits,
                              lc.GRAD_BF16, interval)
        try:
            lc.lioncub_bind_state(h, theta.data_ptr(), [x.data_ptr() for x in m])
            torch.cuda.synchronize()
            s = torch.cuda.current_stream().cuda_stream
            for t in range(K):
                if use_host:
                    lc.lioncub_step_host(h, [x.data_ptr() for x in host[t]], theta_out.data_ptr(), s)
                else:
                    lc.lioncub_step(h, [x.data_ptr() for x in grads[t]], s)
            torch.cuda.synchronize()
        finally:
            lc.lioncub_destroy(h)
        return theta, m

    try:
        th_a, m_a = run(False)
        th_b, m_b = run(True)
        assert torch.equal(th_a.view(torch.int32), th_b.view(torch.int32))
        assert torch.equal(theta_out.tensor.view(torch.int32), th_a.cpu().view(torch.int32))
        for x, y in zip(m_a, m_b):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    finally:
        for row in host:
            for x in row:
                x.close()
        theta_out.close()


@pytest.mark.parametrize("host_mem", ["library", "torch", "pageable"])
def test_host_buffer_entry_point(host_mem):
    """lioncub_step_host from page-locked buffers (lioncub_host_alloc or
    torch's pinned allocator: theta stored into the mapped output by SM
    threads) and from pageable ones (copies); a vector length that is not a
    multiple of 4 covers the download's tail."""
    wl = _small(70000, 4, "bf16", 0, 1)
    parity.run_parity(wl, parity.tensor_pieces(wl.layout, {"flat"}), 3, use_host_step=True, host_mem=host_mem)
    wl = _small(70001, 3, "f32", 1, 4)
    parity.run_parity(wl, parity.tensor_pieces(wl.layout, {"flat"}), 3, use_host_step=True, host_mem=host_mem)


# ---------------------------------------------------------------------------
# determinism, checkpoint / resume, error paths
# ---------------------------------------------------------------------------

def _run_gpu(wl, steps, start=0, state=None, flags=0):
    dev = torch.device("cuda", 0)
    d, W = wl.d, wl.W
    if state is None:
        theta = torch.empty(d, dtype=torch.float32, device=dev)
        synth.fill_theta_(theta, wl)
        m = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
    else:
        theta, m = state
    grads = [torch.empty(d, dtype=synth.grad_dtype(wl), device=dev) for _ in range(W)]
    h = lc.lioncub_create(d, W, synth.abi_layout(wl.layout), wl.beta1, wl.beta2, wl.lr, wl.wd,
                          wl.mode | wl.flags | flags, wl.nbits, lc.GRAD_F32 if wl.grad == "f32" else lc.GRAD_BF16,
                          wl.sync_interval)
    m1 = None
    try:
        lc.lioncub_bind_state(h, theta.data_ptr(), [x.data_ptr() for x in m])
        lc.lioncub_set_step(h, start)
        for t in range(start, start + steps):
            for i in range(W):
                synth.fill_grad_(grads[i], wl, t, i)
            lc.lioncub_step(h, [g.data_ptr() for g in grads], torch.cuda.current_stream().cuda_stream)
        assert lc.lioncub_get_step(h) == start + steps
        if wl.mode == 1:
            m1 = torch.empty((W, len(wl.layout)), dtype=torch.float32, device=dev)
            lc.lioncub_debug_export(h, lc.EXPORT_M1, m1.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
    finally:
        lc.lioncub_destroy(h)
    return theta, m, m1


def test_deterministic_l1():
    """M1 and theta repeat bit for bit from run to run (fixed tiling, fixed
    reduction order), including a tensor spanning hundreds of tiles."""
    layout = [("a", 0, 1 << 20, 0), ("b", 1 << 20, 3 * 2048 + 64, 0), ("c", (1 << 20) + 3 * 2048 + 64, 77, 0)]
    small = synth.Workload(0, "det", 4, layout, "bf16", WL[3].dist, 1, 4, 3)
    a = _run_gpu(small, 3)
    b = _run_gpu(small, 3)
    assert torch.equal(a[2].view(torch.int32), b[2].view(torch.int32))
    assert torch.equal(a[0].view(torch.int32), b[0].view(torch.int32))


@pytest.mark.parametrize("mode,nbits,interval", [(0, 1, 2), (1, 4, 3)])
def test_checkpoint_resume(mode, nbits, interval):
    """10 steps straight equal 5 steps, a save of (theta, m, t), a new handle
    restored to t = 5, and 5 more steps -- bit for bit."""
    layout = _multi_layout()
    wl = _small(synth.layout_total(layout), 4, "bf16", mode, nbits, layout=layout, sync_interval=interval)
    th_a, m_a, _ = _run_gpu(wl, 10)
    th_b, m_b, _ = _run_gpu(wl, 5)
    saved = (th_b.clone(), [x.clone() for x in m_b])
    th_c, m_c, _ = _run_gpu(wl, 5, start=5, state=saved)
    assert torch.equal(th_a.view(torch.int32), th_c.view(torch.int32))
    for x, y in zip(m_a, m_c):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


def test_error_paths():
    dev = torch.device("cuda", 0)
    d, W = 4096, 2
    h = lc.lioncub_create(d, W, None, 0.9, 0.99, 1e-4, 0.1, 0, 1, lc.GRAD_BF16, 0)
    try:
        g = [torch.zeros(d, dtype=torch.bfloat16, device=dev) for _ in range(W)]
        with pytest.raises(lc.LionCubError) as e:
            lc.lioncub_step(h, [x.data_ptr() for x in g])
        assert e.value.code == lc.ERR_STATE
        theta = torch.zeros(d + 4, dtype=torch.float32, device=dev)
        m = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
        with pytest.raises(lc.LionCubError) as e:
            lc.lioncub_bind_state(h, theta.data_ptr() + 4, [x.data_ptr() for x in m])
        assert e.value.code == lc.ERR_ALIGN
        lc.lioncub_bind_state(h, theta.data_ptr(), [x.data_ptr() for x in m])
        with pytest.raises(lc.LionCubError) as e:
            lc.lioncub_step(h, [g[0].data_ptr(), g[1].data_ptr() + 2])
        assert e.value.code == lc.ERR_ALIGN
        with pytest.raises(lc.LionCubError) as e:
            lc.lioncub_step(h, [g[0].data_ptr(), 0])
        assert e.value.code == lc.ERR_ARG
        assert lc.lioncub_get_step(h) == 0  # failed steps do not advance t
        with pytest.raises(lc.LionCubError) as e:
            lc.lioncub_debug_export(h, lc.EXPORT_M1, theta.data_ptr())
        assert e.value.code == lc.ERR_STATE
        lc.lioncub_step(h, [x.data_ptr() for x in g])
        torch.cuda.synchronize()
        assert lc.lioncub_get_step(h) == 1
    finally:
        lc.lioncub_destroy(h)


def test_empty_vector():
    h = lc.lioncub_create(0, 3, None, 0.9, 0.99, 1e-4, 0.1, 1, 4, lc.GRAD_BF16, 1)
    try:
        dev = torch.device("cuda", 0)
        buf = torch.zeros(4, dtype=torch.float32, device=dev)
        lc.lioncub_bind_state(h, buf.data_ptr(), [buf.data_ptr()] * 3)
        lc.lioncub_step(h, [buf.data_ptr()] * 3)
        torch.cuda.synchronize()
        assert lc.lioncub_get_step(h) == 1
        assert lc.lioncub_wire_words(h) == 0
    finally:
        lc.lioncub_destroy(h)


def test_profile_counts_launches():
    wl = _small(100000, 4, "bf16", 1, 4)
    dev = torch.device("cuda", 0)
    theta = torch.zeros(wl.d, dtype=torch.float32, device=dev)
    m = [torch.zeros(wl.d, dtype=torch.float32, device=dev) for _ in range(wl.W)]
    g = [torch.ones(wl.d, dtype=torch.bfloat16, device=dev) for _ in range(wl.W)]
    h = lc.lioncub_create(wl.d, wl.W, None, 0.9, 0.99, 1e-4, 0.1, 1, 4, lc.GRAD_BF16, 0)
    try:
        lc.lioncub_bind_state(h, theta.data_ptr(), [x.data_ptr() for x in m])
        lc.lioncub_profile(h, 3)
        for _ in range(5):
            lc.lioncub_step(h, [x.data_ptr() for x in g])
        for k in (lc.KERNEL_COMPRESS, lc.KERNEL_M1, lc.KERNEL_M1_FINAL, lc.KERNEL_REDUCE_APPLY):
            ms, n = lc.lioncub_profile_read(h, k)
            assert n == 3 and ms > 0.0
        assert lc.lioncub_profile_read(h, lc.KERNEL_DIAGNOSE) == (0.0, 0)
    finally:
        lc.lioncub_destroy(h)


# ---------------------------------------------------------------------------
# diagnostics (sign match / flip, ties, momentum spread)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode,nbits,flags", [(0, 1, 0), (0, 1, lc.FLAG_TIE_ALTERNATE), (0, 1, lc.FLAG_AVERAGE),
                                              (1, 2, 0), (1, 4, 0), (1, 8, 0)])
def test_diagnose_small(mode, nbits, flags):
    layout = _multi_layout(sync=False)
    wl = _small(synth.layout_total(layout), 6, "bf16", mode, nbits, layout=layout)
    parity.run_diag_parity(wl, {n for (n, _, _, _) in layout}, warm_steps=3, mode_flags=flags)


@pytest.mark.parametrize("W", [6, 8])
@pytest.mark.parametrize("warm", [2, 3])
@pytest.mark.parametrize("mode,nbits", [(0, 1), (1, 2), (1, 4)])
def test_diagnose_exact_zero_updates(mode, nbits, warm, W):
    """Elements whose update vector is exactly 0 at both step parities (their
    vote is the step's zero sign in sign mode, code 0 in L1 mode), with a
    power-of-two and another worker count (the mean's two code paths)."""
    layout = _multi_layout(sync=False)
    wl = _small(synth.layout_total(layout), W, "bf16", mode, nbits, layout=layout)
    res = parity.run_diag_parity(wl, {n for (n, _, _, _) in layout}, warm_steps=warm, zero_stride=5)
    assert any(r["dropped"] + r["spurious"] > 0 for _, r in res) or mode == 1


@pytest.mark.parametrize("warm", [2, 3])
def test_diagnose_many_tiles_odd_workers(warm):
    """Sign-mode diagnostics on more tiles than the persistent grid holds
    (each block loops over several tiles and asks L2 for the next), with a
    worker count that is not a power of two (the mean by division) and
    ragged tensors, every tensor checked whole at both step parities."""
    sizes = [1_000_003 // 32 * 32, 2048 * 700 + 96, 32, 2_100_000 // 32 * 32, 4096 + 480]
    layout, off = [], 0
    for k, n in enumerate(sizes):
        layout.append((f"t{k}", off, n, 0))
        off += n
    wl = _small(off, 6, "bf16", 0, 1, layout=layout)
    parity.run_diag_parity(wl, {n for (n, _, _, _) in layout}, warm_steps=warm, zero_stride=97)


def test_diagnose_full_size_workloads():
    for key, names in ((2, {"wpe", "h5.mlp.c_fc.b", "ln_f.w"}), (3, {"wpe", "h0.attn.c_attn.b", "ln_f.b"}),
                       (4, {"h3.attn.c_proj.w", "ln_f.w"})):
        res = parity.run_diag_parity(WL[key], names, warm_steps=2)
        for name, r in res:
            print(key, name, r)


@pytest.mark.parametrize("mode,nbits,flags,qbits", [(0, 1, 0, 2), (0, 1, lc.FLAG_TIE_ALTERNATE, 4), (1, 4, 0, 4),
                                                      (1, 2, 0, 8), (0, 1, lc.FLAG_AVERAGE, 4)])
def test_diagnose_qinf_small(mode, nbits, flags, qbits):
    """The Q_inf comparator ("Lion Cub" page, "Core claim" and Fig. 4 caption)
    against the oracle on every tensor of a ragged multi-tensor layout:
    every count exact, with each code width and tie rule."""
    layout = _multi_layout(sync=False)
    wl = _small(synth.layout_total(layout), 6, "bf16", mode, nbits, layout=layout)
    parity.run_qinf_parity(wl, {n for (n, _, _, _) in layout}, qbits, seed=12345, warm_steps=3, mode_flags=flags)


def test_diagnose_qinf_full_size_workloads():
    """Q_inf at full size: GPT-2 small (W = 8) and the 1.3B layout (n = 2 as
    its codes), sampled tensors checked whole; most Q_inf codes are zero on
    the heavy-tailed update (the pages' observation)."""
    for key, names, qbits in ((2, {"wpe", "h5.mlp.c_fc.b", "h7.attn.c_proj.w", "ln_f.w"}, 4),
                              (5, {"wpe", "h3.ln_1.b", "h9.attn.c_proj.w", "ln_f.b"}, 2)):
        res = parity.run_qinf_parity(WL[key], names, qbits, seed=7, warm_steps=2)
        for name, r in res:
            n = [x for x in WL[key].layout if x[0] == name][0][2]
            if n >= 500_000:  # a large tensor's max-norm sits far out in the tail
                assert r["zero_codes"] > 0.5 * WL[key].W * n, (key, name, r)
            print(key, name, r)


# ---------------------------------------------------------------------------
# beyond 32-bit element indices
# ---------------------------------------------------------------------------

def test_beyond_int32_elements():
    """d = 2^31 + 4133 elements (two tensors, the second ragged): every index
    in the kernels is 64-bit.  Sign mode, W = 2, bf16 gradients (~35 GB on the
    device); the oracle checks pieces at the start, across the 2^31 boundary
    and at the ragged end."""
    big = (1 << 31) - (1 << 20)
    d = (1 << 31) + 4096 + 37
    layout = [("a", 0, big, 0), ("b", big, d - big, 0)]
    wl = _small(d, 2, "bf16", 0, 1, layout=layout)
    pieces = [parity.Piece(0, 4096, 0, -1), parity.Piece((1 << 31) - 2048, 4096, 0, -1),
              parity.Piece(d - 101, 101, 0, -1)]
    parity.run_parity(wl, pieces, 2)
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# guard bands: no kernel writes outside the caller's buffers
# ---------------------------------------------------------------------------

GUARD = 64  # floats of sentinel before and after every buffer (256 bytes keeps alignment)


def _guarded(n, dtype, fill):
    dev = torch.device("cuda", 0)
    buf = torch.empty(n + 2 * GUARD * (4 // torch.tensor([], dtype=dtype).element_size()), dtype=dtype, device=dev)
    g = GUARD * (4 // buf.element_size())
    buf.view(torch.uint8).fill_(0xA5)
    inner = buf[g:g + n]
    fill(inner)
    return buf, inner, g


@pytest.mark.parametrize("mode,nbits,d,sync", [(0, 1, 2049, 1), (0, 1, 33, 0), (1, 2, 4099, 1), (1, 8, 70001, 0)])
def test_guard_bands_untouched(mode, nbits, d, sync):
    W = 3
    layout = [("a", 0, 32 * (d // 64), synth.SYNC_M if sync else 0), ("b", 32 * (d // 64), d - 32 * (d // 64), 0)]
    wl = _small(d, W, "bf16", mode, nbits, layout=layout, sync_interval=sync)
    tb, theta, gt = _guarded(d, torch.float32, lambda x: synth.fill_theta_(x, wl))
    ms = [_guarded(d, torch.float32, lambda x: x.zero_()) for _ in range(W)]
    gs = [_guarded(d, torch.bfloat16, lambda x: x.zero_()) for _ in range(W)]
    h = lc.lioncub_create(d, W, synth.abi_layout(layout), 0.9, 0.99, 1e-4, 0.1, mode, nbits, lc.GRAD_BF16, sync)
    try:
        lc.lioncub_bind_state(h, theta.data_ptr(), [x[1].data_ptr() for x in ms])
        for t in range(3):
            for i in range(W):
                synth.fill_grad_(gs[i][1], wl, t, i)
            lc.lioncub_step(h, [x[1].data_ptr() for x in gs], torch.cuda.current_stream().cuda_stream)
        out = torch.empty(len(layout) * lc.DIAG_BYTES, dtype=torch.uint8, device=theta.device)
        lc.lioncub_diagnose(h, [x[1].data_ptr() for x in gs], out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        status = torch.ones(1, dtype=torch.int32, device=theta.device)
        lc.lioncub_debug_export(h, lc.EXPORT_STATUS, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for buf, inner, g in [(tb, theta, gt)] + ms + gs:
            raw = buf.view(torch.uint8)
            eb = buf.element_size()
            assert bool((raw[: g * eb] == 0xA5).all()), "write before the buffer"
            assert bool((raw[(g + d) * eb:] == 0xA5).all()), "write after the buffer"
    finally:
        lc.lioncub_destroy(h)


@pytest.mark.parametrize("mode,nbits", [(0, 1), (1, 4)])
def test_all_layer_momentum_sync(mode, nbits):
    """Every tensor flagged: the momenta of all workers are equal after each
    sync step (interval 2) and match the oracle."""
    layout = [(n, o, k, synth.SYNC_M) for (n, o, k, _) in _multi_layout(sync=False)]
    wl = _small(synth.layout_total(layout), 5, "bf16", mode, nbits, layout=layout, sync_interval=2)
    parity.run_parity(wl, parity.tensor_pieces(layout, {n for (n, _, _, _) in layout}), 6)


# ---------------------------------------------------------------------------
# the torch-tensor convenience wrapper is marshalling only
# ---------------------------------------------------------------------------

def test_optimizer_wrapper_matches_c_abi():
    from communication_compressed_sign_gb300 import LionCubOptimizer
    layout = _multi_layout()
    wl = _small(synth.layout_total(layout), 3, "bf16", 1, 4, layout=layout, sync_interval=2)
    ref_theta, ref_m, _ = _run_gpu(wl, 4)
    dev = torch.device("cuda", 0)
    theta = torch.empty(wl.d, dtype=torch.float32, device=dev)
    synth.fill_theta_(theta, wl)
    m = [torch.zeros(wl.d, dtype=torch.float32, device=dev) for _ in range(wl.W)]
    opt = LionCubOptimizer(wl.d, wl.W, synth.abi_layout(layout), beta1=wl.beta1, beta2=wl.beta2, lr=wl.lr,
                           wd=wl.wd, mode=1, nbits=4, sync_interval=2)
    opt.bind(theta, m)
    grads = [torch.empty(wl.d, dtype=torch.bfloat16, device=dev) for _ in range(wl.W)]
    for t in range(4):
        for i in range(wl.W):
            synth.fill_grad_(grads[i], wl, t, i)
        opt.step(grads)
    torch.cuda.synchronize()
    assert opt.t == 4
    assert torch.equal(theta.view(torch.int32), ref_theta.view(torch.int32))
    for x, y in zip(m, ref_m):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    with pytest.raises(ValueError):
        opt.step(grads[:-1])
    with pytest.raises(ValueError):
        opt.step([g.float() for g in grads])  # the handle takes bf16 gradients
    with pytest.raises(ValueError):
        opt.bind(theta, m[:-1])
    opt.close()


def test_create_out_of_memory_leaks_nothing():
    """A layout whose wire buffer cannot fit (W = 128 workers of 2^35
    elements: 512 GB of packed signs) fails with LIONCUB_ERR_OOM and leaves
    device memory as it was."""
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    with pytest.raises(lc.LionCubError) as e:
        lc.lioncub_create(1 << 35, 128, None, 0.9, 0.99, 1e-4, 0.1, 0, 1, lc.GRAD_BF16, 0)
    assert e.value.code == lc.ERR_OOM
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free1 - free0) < (64 << 20)
    # the library is still usable afterwards
    h = lc.lioncub_create(4096, 2, None, 0.9, 0.99, 1e-4, 0.1, 0, 1, lc.GRAD_BF16, 0)
    lc.lioncub_destroy(h)


# ---------------------------------------------------------------------------
# CUDA graphs and concurrent handles
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode,nbits", [(0, 1), (1, 4)])
def test_step_replays_from_cuda_graphs(mode, nbits):
    """lioncub_step only enqueues kernels, so it can be captured.  The step
    counter advances when a step is enqueued (and its parity picks the sign
    of exact zeros), so a loop with fixed gradient buffers captures one even
    and one odd step and replays them alternately; the result must equal
    plain steps bit for bit."""
    layout = _multi_layout()
    wl = _small(synth.layout_total(layout), 4, "bf16", mode, nbits, layout=layout, sync_interval=2)
    ref_theta, ref_m, _ = _run_gpu(wl, 6)

    dev = torch.device("cuda", 0)
    theta = torch.empty(wl.d, dtype=torch.float32, device=dev)
    synth.fill_theta_(theta, wl)
    m = [torch.zeros(wl.d, dtype=torch.float32, device=dev) for _ in range(wl.W)]
    grads = [torch.zeros(wl.d, dtype=torch.bfloat16, device=dev) for _ in range(wl.W)]
    h = lc.lioncub_create(wl.d, wl.W, synth.abi_layout(layout), wl.beta1, wl.beta2, wl.lr, wl.wd, mode, nbits,
                          lc.GRAD_BF16, 2)
    try:
        lc.lioncub_bind_state(h, theta.data_ptr(), [x.data_ptr() for x in m])
        s = torch.cuda.Stream()
        gp = [g.data_ptr() for g in grads]
        graphs = []
        saved = (theta.clone(), [x.clone() for x in m])
        with torch.cuda.stream(s):
            for _ in range(2):  # t = 0 (even) and t = 1 (odd); sync_now differs too (interval 2)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    lc.lioncub_step(h, gp, s.cuda_stream)
                graphs.append(g)
        torch.cuda.synchronize()
        # capture ran nothing on the data: restore the state anyway, then replay
        theta.copy_(saved[0])
        for x, y in zip(m, saved[1]):
            x.copy_(y)
        for t in range(6):
            for i in range(wl.W):
                synth.fill_grad_(grads[i], wl, t, i)
            graphs[t % 2].replay()
        torch.cuda.synchronize()
        assert torch.equal(theta.view(torch.int32), ref_theta.view(torch.int32))
        for x, y in zip(m, ref_m):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    finally:
        lc.lioncub_destroy(h)


def test_two_handles_on_two_streams():
    """Handles share no state: two steps running concurrently on two streams
    give the same results as running them one after the other."""
    wl_a = _small(300_000, 4, "bf16", 0, 1, seed=1)
    wl_b = _small(200_000 + 45, 3, "bf16", 1, 2, seed=2)
    ref_a = _run_gpu(wl_a, 3)
    ref_b = _run_gpu(wl_b, 3)
    dev = torch.device("cuda", 0)

    def setup(wl):
        theta = torch.empty(wl.d, dtype=torch.float32, device=dev)
        synth.fill_theta_(theta, wl)
        m = [torch.zeros(wl.d, dtype=torch.float32, device=dev) for _ in range(wl.W)]
        grads = [[torch.empty(wl.d, dtype=torch.bfloat16, device=dev) for _ in range(wl.W)] for _ in range(3)]
        for t in range(3):
            for i in range(wl.W):
                synth.fill_grad_(grads[t][i], wl, t, i)
        h = lc.lioncub_create(wl.d, wl.W, None, wl.beta1, wl.beta2, wl.lr, wl.wd, wl.mode, wl.nbits,
                              lc.GRAD_BF16, 0)
        lc.lioncub_bind_state(h, theta.data_ptr(), [x.data_ptr() for x in m])
        return h, theta, m, grads

    ha, ta, ma, ga = setup(wl_a)
    hb, tb, mb, gb = setup(wl_b)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    try:
        for t in range(3):
            lc.lioncub_step(ha, [g.data_ptr() for g in ga[t]], sa.cuda_stream)
            lc.lioncub_step(hb, [g.data_ptr() for g in gb[t]], sb.cuda_stream)
        torch.cuda.synchronize()
        for (theta, m), ref in (((ta, ma), ref_a), ((tb, mb), ref_b)):
            assert torch.equal(theta.view(torch.int32), ref[0].view(torch.int32))
            for x, y in zip(m, ref[1]):
                assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    finally:
        lc.lioncub_destroy(ha)
        lc.lioncub_destroy(hb)
