"""GPU-vs-oracle parity harness (used by the gpu-marked tests and smoke()).

The CUDA library runs the whole workload on the GPU through its C ABI; the
CPU oracle runs the same steps on a set of *pieces* of the flat parameter
vector, fed with a host copy of exactly the gradient bits the GPU used.  In
sign mode every element is independent, so any 32-aligned piece is a valid
sub-problem; in L1 mode M1 spans a whole tensor, so pieces are whole
tensors.  After every step the harness compares, piece by piece, the wire
words, the aggregates, M1 (L1 mode), theta and the momenta.

Tolerances (sign mode: everything bit-exact):
  L1 mode -- M1 within 1e-6 relative; codes differ by at most one quantum on
  at most 1e-5 of the elements (near-ties that follow from the last bits of
  M1, whose fp64 summation order differs); theta within 1e-6 relative except
  at elements whose aggregate differed at some step; momenta bit-exact (they
  do not depend on the quantization).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle
import synth
from communication_compressed_sign_gb300 import lioncub as lc

M1_RTOL = 1e-6
CODE_FRAC = 1e-5
THETA_RTOL = 1e-6


@dataclass
class Piece:
    src: int        # offset in the full flat vector (multiple of 32)
    n: int
    flags: int
    tensor: int     # index of the tensor in the full layout (for M1), -1 if partial


def tensor_pieces(layout, names):
    out = []
    for k, (name, off, n, fl) in enumerate(layout):
        if name in names:
            out.append(Piece(off, n, fl, k))
    return out


def chunk_pieces(layout, name, count, length, seed=0):
    """`count` random 32-aligned chunks of `length` elements inside tensor `name`."""
    k = [i for i, t in enumerate(layout) if t[0] == name][0]
    _, off, n, fl = layout[k]
    rng = np.random.default_rng(seed)
    starts = sorted(set(int(s) * 32 for s in rng.integers(0, (n - length) // 32, size=count)))
    res, last = [], -1
    for s in starts:
        if s < last:
            continue
        res.append(Piece(off + s, length, fl, -1))
        last = s + length
    return res


def _words_range(p: Piece, bits: int):
    w0 = p.src * bits // 32
    return w0, (p.n * bits + 31) // 32


@dataclass
class ParityReport:
    steps: int = 0
    elements: int = 0
    wire_mismatch_words: int = 0
    agg_mismatch: int = 0
    code_offby1: int = 0
    code_worse: int = 0
    m1_max_rel: float = 0.0
    m1_inexact: int = 0
    theta_max_rel: float = 0.0
    theta_mismatch: int = 0
    theta_mismatch_outside_agg: int = 0
    m_mismatch: int = 0


def run_parity(wl: synth.Workload, pieces, steps: int, *, mode_flags: int = 0, strict: bool = True,
               use_host_step: bool = False, host_mem: str = "library", grad_hook=None):
    """Run `steps` steps of workload `wl` on the GPU and on the oracle (over
    `pieces`); return a ParityReport.  With strict=True, assert the bounds.
    grad_hook(t, i, tensor), if given, edits worker i's step-t gradients on
    the GPU after they are generated (both sides see the edited bits).
    use_host_step runs lioncub_step_host from host buffers of kind host_mem
    ("library": lioncub_host_alloc, "torch": torch's pinned allocator,
    "pageable") and checks its theta output too."""
    import torch

    dev = torch.device("cuda", 0)
    W, d = wl.W, wl.d
    l1 = wl.mode == 1
    bits = wl.nbits if l1 else 1
    gdt = synth.grad_dtype(wl)

    theta = torch.empty(d, dtype=torch.float32, device=dev)
    synth.fill_theta_(theta, wl)
    m = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
    grads = [torch.empty(d, dtype=gdt, device=dev) for _ in range(W)]

    mode_flags |= wl.flags
    h = lc.lioncub_create(d, W, synth.abi_layout(wl.layout), wl.beta1, wl.beta2, wl.lr, wl.wd,
                          wl.mode | mode_flags, wl.nbits, lc.GRAD_F32 if wl.grad == "f32" else lc.GRAD_BF16,
                          wl.sync_interval)
    try:
        lc.lioncub_bind_state(h, theta.data_ptr(), [x.data_ptr() for x in m])
        nwords = lc.lioncub_wire_words(h)
        wire = torch.empty((W, max(nwords, 1)), dtype=torch.int32, device=dev)
        agg = torch.empty(max(d, 1), dtype=torch.int32, device=dev)
        K = len(wl.layout)
        m1 = torch.empty((W, K), dtype=torch.float32, device=dev) if l1 else None

        # oracle sub-problem: the pieces laid end to end (inner pieces have
        # 32-multiple lengths, so every destination offset stays 32-aligned)
        for p in pieces[:-1]:
            assert p.n % 32 == 0, "inner pieces must have 32-multiple lengths"
        dsub = sum(p.n for p in pieces)
        sub_layout, dst = [], 0
        for p in pieces:
            sub_layout.append((dst, p.n, p.flags))
            dst += p.n
        if l1:
            assert all(p.tensor >= 0 for p in pieces), "L1 mode needs whole-tensor pieces (M1 is per tensor)"
        wranges = [_words_range(p, bits) for p in pieces]

        # Pieces are gathered by slicing (views, no gather kernel).
        for p in pieces:
            assert 0 <= p.src and p.src + p.n <= d and p.src % 32 == 0, f"piece {p} outside [0, {d})"

        def gather(x):
            return torch.cat([x[p.src:p.src + p.n] for p in pieces])

        def gather_words(x):
            return torch.cat([x[:, w0:w0 + nw] for (w0, nw) in wranges], dim=1)

        theta_o = gather(theta).cpu().numpy().copy()
        m_o = [np.zeros(dsub, np.float32) for _ in range(W)]
        rep = ParityReport(elements=dsub)
        agg_diverged = np.zeros(dsub, bool)
        stream = torch.cuda.current_stream()

        pinned = None
        theta_host = None
        if use_host_step:
            keep = []

            def host_buf(dtype):
                if host_mem == "library":
                    keep.append(lc.HostBuffer(d, dtype))
                    return keep[-1].tensor
                x = torch.empty(d, dtype=dtype)
                return x.pin_memory() if host_mem == "torch" else x
            pinned = [host_buf(gdt) for _ in range(W)]
            theta_host = host_buf(torch.float32)

        for t in range(steps):
            for i in range(W):
                synth.fill_grad_(grads[i], wl, t, i)
                if grad_hook is not None:
                    grad_hook(t, i, grads[i])
            g_o = []
            for i in range(W):
                gi = gather(grads[i]).cpu()
                g_o.append(gi.view(torch.int16).numpy().view(np.uint16).copy() if wl.grad == "bf16"
                           else gi.numpy().copy())
            if use_host_step:
                for i in range(W):
                    pinned[i].copy_(grads[i])
                torch.cuda.synchronize()
                lc.lioncub_step_host(h, [x.data_ptr() for x in pinned], theta_host.data_ptr(),
                                     stream.cuda_stream)
            else:
                lc.lioncub_step(h, [g.data_ptr() for g in grads], stream.cuda_stream)
            lc.lioncub_debug_export(h, lc.EXPORT_WIRE, wire.data_ptr(), stream.cuda_stream)
            lc.lioncub_debug_export(h, lc.EXPORT_AGG, agg.data_ptr(), stream.cuda_stream)
            if l1:
                lc.lioncub_debug_export(h, lc.EXPORT_M1, m1.data_ptr(), stream.cuda_stream)
            torch.cuda.synchronize()
            if use_host_step:
                assert torch.equal(theta_host, theta.cpu()), "host-step theta copy differs from device theta"

            out = oracle.step(d=dsub, W=W, layout=sub_layout, beta1=wl.beta1, beta2=wl.beta2, lr=wl.lr,
                              wd=wl.wd, mode=wl.mode, nbits=wl.nbits, flags=mode_flags,
                              sync_interval=wl.sync_interval, t=t, grads=g_o, theta=theta_o, m=m_o)
            rep.steps += 1
            wire_h = gather_words(wire).cpu().numpy().view(np.uint32)
            agg_h = gather(agg).cpu().numpy()
            agg_diff = agg_h != out.agg
            rep.agg_mismatch += int(agg_diff.sum())
            agg_diverged |= agg_diff

            # wire words / codes
            dst, gsel = 0, 0
            for k_sub, (p, (_, nw)) in enumerate(zip(pieces, wranges)):
                ow0 = dst * bits // 32
                for i in range(W):
                    gw = wire_h[i, gsel:gsel + nw]
                    ow = out.wire[i][ow0:ow0 + nw]
                    neq = gw != ow
                    if neq.any():
                        rep.wire_mismatch_words += int(neq.sum())
                        if l1:
                            gc = _decode(gw, bits, p.n)
                            oc = _decode(ow, bits, p.n)
                            dd = np.abs(gc - oc)
                            rep.code_offby1 += int((dd == 1).sum())
                            rep.code_worse += int((dd > 1).sum())
                if l1 and p.tensor >= 0:
                    g_m1 = m1[:, p.tensor].cpu().numpy()
                    o_m1 = out.m1[:, k_sub]
                    rel = np.abs(g_m1.astype(np.float64) - o_m1) / np.maximum(np.abs(o_m1), 1e-30)
                    rep.m1_max_rel = max(rep.m1_max_rel, float(rel.max()))
                    rep.m1_inexact += int((g_m1 != o_m1).sum())
                dst += p.n
                gsel += nw

            th_g = gather(theta).cpu().numpy()
            neq = th_g.view(np.uint32) != theta_o.view(np.uint32)
            rep.theta_mismatch = int(neq.sum())
            rep.theta_mismatch_outside_agg = int((neq & ~agg_diverged).sum())
            rel = np.abs(th_g.astype(np.float64) - theta_o) / np.maximum(np.abs(theta_o), 1e-30)
            rel_ok = rel[~agg_diverged]
            rep.theta_max_rel = float(rel_ok.max()) if rel_ok.size else 0.0
            mm = 0
            for i in range(W):
                mm += int((gather(m[i]).cpu().numpy().view(np.uint32) != m_o[i].view(np.uint32)).sum())
            rep.m_mismatch = mm

            if strict:
                _assert_bounds(rep, l1, W, t)
        # the status word: no bounded wait gave up, no index left its buffer
        # (bounds-checked builds), no guard band around the scratch changed
        status = torch.ones(1, dtype=torch.int32, device=dev)
        lc.lioncub_debug_export(h, lc.EXPORT_STATUS, status.data_ptr(), stream.cuda_stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"device status word {int(status.item())}"
        return rep
    finally:
        lc.lioncub_destroy(h)


def _decode(words, bits, n):
    per = 32 // bits
    e = np.arange(n)
    f = (words[e // per].astype(np.int64) >> (bits * (e % per))) & ((1 << bits) - 1)
    return np.where(f >= (1 << (bits - 1)), f - (1 << bits), f)


def _assert_bounds(rep: ParityReport, l1: bool, W: int, t: int):
    if not l1:
        assert rep.wire_mismatch_words == 0, f"step {t}: packed sign words differ: {rep}"
        assert rep.agg_mismatch == 0, f"step {t}: vote counts differ: {rep}"
        assert rep.theta_mismatch == 0, f"step {t}: theta differs: {rep}"
        assert rep.m_mismatch == 0, f"step {t}: momentum differs: {rep}"
    else:
        assert rep.m1_max_rel <= M1_RTOL, f"step {t}: M1 beyond {M1_RTOL} relative: {rep}"
        assert rep.code_worse == 0, f"step {t}: a code differs by more than one quantum: {rep}"
        limit = CODE_FRAC * rep.elements * W * rep.steps
        assert rep.code_offby1 <= max(limit, 0), f"step {t}: too many off-by-one codes: {rep}"
        assert rep.theta_max_rel <= THETA_RTOL, f"step {t}: theta beyond {THETA_RTOL}: {rep}"
        assert rep.theta_mismatch_outside_agg == 0, f"step {t}: theta differs where the aggregate agreed: {rep}"
        assert rep.m_mismatch == 0, f"step {t}: momentum differs: {rep}"


def run_diag_parity(wl: synth.Workload, tensor_names, warm_steps: int = 2, mode_flags: int = 0,
                    zero_stride: int = 0):
    """Warm the state up with `warm_steps` GPU steps, then compare
    lioncub_diagnose for the next step's gradients with the oracle's
    diagnostics on the named whole tensors (every field exact).  With
    zero_stride > 0 every zero_stride-th gradient is 0 at every step, so the
    momentum and the update vector stay exactly 0 there.  Returns the GPU
    records of those tensors."""
    import torch

    dev = torch.device("cuda", 0)
    W, d = wl.W, wl.d
    gdt = synth.grad_dtype(wl)
    theta = torch.empty(d, dtype=torch.float32, device=dev)
    synth.fill_theta_(theta, wl)
    m = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
    grads = [torch.empty(d, dtype=gdt, device=dev) for _ in range(W)]
    mode_flags |= wl.flags
    h = lc.lioncub_create(d, W, synth.abi_layout(wl.layout), wl.beta1, wl.beta2, wl.lr, wl.wd,
                          wl.mode | mode_flags, wl.nbits, lc.GRAD_F32 if wl.grad == "f32" else lc.GRAD_BF16,
                          wl.sync_interval)
    try:
        lc.lioncub_bind_state(h, theta.data_ptr(), [x.data_ptr() for x in m])
        s = torch.cuda.current_stream().cuda_stream
        def fill(t):
            for i in range(W):
                synth.fill_grad_(grads[i], wl, t, i)
                if zero_stride:
                    grads[i][::zero_stride] = 0

        for t in range(warm_steps):
            fill(t)
            lc.lioncub_step(h, [g.data_ptr() for g in grads], s)
        t = warm_steps
        fill(t)
        K = len(wl.layout)
        out = torch.zeros(K * lc.DIAG_BYTES, dtype=torch.uint8, device=dev)
        theta_before = theta.clone()
        lc.lioncub_diagnose(h, [g.data_ptr() for g in grads], out.data_ptr(), s)
        torch.cuda.synchronize()
        assert lc.lioncub_get_step(h) == t and torch.equal(theta, theta_before)  # nothing updated
        gpu = lc.decode_diag(out.cpu().numpy().tobytes(), K)
        status = torch.ones(1, dtype=torch.int32, device=dev)
        lc.lioncub_debug_export(h, lc.EXPORT_STATUS, status.data_ptr(), s)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, "a kernel reported a timed-out wait or an out-of-bounds index"
        res = []
        for k, (name, off, n, fl) in enumerate(wl.layout):
            if name not in tensor_names:
                continue
            g_o = []
            for i in range(W):
                gi = grads[i][off:off + n].cpu()
                g_o.append(gi.view(torch.int16).numpy().view(np.uint16).copy() if wl.grad == "bf16"
                           else gi.numpy().copy())
            m_o = [x[off:off + n].cpu().numpy().copy() for x in m]
            o = oracle.diagnose(d=n, W=W, layout=None, beta1=wl.beta1, mode=wl.mode, nbits=wl.nbits,
                                flags=mode_flags, t=t, grads=g_o, m=m_o)[0]
            assert gpu[k] == o, (name, gpu[k], o)
            assert sum(gpu[k][f] for f in ("match", "flip", "dropped", "spurious")) == n
            res.append((name, gpu[k]))
        return res
    finally:
        lc.lioncub_destroy(h)


def run_qinf_parity(wl: synth.Workload, tensor_names, nbits: int, seed: int, warm_steps: int = 2,
                    mode_flags: int = 0):
    """Warm the state up with `warm_steps` GPU steps, then compare
    lioncub_diagnose_qinf for the next step's gradients with the oracle's
    Q_inf comparison on the named whole tensors (every field exact; the
    random counters use each tensor's flat offset).  Returns the GPU records
    of those tensors."""
    import torch

    dev = torch.device("cuda", 0)
    W, d = wl.W, wl.d
    gdt = synth.grad_dtype(wl)
    theta = torch.empty(d, dtype=torch.float32, device=dev)
    synth.fill_theta_(theta, wl)
    m = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
    grads = [torch.empty(d, dtype=gdt, device=dev) for _ in range(W)]
    mode_flags |= wl.flags
    h = lc.lioncub_create(d, W, synth.abi_layout(wl.layout), wl.beta1, wl.beta2, wl.lr, wl.wd,
                          wl.mode | mode_flags, wl.nbits, lc.GRAD_F32 if wl.grad == "f32" else lc.GRAD_BF16,
                          wl.sync_interval)
    try:
        lc.lioncub_bind_state(h, theta.data_ptr(), [x.data_ptr() for x in m])
        s = torch.cuda.current_stream().cuda_stream
        for t in range(warm_steps):
            for i in range(W):
                synth.fill_grad_(grads[i], wl, t, i)
            lc.lioncub_step(h, [g.data_ptr() for g in grads], s)
        t = warm_steps
        for i in range(W):
            synth.fill_grad_(grads[i], wl, t, i)
        K = len(wl.layout)
        out = torch.full((K * lc.QINF_BYTES,), 0xAB, dtype=torch.uint8, device=dev)
        theta_before = theta.clone()
        lc.lioncub_diagnose_qinf(h, [g.data_ptr() for g in grads], nbits, seed, out.data_ptr(), s)
        torch.cuda.synchronize()
        assert lc.lioncub_get_step(h) == t and torch.equal(theta, theta_before)  # nothing updated
        gpu = lc.decode_qinf(out.cpu().numpy().tobytes(), K)
        res = []
        for k, (name, off, n, fl) in enumerate(wl.layout):
            if name not in tensor_names:
                continue
            g_o = []
            for i in range(W):
                gi = grads[i][off:off + n].cpu()
                g_o.append(gi.view(torch.int16).numpy().view(np.uint16).copy() if wl.grad == "bf16"
                           else gi.numpy().copy())
            m_o = [x[off:off + n].cpu().numpy().copy() for x in m]
            o = oracle.diagnose_qinf(d=n, W=W, layout=None, beta1=wl.beta1, nbits=nbits, flags=mode_flags, t=t,
                                     seed=seed, e_base=off, grads=g_o, m=m_o)[0]
            assert gpu[k] == o, (name, gpu[k], o)
            assert sum(gpu[k][f] for f in ("match", "flip", "dropped", "spurious")) == n
            res.append((name, gpu[k]))
        return res
    finally:
        lc.lioncub_destroy(h)
