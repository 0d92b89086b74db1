"""The compressed Lion step with its W workers spread over the ranks of a
torch.distributed process group (one GPU per rank).

"Lion Cub: Minimizing Communication Overhead in Distributed Lion" (quoted
body text on the implementation; "What carries the argument"): 1-bit Lion
Cub exchanges its packed signs with an AlltoAll -- each rank receives every
worker's signs for the chunk of the parameter vector it owns, takes their
majority, and the results are gathered back -- while the 4-bit and wider
variants sum their integer codes with an AllReduce; the momenta of the
input-embedding and output layers are averaged over the workers.

Each of the N ranks holds W/N workers (their gradients and momenta) and a
copy of theta.  The library's kernels do every arithmetic step
(``lioncub_dist_compress`` / ``lioncub_dist_reduce`` / ``lioncub_dist_apply``);
this module only allocates the exchange buffers the library's plan asks for
and issues the collectives between those calls, on the step's stream:

    sign mode   compress | all-to-all SEND -> RECV | reduce |
                allgather DIR_CHUNK -> DIR_ALL | apply
    L1 mode     compress | reduce | allreduce (sum) AGG | apply
    sync steps  allgather SYNC_SEND -> SYNC_RECV before the apply

With NCCL the collectives run on the current CUDA stream's order (torch
makes its communication stream wait for the current stream, and the current
stream wait for the collective), so the three launches and the collectives
form one ordered sequence without host synchronization.  Every rank ends the
step with the same theta, and each rank's momenta equal those of the same
workers in a single-GPU step over all W workers, bit for bit.
"""
from __future__ import annotations

from . import lioncub as lc


def buffer_dtypes(plan):
    """torch dtype of each exchange buffer (the collectives move them as such;
    the code sums are added as int8 or int32)."""
    import torch
    agg = torch.int8 if plan.agg_bytes == 1 else torch.int32
    return (torch.int32, torch.int32, torch.int32, torch.int32, agg, torch.float32, torch.float32)


def allocate_buffers(plan, device):
    """One tensor per exchange buffer of the plan (None where it needs none)."""
    import torch
    out = []
    for b, dt in enumerate(buffer_dtypes(plan)):
        nbytes = int(plan.bytes[b])
        if nbytes == 0:
            out.append(None)
            continue
        item = torch.empty(0, dtype=dt).element_size()
        assert nbytes % item == 0
        out.append(torch.zeros(nbytes // item, dtype=dt, device=device))
    return out


def is_sync_step(t: int, sync_interval: int, plan) -> bool:
    """Whether the step at counter t averages the synchronized momenta."""
    return sync_interval > 0 and plan.sync_slots > 0 and (t + 1) % sync_interval == 0


def exchange_after_compress(bufs, mode: int, sync: bool, group=None) -> None:
    """Sign mode: the all-to-all of the packed words (segment r of SEND goes
    to rank r).  Sync steps: the allgather of the new momenta to average."""
    import torch.distributed as dist
    if (mode & 0xff) == lc.MODE_SIGN_MAJORITY:
        dist.all_to_all_single(bufs[lc.DIST_RECV], bufs[lc.DIST_SEND], group=group)
    if sync:
        dist.all_gather_into_tensor(bufs[lc.DIST_SYNC_RECV], bufs[lc.DIST_SYNC_SEND], group=group)


def exchange_after_reduce(bufs, mode: int, group=None) -> None:
    """Sign mode: the allgather of the chunk owners' directions.  L1 mode:
    the allreduce (sum) of the code sums."""
    import torch.distributed as dist
    if (mode & 0xff) == lc.MODE_SIGN_MAJORITY:
        dist.all_gather_into_tensor(bufs[lc.DIST_DIR_ALL], bufs[lc.DIST_DIR_CHUNK], group=group)
    else:
        dist.all_reduce(bufs[lc.DIST_AGG], op=dist.ReduceOp.SUM, group=group)


class DistLionCub:
    """One rank's share of the data-parallel step.

    d, W, layout and the hyper-parameters are those of the whole step (as
    for ``lioncub_create``); this rank holds workers
    ``plan.first_worker .. plan.first_worker + plan.local_workers - 1``.
    theta: (d,) float32 CUDA tensor (every rank its own copy); m: the local
    workers' (d,) float32 momenta; gradients passed to :meth:`step`: the
    local workers' (d,) bfloat16 or float32 tensors.
    """

    def __init__(self, d, W, layout, *, group=None, beta1=0.9, beta2=0.99, lr=1e-4, wd=0.1,
                 mode=lc.MODE_SIGN_MAJORITY, nbits=1, grad_dtype=lc.GRAD_BF16, sync_interval=0, device=None):
        import torch
        import torch.distributed as dist
        self.group = group
        self.nranks = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.d, self.W, self.mode, self.sync_interval = int(d), int(W), int(mode), int(sync_interval)
        self.grad_dtype = grad_dtype
        self.plan = lc.lioncub_dist_plan_make(self.d, self.W, self.nranks, self.rank, layout, mode, nbits,
                                              sync_interval)
        self.local_workers = self.plan.local_workers
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.h = lc.lioncub_dist_create(self.d, self.W, self.nranks, self.rank, layout, beta1, beta2, lr, wd, mode,
                                        nbits, grad_dtype, sync_interval)
        self.bufs = allocate_buffers(self.plan, self.device)
        lc.lioncub_dist_bind_buffers(self.h, [b.data_ptr() if b is not None else 0 for b in self.bufs])
        self._keep = None

    def bind(self, theta, m_local) -> None:
        import torch
        if len(m_local) != self.local_workers:
            raise ValueError(f"expected {self.local_workers} momentum tensors")
        for x in (theta, *m_local):
            if not (x.is_cuda and x.is_contiguous()) or x.dtype != torch.float32 or x.numel() != self.d:
                raise ValueError("theta and m must be contiguous float32 CUDA tensors of d elements")
        lc.lioncub_bind_state(self.h, theta.data_ptr(), [x.data_ptr() for x in m_local])
        self._keep = (theta, list(m_local))

    @property
    def t(self) -> int:
        return lc.lioncub_get_step(self.h)

    def step(self, grads_local, stream=None) -> None:
        """One step: the three launches and the collectives between them, all
        ordered on `stream` (default: the current stream)."""
        import torch
        if len(grads_local) != self.local_workers:
            raise ValueError(f"expected {self.local_workers} gradient tensors")
        want = torch.bfloat16 if self.grad_dtype == lc.GRAD_BF16 else torch.float32
        for g in grads_local:
            if not (g.is_cuda and g.is_contiguous()) or g.dtype != want or g.numel() != self.d:
                raise ValueError(f"gradients must be contiguous {want} CUDA tensors of d elements")
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        sync = is_sync_step(self.t, self.sync_interval, self.plan)
        with torch.cuda.stream(s):
            lc.lioncub_dist_compress(self.h, [g.data_ptr() for g in grads_local], s.cuda_stream)
            exchange_after_compress(self.bufs, self.mode, sync, self.group)
            lc.lioncub_dist_reduce(self.h, s.cuda_stream)
            exchange_after_reduce(self.bufs, self.mode, self.group)
            lc.lioncub_dist_apply(self.h, s.cuda_stream)

    def close(self) -> None:
        if self.h:
            lc.lioncub_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
