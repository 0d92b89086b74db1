"""GB300 library for the compressed Lion update step of Lion Cub / Distributed
Lion, with W data-parallel workers simulated as W buffer sets in one GPU.

The compute path is liblioncub.so (hand-written CUDA for sm_103a behind the C
ABI of include/lioncub.h); :mod:`.lioncub` is its ctypes binding and
:class:`LionCubOptimizer` a small convenience wrapper that takes torch CUDA
tensors and passes their pointers through.
"""
from __future__ import annotations

from . import lioncub
from .lioncub import (  # noqa: F401
    FLAG_AVERAGE, FLAG_TIE_ALTERNATE, GRAD_BF16, GRAD_F32, MODE_L1_INTSUM, MODE_SIGN_MAJORITY,
    TENSOR_SYNC_M, LionCubError,
)


class LionCubOptimizer:
    """Owns one library handle; state and gradients are torch CUDA tensors.

    theta: (d,) float32; m: list of W (d,) float32 tensors; gradients passed
    to :meth:`step` are W (d,) tensors of bfloat16 or float32 (matching
    ``grad_dtype``).  All must be contiguous and stay alive while used.
    """

    def __init__(self, d, W, layout, *, beta1=0.9, beta2=0.99, lr=1e-4, wd=0.1,
                 mode=MODE_SIGN_MAJORITY, nbits=1, grad_dtype=GRAD_BF16, sync_interval=0):
        self.d, self.W = int(d), int(W)
        self.mode, self.nbits, self.grad_dtype = mode, nbits, grad_dtype
        self.h = lioncub.lioncub_create(self.d, self.W, layout, beta1, beta2, lr, wd, mode, nbits,
                                        grad_dtype, sync_interval)
        self._keep = None

    def bind(self, theta, m):
        import torch
        if len(m) != self.W:
            raise ValueError(f"expected {self.W} momentum tensors")
        for x in (theta, *m):
            if not (x.is_cuda and x.is_contiguous()) or x.dtype != torch.float32 or x.numel() != self.d:
                raise ValueError("theta and m must be contiguous float32 CUDA tensors of d elements")
        lioncub.lioncub_bind_state(self.h, theta.data_ptr(), [x.data_ptr() for x in m])
        self._keep = (theta, list(m))

    def step(self, grads, stream=None):
        import torch
        if len(grads) != self.W:
            raise ValueError(f"expected {self.W} gradient tensors")
        want = torch.bfloat16 if self.grad_dtype == GRAD_BF16 else torch.float32
        for g in grads:
            if not (g.is_cuda and g.is_contiguous()) or g.dtype != want or g.numel() != self.d:
                raise ValueError(f"gradients must be contiguous {want} CUDA tensors of d elements")
        s = stream.cuda_stream if stream is not None else _current_stream()
        lioncub.lioncub_step(self.h, [g.data_ptr() for g in grads], s)

    @property
    def t(self) -> int:
        return lioncub.lioncub_get_step(self.h)

    @t.setter
    def t(self, value: int) -> None:
        lioncub.lioncub_set_step(self.h, value)

    def close(self):
        if self.h:
            lioncub.lioncub_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _current_stream() -> int:
    import torch
    return torch.cuda.current_stream().cuda_stream
