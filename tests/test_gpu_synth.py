"""The seeded input generator (synth/synth.cu) against the distributions the
workloads state, on the GPU: N(0, 1e-3^2) gradients, 1e-3 * Student-t(nu)
gradients for nu = 3 and nu = 2.5 (with 0.1 % of entries scaled by 100),
U(-0.05, 0.05) parameters; bf16 outputs are the fp32 samples rounded to
nearest even; streams are reproducible and distinct per (step, worker).
Quantiles come from scipy's Student-t and normal distributions."""
import math

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
stats = pytest.importorskip("scipy.stats")

N = 1 << 23


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"


def _fill(kind, p, dtype=torch.float32, stream_id=7, n=N):
    x = torch.empty(n, dtype=dtype, device="cuda")
    synth.fill_(x, kind, 0, stream_id, p)
    torch.cuda.synchronize()
    return x


def _abs_quantile(x, q):
    return float(torch.quantile(x.abs().float()[: 1 << 24], q).item())


def test_normal():
    sigma = 1e-3
    x = _fill(0, (sigma, 0, 0, 0)).double()
    assert abs(float(x.mean())) < 5 * sigma / math.sqrt(N)
    assert abs(float(x.std()) / sigma - 1) < 5e-3
    med = float(x.abs().median()) / sigma
    assert abs(med / stats.norm.ppf(0.75) - 1) < 5e-3


@pytest.mark.parametrize("nu", [3.0, 2.5])
def test_student_t_quantiles(nu):
    scale = 1e-3
    x = _fill(2, (nu, scale, 0.0, 1.0), dtype=torch.bfloat16).float() / scale
    for q in (0.5, 0.9, 0.98):
        want = stats.t.ppf(0.5 + q / 2, nu)  # quantile q of |t|
        got = _abs_quantile(x, q)
        assert abs(got / want - 1) < 0.02, (nu, q, got, want)


def test_outlier_fraction():
    """nu = 2.5, 0.1 % of entries times 100: the share of |x| > 100 * scale
    is (1 - f) P(|t| > 100) + f P(|t| > 1)."""
    nu, scale, f = 2.5, 1e-3, 0.001
    x = _fill(2, (nu, scale, f, 100.0)).float() / scale
    expect = N * ((1 - f) * 2 * stats.t.sf(100, nu) + f * 2 * stats.t.sf(1, nu))
    got = int((x.abs() > 100).sum())
    assert abs(got - expect) < 6 * math.sqrt(expect), (got, expect)


def test_uniform_theta():
    x = _fill(1, (-0.05, 0.05, 0, 0)).double()
    lo, hi = float(np.float32(-0.05)), float(np.float32(0.05))  # the bounds as fp32 values
    assert float(x.min()) >= lo and float(x.max()) <= hi
    assert abs(float(x.mean())) < 5 * 0.1 / math.sqrt(12 * N)
    assert abs(float(x.var()) / (0.1 ** 2 / 12) - 1) < 5e-3


def test_bf16_is_the_fp32_sample_rounded_to_nearest_even():
    p = (3.0, 1e-3, 0.001, 100.0)
    x32 = _fill(2, p, dtype=torch.float32, n=1 << 20)
    x16 = _fill(2, p, dtype=torch.bfloat16, n=1 << 20)
    assert torch.equal(x16.view(torch.int16), x32.to(torch.bfloat16).view(torch.int16))


def test_streams_reproducible_and_distinct():
    wl = synth.workloads()[2]
    a, b, c, d = (torch.empty(1 << 20, dtype=torch.bfloat16, device="cuda") for _ in range(4))
    synth.fill_grad_(a, wl, 3, 1)
    synth.fill_grad_(b, wl, 3, 1)
    synth.fill_grad_(c, wl, 3, 2)
    synth.fill_grad_(d, wl, 4, 1)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for other in (c, d):
        same = (a.view(torch.int16) == other.view(torch.int16)).float().mean().item()
        assert same < 0.05
