"""Pins for the CPU oracle against facts fixed by the pages or by mathematics.

None of these tests re-types the oracle's own formulas: each checks a
hand-worked value, a closed form, an exact-arithmetic result, a brute-force
count or an invariant, chosen so that a dropped term, a swapped operand or a
wrong sign or index in the oracle fails at least one of them.

Sources: "Lion Cub: Minimizing Communication Overhead in Distributed Lion"
(machine review page: "What carries the argument", Eq. (1), the assumptions
list on the alternating-sign rule and Fig. 10, the quoted body text on tied
majority votes) and "Communication Efficient Distributed Training with
Distributed Lion" (summary page, "Approach").
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(x):
    return np.float32(x)


# ---------------------------------------------------------------------------
# Eq. (1): L1 quantization
# ---------------------------------------------------------------------------

def _golden_q1():
    with open(os.path.join(GOLDEN, "q1_hand_vectors.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden_q1()["cases"], ids=lambda c: c["name"])
def test_q1_hand_vectors(oracle_lib, case):
    x = np.array(case["x"], dtype=np.float32)
    m1 = oracle.m1(x)
    expect_m1 = np.float32(case["m1_num"] / case["m1_den"])
    assert m1 == expect_m1
    q = oracle.q1(x, case["nbits"])
    assert q.tolist() == case["q"]
    words = oracle.pack_codes(q, case["nbits"])
    assert [int(h, 16) for h in case["packed_hex"]] == words.tolist()


def test_q1_two_workers_per_worker_m1(oracle_lib):
    """Each worker scales by its own M1; the integer codes are summed."""
    g = _golden_q1()["two_workers"]
    d = len(g["c0"])
    # beta1 = 0 makes c equal to the gradient exactly (0*m + 1*g).
    grads = [np.array(g["c0"], np.float32), np.array(g["c1"], np.float32)]
    theta = np.zeros(d, np.float32)
    m = [np.zeros(d, np.float32), np.zeros(d, np.float32)]
    out = oracle.step(d=d, W=2, layout=None, beta1=0.0, beta2=0.5, lr=1.0, wd=0.0,
                      mode=oracle.MODE_L1, nbits=g["nbits"], flags=0, sync_interval=0, t=0,
                      grads=grads, theta=theta, m=m)
    assert out.agg.tolist() == g["agg"]
    assert [oracle.code_sum(out.wire, g["nbits"], e) for e in range(d)] == g["agg"]
    # theta = 0 - 1*(sign(agg) + 0)
    assert theta.tolist() == [-float(np.sign(a)) for a in g["agg"]]


def _exact_q1(x, nbits):
    """Eq. (1) in exact rational arithmetic, Python's round() = ties to even."""
    qmax = 2 ** (nbits - 1) - 1
    xs = [Fraction(float(v)) for v in x]
    m1 = sum(abs(v) for v in xs) / len(xs)
    if m1 == 0:
        return [0] * len(xs), [Fraction(0)] * len(xs)
    ys = [qmax * v / m1 for v in xs]
    return [max(-qmax, min(qmax, round(y))) for y in ys], ys


@pytest.mark.parametrize("nbits", [2, 4, 8])
def test_q1_matches_exact_rational(oracle_lib, nbits):
    """fp32 Q1 equals exact-arithmetic Q1 wherever y is not within fp32 rounding
    error of a rounding boundary (k + 1/2)."""
    rng = np.random.default_rng(1234 + nbits)
    checked = 0
    for trial in range(40):
        n = int(rng.integers(1, 200))
        x = (rng.laplace(size=n) * 10.0 ** rng.integers(-4, 3)).astype(np.float32)
        q = oracle.q1(x, nbits)
        qe, ys = _exact_q1(x, nbits)
        for e in range(n):
            frac = abs(ys[e]) - math.floor(abs(ys[e]))
            if abs(frac - Fraction(1, 2)) < Fraction(1, 10 ** 5) * (1 + abs(ys[e])):
                continue
            assert q[e] == qe[e], (trial, e, float(ys[e]))
            checked += 1
    assert checked > 1000


def test_q1_range_and_sign(oracle_lib):
    rng = np.random.default_rng(7)
    x = (rng.standard_t(2.5, size=5000) * 1e-3).astype(np.float32)
    for nbits in (2, 4, 8):
        qmax = 2 ** (nbits - 1) - 1
        q = oracle.q1(x, nbits).astype(np.int64)
        assert q.max() <= qmax and q.min() >= -qmax
        # the code never has the opposite sign of x
        assert np.all(q * np.sign(x) >= 0)


# ---------------------------------------------------------------------------
# M1: mean absolute value, fp64 accumulation
# ---------------------------------------------------------------------------

def test_m1_against_exact_sum(oracle_lib):
    rng = np.random.default_rng(5)
    for n in (1, 2, 31, 1000, 100_003):
        x = (rng.standard_t(3.0, size=n) * 1e-3).astype(np.float32)
        exact = Fraction(math.fsum(abs(float(v)) for v in x)) / n
        got = oracle.m1(x)
        # correctly rounded value of the exact mean, within one fp32 ulp
        ref = np.float32(float(exact))
        assert abs(float(got) - float(ref)) <= float(np.spacing(ref)), (n, got, ref)


def test_m1_exact_when_sum_is_exact(oracle_lib):
    x = np.array([0.5, -0.25, 0.125, -1.0, 2.0, -0.0, 0.0, 4.0], np.float32)
    assert oracle.m1(x) == np.float32(7.875 / 8)
    assert oracle.m1(np.zeros(0, np.float32)) == 0.0


# ---------------------------------------------------------------------------
# Sign packing and the alternating zero rule
# ---------------------------------------------------------------------------

def _unpack(words, n):
    bits = np.unpackbits(np.asarray(words, dtype="<u4").view(np.uint8), bitorder="little")
    return bits[:n], bits[n:]


@pytest.mark.parametrize("n", [1, 31, 32, 33, 1000])
@pytest.mark.parametrize("t", [0, 1])
def test_pack_roundtrip_and_tail(oracle_lib, n, t):
    rng = np.random.default_rng(n * 7 + t)
    c = rng.standard_normal(n).astype(np.float32)
    c[:: 5] = 0.0
    c[1:: 7] = -0.0
    words = oracle.pack_signs(c, t)
    assert words.size == (n + 31) // 32
    bits, tail = _unpack(words, n)
    want = np.where(c > 0, 1, np.where(c < 0, 0, 1 if t % 2 == 0 else 0))
    assert bits.tolist() == want.tolist()
    assert not tail.any()


def test_zero_alternates_by_step(oracle_lib):
    z = np.zeros(32, np.float32)
    assert oracle.pack_signs(z, 0)[0] == 0xFFFFFFFF
    assert oracle.pack_signs(z, 1)[0] == 0
    assert oracle.pack_signs(z, 2)[0] == 0xFFFFFFFF
    assert oracle.pack_signs(-z, 7)[0] == 0
    assert oracle.sign_bit(1e-30, 1) == 1 and oracle.sign_bit(-1e-30, 0) == 0


def test_zero_rule_closed_form(oracle_lib):
    """Every worker has g = m = 0, so all bits are the step's zero sign, the vote
    is +W (even t) or -W (odd t), and theta follows
    theta_{t+1} = theta_t (1 - lr*wd) -/+ lr."""
    d, W, lr, wd = 64, 3, 1e-2, 0.1
    theta = np.linspace(-0.05, 0.05, d).astype(np.float32)
    th64 = theta.astype(np.float64)
    m = [np.zeros(d, np.float32) for _ in range(W)]
    grads = [np.zeros(d, np.uint16) for _ in range(W)]
    for t in range(8):
        out = oracle.step(d=d, W=W, layout=None, beta1=0.9, beta2=0.99, lr=lr, wd=wd,
                          mode=oracle.MODE_SIGN, nbits=1, flags=0, sync_interval=0, t=t,
                          grads=grads, theta=theta, m=m)
        s = 1.0 if t % 2 == 0 else -1.0
        assert all(w.tolist() == ([0xFFFFFFFF] * 2 if s > 0 else [0, 0]) for w in out.wire)
        assert (out.agg == int(s) * W).all()
        th64 = th64 - lr * (s + wd * th64)
        np.testing.assert_allclose(theta, th64, rtol=0, atol=4e-8)


# ---------------------------------------------------------------------------
# Majority vote, integer sums, aggregation rules
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("W", [1, 2, 3, 4, 5])
def test_vote_brute_force(oracle_lib, W):
    """Bit p of worker i's word is bit i of p, so the 32 positions of one word
    cover every sign pattern of W <= 5 workers."""
    words = [np.array([sum(((p >> i) & 1) << p for p in range(32))], np.uint32) for i in range(W)]
    for p in range(32):
        if p >= 2 ** W:
            continue
        pos = bin(p).count("1")
        want = pos - (W - pos)
        assert oracle.vote(words, p) == want
        want_sign = 1.0 if pos * 2 > W else (-1.0 if pos * 2 < W else 0.0)
        assert oracle.direction(want, W, 0, 0) == want_sign


@pytest.mark.parametrize("W", [1, 2, 7, 16])
def test_vote_popcount_identity(oracle_lib, W):
    """sum of +-1 over workers == 2 * popcount - W."""
    rng = np.random.default_rng(W)
    words = [rng.integers(0, 2 ** 32, size=4, dtype=np.uint64).astype(np.uint32) for _ in range(W)]
    bits = np.stack([_unpack(w, 128)[0] for w in words])  # W x 128
    pop = bits.sum(axis=0)
    for e in range(128):
        assert oracle.vote(words, e) == 2 * int(pop[e]) - W


@pytest.mark.parametrize("nbits", [2, 4, 8])
def test_code_sum_brute_force(oracle_lib, nbits):
    rng = np.random.default_rng(nbits)
    qmax = 2 ** (nbits - 1) - 1
    W, n = 6, 77
    codes = [rng.integers(-qmax, qmax + 1, size=n).astype(np.int8) for _ in range(W)]
    words = [oracle.pack_codes(q, nbits) for q in codes]
    total = np.sum(np.stack(codes).astype(np.int64), axis=0)
    for e in range(n):
        assert oracle.code_sum(words, nbits, e) == total[e]
        assert abs(total[e]) <= W * qmax


def test_tie_rules(oracle_lib):
    assert oracle.direction(0, 4, 0, 0) == 0.0
    assert oracle.direction(0, 4, 0, 1) == 0.0
    assert oracle.direction(0, 4, oracle.FLAG_TIE_ALTERNATE, 0) == 1.0
    assert oracle.direction(0, 4, oracle.FLAG_TIE_ALTERNATE, 3) == -1.0
    assert oracle.direction(2, 4, oracle.FLAG_TIE_ALTERNATE, 1) == 1.0


@pytest.mark.parametrize("W", [1, 3, 4, 8])
def test_average_rule(oracle_lib, W):
    """D-Lion Avg: the update is the mean of the workers' +-1 signs."""
    for pos in range(W + 1):
        agg = 2 * pos - W
        want = np.float32(Fraction(agg, W).numerator / Fraction(agg, W).denominator)
        assert oracle.direction(agg, W, oracle.FLAG_AVERAGE, 0) == want


def test_apply_closed_forms(oracle_lib):
    # u = 0: pure decoupled weight decay
    for th in (0.05, -0.03, 1.0):
        th = float(np.float32(th))
        got = oracle.apply(th, 0.0, 1e-4, 0.1)
        assert abs(got - th * (1 - 1e-5)) <= 2 * abs(float(np.spacing(np.float32(th))))
    # wd = 0: theta moves by exactly -lr*u
    assert oracle.apply(0.5, 1.0, 0.25, 0.0) == 0.25
    assert oracle.apply(0.5, -1.0, 0.25, 0.0) == 0.75


# ---------------------------------------------------------------------------
# W = 1 reduces to textbook Lion
# ---------------------------------------------------------------------------

def test_single_worker_is_textbook_lion(oracle_lib):
    """With one worker and no exact-zero update vector, the vote is that worker's
    sign, so ten steps must equal Lion (Chen et al. 2023) written with
    np.sign in fp32, bit for bit."""
    rng = np.random.default_rng(0)
    d = 4096
    b1, b2, lr, wd = np.float32(0.9), np.float32(0.99), np.float32(1e-4), np.float32(0.1)
    theta = rng.uniform(-0.05, 0.05, d).astype(np.float32)
    m = [np.zeros(d, np.float32)]
    th_ref, m_ref = theta.copy(), np.zeros(d, np.float32)
    one = np.float32(1.0)
    for t in range(10):
        g = (rng.standard_normal(d) * 1e-3).astype(np.float32)
        g[g == 0] = np.float32(1e-3)
        # textbook Lion
        upd = np.sign(b1 * m_ref + (one - b1) * g).astype(np.float32)
        assert (upd != 0).all()
        th_ref = th_ref - lr * (upd + wd * th_ref)
        m_ref = b2 * m_ref + (one - b2) * g
        oracle.step(d=d, W=1, layout=None, beta1=float(b1), beta2=float(b2), lr=float(lr),
                    wd=float(wd), mode=oracle.MODE_SIGN, nbits=1, flags=0, sync_interval=0, t=t,
                    grads=[g], theta=theta, m=m)
        assert np.array_equal(theta.view(np.uint32), th_ref.view(np.uint32)), t
        assert np.array_equal(m[0].view(np.uint32), m_ref.view(np.uint32)), t


def test_bf16_gradients_equal_their_fp32_values(oracle_lib):
    """A bf16 number is the upper half of the fp32 bit pattern of the same
    value (bfloat16 format: 1 sign, 8 exponent, 7 fraction bits).  So
    (1) the bf16 patterns 0x3F80, 0xC020, 0x3E20 and 0x0000 are 1.0, -2.5,
    0.15625 and 0.0, which a single step from m = 0 exposes as
    m' = RN(omega2 * g); and (2) gradients whose fp32 patterns have a zero low
    half give the same step -- wire words, theta, m, in both modes -- whether
    passed as bf16 patterns or as fp32."""
    b2 = 0.99
    om2 = np.float32(1.0) - np.float32(b2)
    g16 = np.array([0x3F80, 0xC020, 0x3E20, 0x0000], dtype=np.uint16)
    values = np.array([1.0, -2.5, 0.15625, 0.0], dtype=np.float32)
    m = [np.zeros(4, np.float32)]
    oracle.step(d=4, W=1, layout=None, beta1=0.9, beta2=b2, lr=1e-4, wd=0.1, mode=oracle.MODE_SIGN,
                nbits=1, flags=0, sync_interval=0, t=0, grads=[g16], theta=np.zeros(4, np.float32), m=m)
    assert np.array_equal(m[0], om2 * values)

    rng = np.random.default_rng(5)
    d, W = 3000, 3
    g32 = [((rng.standard_t(3, d) * 1e-3).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000))
           .view(np.float32) for _ in range(W)]
    g16 = [(x.view(np.uint32) >> 16).astype(np.uint16) for x in g32]
    theta0 = rng.uniform(-0.05, 0.05, d).astype(np.float32)
    layout = [(0, 1024, 0), (1024, d - 1024, 0)]
    for mode, nbits in ((oracle.MODE_SIGN, 1), (oracle.MODE_L1, 4)):
        runs = []
        for grads in (g32, g16):
            theta, m = theta0.copy(), [np.zeros(d, np.float32) for _ in range(W)]
            outs = [oracle.step(d=d, W=W, layout=layout, beta1=0.9, beta2=0.99, lr=1e-4, wd=0.1, mode=mode,
                                nbits=nbits, flags=0, sync_interval=0, t=t, grads=grads, theta=theta, m=m)
                    for t in range(3)]
            runs.append((theta, m, outs[-1].wire))
        (ta, ma, wa), (tb, mb, wb) = runs
        assert np.array_equal(ta.view(np.uint32), tb.view(np.uint32))
        for x, y in zip(ma + wa, mb + wb):
            assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def test_omega(oracle_lib):
    assert oracle.omega(0.9) == np.float32(1.0) - np.float32(0.9)
    assert oracle.omega(0.5) == 0.5


# ---------------------------------------------------------------------------
# Momentum sync and step-level invariants
# ---------------------------------------------------------------------------

def test_sync_average_against_exact_mean(oracle_lib):
    rng = np.random.default_rng(11)
    for W in (1, 2, 3, 16):
        ms = [rng.standard_normal(300).astype(np.float32) for _ in range(W)]
        exact = np.mean(np.stack([a.astype(np.float64) for a in ms]), axis=0)
        bound = np.sum(np.abs(np.stack(ms)).astype(np.float64), axis=0) / W * (W + 1) * 2.0 ** -24
        oracle.sync_average(ms, 0, 300)
        for a in ms[1:]:
            assert np.array_equal(a, ms[0])
        assert np.all(np.abs(ms[0].astype(np.float64) - exact) <= bound + 1e-45)
    # power-of-two W with exactly representable sums: exact mean
    ms = [np.full(4, v, np.float32) for v in (1.0, 2.0, 3.0, 6.0)]
    oracle.sync_average(ms, 1, 3)
    assert ms[0].tolist() == [1.0, 3.0, 3.0, 1.0] and ms[3].tolist() == [6.0, 3.0, 3.0, 6.0]


def _gpt_like_layout():
    # three tensors: a flagged "embedding", a middle weight, a ragged last vector
    return [(0, 320, oracle.TENSOR_SYNC_M), (320, 640, 0), (960, 45, 0)]


@pytest.mark.parametrize("mode,nbits", [(oracle.MODE_SIGN, 1), (oracle.MODE_L1, 4), (oracle.MODE_L1, 2)])
def test_step_invariants(oracle_lib, mode, nbits):
    rng = np.random.default_rng(3)
    layout = _gpt_like_layout()
    d, W = 1005, 4
    theta = rng.uniform(-0.05, 0.05, d).astype(np.float32)
    m = [(rng.standard_normal(d) * 1e-3).astype(np.float32) for _ in range(W)]
    grads = [(rng.standard_t(3.0, d) * 1e-3).astype(np.float32) for _ in range(W)]
    # a reference run with sync off, for the untouched tensors
    theta_ns, m_ns = theta.copy(), [a.copy() for a in m]
    th0 = theta.copy()
    oracle.step(d=d, W=W, layout=layout, beta1=0.9, beta2=0.99, lr=1e-4, wd=0.1, mode=mode,
                nbits=nbits, flags=0, sync_interval=0, t=0, grads=grads, theta=theta_ns, m=m_ns)
    out = oracle.step(d=d, W=W, layout=layout, beta1=0.9, beta2=0.99, lr=1e-4, wd=0.1, mode=mode,
                      nbits=nbits, flags=0, sync_interval=1, t=0, grads=grads, theta=theta, m=m)
    assert np.array_equal(theta, theta_ns)  # sync never touches theta
    for i in range(1, W):
        assert np.array_equal(m[i][:320], m[0][:320])  # flagged: all workers equal
    for i in range(W):
        assert np.array_equal(m[i][320:], m_ns[i][320:])  # unflagged: untouched
    qmax = 1 if mode == oracle.MODE_SIGN else 2 ** (nbits - 1) - 1
    assert np.abs(out.agg).max() <= W * qmax
    if mode == oracle.MODE_SIGN:
        assert ((out.agg + W) % 2 == 0).all()
    # padding bits beyond d are zero
    bits_total = 32 * out.wire[0].size
    used = d * (1 if mode == oracle.MODE_SIGN else nbits)
    for w in out.wire:
        allbits = np.unpackbits(w.view(np.uint8), bitorder="little")
        assert not allbits[used:bits_total].any()
    # where the aggregate is zero, theta moved by weight decay only
    z = out.agg == 0
    wdonly = np.array([oracle.apply(float(v), 0.0, 1e-4, 0.1) for v in th0[z]], np.float32)
    assert np.array_equal(theta[z], wdonly)
    if mode == oracle.MODE_L1:
        assert out.m1.shape == (W, 3)
        assert (out.m1 > 0).all()


def test_sync_interval(oracle_lib):
    rng = np.random.default_rng(9)
    layout = [(0, 64, oracle.TENSOR_SYNC_M)]
    d, W = 64, 3
    theta = np.zeros(d, np.float32)
    m = [np.zeros(d, np.float32) for _ in range(W)]
    for t in range(6):
        grads = [rng.standard_normal(d).astype(np.float32) for _ in range(W)]
        oracle.step(d=d, W=W, layout=layout, beta1=0.9, beta2=0.95, lr=1e-3, wd=0.0,
                    mode=oracle.MODE_SIGN, nbits=1, flags=0, sync_interval=3, t=t,
                    grads=grads, theta=theta, m=m)
        synced = all(np.array_equal(m[0], m[i]) for i in range(W))
        assert synced == ((t + 1) % 3 == 0), t


def test_tie_fraction_statistics(oracle_lib):
    """At step 0 with m = 0 and i.i.d. symmetric gradients, a tie happens with
    probability C(W, W/2) / 2^W (37.5% at W=4, 27.3% at W=8, 19.6% at W=16), in
    line with 'over 30% of the parameters' tied at 4 workers and fewer at 8."""
    rng = np.random.default_rng(21)
    d = 20000
    for W in (4, 8, 16):
        grads = [(rng.standard_t(3.0, d) * 1e-3).astype(np.float32) for _ in range(W)]
        theta = np.zeros(d, np.float32)
        m = [np.zeros(d, np.float32) for _ in range(W)]
        out = oracle.step(d=d, W=W, layout=None, beta1=0.9, beta2=0.99, lr=1e-4, wd=0.1,
                          mode=oracle.MODE_SIGN, nbits=1, flags=0, sync_interval=0, t=0,
                          grads=grads, theta=theta, m=m)
        p = math.comb(W, W // 2) / 2 ** W
        frac = float(np.mean(out.agg == 0))
        assert abs(frac - p) < 5 * math.sqrt(p * (1 - p) / d), (W, frac, p)


def test_step_rejects_bad_arguments(oracle_lib):
    d = 40
    g = [np.zeros(d, np.float32)]
    m = [np.zeros(d, np.float32)]
    th = np.zeros(d, np.float32)
    kw = dict(d=d, W=1, beta1=0.9, beta2=0.99, lr=1e-4, wd=0.1, flags=0, sync_interval=0, t=0,
              grads=g, theta=th, m=m)
    with pytest.raises(ValueError):
        oracle.step(layout=[(0, 20, 0), (20, 20, 0)], mode=0, nbits=1, **kw)  # offset not 32-aligned
    with pytest.raises(ValueError):
        oracle.step(layout=[(0, 32, 0)], mode=0, nbits=1, **kw)  # does not cover d
    with pytest.raises(ValueError):
        oracle.step(layout=None, mode=1, nbits=3, **kw)


# ---------------------------------------------------------------------------
# Diagnostics (Fig. 4 / Fig. 11 sign match and flip, Fig. 6 momentum std,
# tied votes)
# ---------------------------------------------------------------------------

def test_worker_std_closed_forms(oracle_lib):
    assert oracle.worker_std([1.0, 3.0]) == 1.0
    assert oracle.worker_std([0.0, 0.0, 0.0, 4.0]) == np.float32(math.sqrt(3.0))
    assert oracle.worker_std([2.5]) == 0.0
    assert oracle.worker_std([-1.0, 1.0, -1.0, 1.0]) == 1.0


def test_classify_table(oracle_lib):
    assert oracle.classify(1.0, 1.0) == 0 and oracle.classify(0.0, 0.0) == 0
    assert oracle.classify(1.0, -1.0) == 1 and oracle.classify(-1.0, 1.0) == 1
    assert oracle.classify(0.0, 1.0) == 2 and oracle.classify(0.0, -1.0) == 2
    assert oracle.classify(1.0, 0.0) == 3


def test_diagnose_hand_cases(oracle_lib):
    """beta1 = 0 makes c = g exactly.  Element by element (W = 3):
    (2, 2, 2)    votes +3, sum +6  -> match
    (-3, 1, 1)   votes +1, sum -1  -> flip (majority disagrees with the sum)
    (3, -1, 0)   t = 1: zero sends -1, votes -1, sum +2 -> flip
    (1, -1, 0)   t = 1: votes -1, sum 0 -> spurious
    and W = 2: (3, -1) votes 0 (tie), sum +2 -> dropped."""
    g3 = [np.array(v, np.float32) for v in ([2, -3, 3, 1], [2, 1, -1, -1], [2, 1, 0, 0])]
    m3 = [np.array([0, 0, 0, 0], np.float32), np.array([1, 0, 0, 0], np.float32),
          np.array([3, 0, 0, 0], np.float32)]
    r = oracle.diagnose(d=4, W=3, layout=None, beta1=0.0, mode=oracle.MODE_SIGN, nbits=1, flags=0, t=1,
                        grads=g3, m=m3)[0]
    assert (r["match"], r["flip"], r["dropped"], r["spurious"], r["ties"]) == (1, 2, 0, 1, 0)
    # momentum std of element 0 over workers: values (0, 1, 3): mean 4/3
    assert r["max_std_m"] == oracle.worker_std([0.0, 1.0, 3.0])
    g2 = [np.array([3], np.float32), np.array([-1], np.float32)]
    m2 = [np.zeros(1, np.float32), np.zeros(1, np.float32)]
    r = oracle.diagnose(d=1, W=2, layout=None, beta1=0.0, mode=oracle.MODE_SIGN, nbits=1, flags=0, t=0,
                        grads=g2, m=m2)[0]
    assert (r["match"], r["flip"], r["dropped"], r["spurious"], r["ties"]) == (0, 0, 1, 0, 1)
    # with the alternating tie rule the tie at even t becomes +1: a match
    r = oracle.diagnose(d=1, W=2, layout=None, beta1=0.0, mode=oracle.MODE_SIGN, nbits=1,
                        flags=oracle.FLAG_TIE_ALTERNATE, t=0, grads=g2, m=m2)[0]
    assert (r["match"], r["dropped"], r["ties"]) == (1, 0, 1)


def test_diagnose_max_std_is_a_maximum_per_tensor(oracle_lib):
    """Two workers, m0 = 0 and m1 = (1, 4, 2 | 6, 0): the per-element std is
    |m1| / 2, so the per-tensor maxima are 2 (second element, not the first)
    and 3."""
    m = [np.zeros(5, np.float32), np.array([1, 4, 2, 6, 0], np.float32)]
    g = [np.zeros(5, np.float32), np.zeros(5, np.float32)]
    rs = oracle.diagnose(d=5, W=2, layout=[(0, 3, 0), (3, 2, 0)], beta1=0.9, mode=oracle.MODE_SIGN, nbits=1,
                         flags=0, t=0, grads=g, m=m)
    assert [r["max_std_m"] for r in rs] == [2.0, 3.0]


def test_diagnose_l1_uses_q1_codes(oracle_lib):
    """Two workers, the golden two-worker Q1 case: agg = [9,-4,-1,-1,-4,9]
    against the full-precision sums [1001,-2,-397,296,-200,110]."""
    g = _golden_q1()["two_workers"]
    grads = [np.array(g["c0"], np.float32), np.array(g["c1"], np.float32)]
    m = [np.zeros(6, np.float32), np.zeros(6, np.float32)]
    r = oracle.diagnose(d=6, W=2, layout=None, beta1=0.0, mode=oracle.MODE_L1, nbits=4, flags=0, t=0,
                        grads=grads, m=m)[0]
    # signs: agg (+,-,-,-,-,+) vs sums (+,-,-,+,-,+): one flip (element 3)
    assert (r["match"], r["flip"], r["dropped"], r["spurious"], r["ties"]) == (5, 1, 0, 0, 0)
    assert r["max_std_m"] == 0.0


def test_diagnose_single_worker_and_partition(oracle_lib):
    rng = np.random.default_rng(12)
    layout = [(0, 64, 0), (64, 96, 0), (160, 7, 0)]
    d = 167
    grads = [(rng.standard_normal(d) * 1e-3).astype(np.float32)]
    m = [(rng.standard_normal(d) * 1e-3).astype(np.float32)]
    rs = oracle.diagnose(d=d, W=1, layout=layout, beta1=0.9, mode=oracle.MODE_SIGN, nbits=1, flags=0, t=0,
                         grads=grads, m=m)
    for r, (_, n, _) in zip(rs, layout):
        assert r["match"] == n and r["max_std_m"] == 0.0  # one worker: the vote is its own sign
    W = 4
    grads = [(rng.standard_t(3.0, d) * 1e-3).astype(np.float32) for _ in range(W)]
    m = [(rng.standard_normal(d) * 1e-3).astype(np.float32) for _ in range(W)]
    for mode, nbits in ((oracle.MODE_SIGN, 1), (oracle.MODE_L1, 2)):
        rs = oracle.diagnose(d=d, W=W, layout=layout, beta1=0.9, mode=mode, nbits=nbits, flags=0, t=3,
                             grads=grads, m=m)
        for r, (_, n, _) in zip(rs, layout):
            assert r["match"] + r["flip"] + r["dropped"] + r["spurious"] == n
            assert r["ties"] >= r["dropped"]


def test_diagnose_tie_rate_statistics(oracle_lib):
    """Dropped updates at step 0 (m = 0, symmetric i.i.d. gradients) are the
    tied votes: C(W, W/2) / 2^W of the elements."""
    rng = np.random.default_rng(31)
    d = 20000
    for W in (4, 8):
        grads = [(rng.standard_t(3.0, d) * 1e-3).astype(np.float32) for _ in range(W)]
        m = [np.zeros(d, np.float32) for _ in range(W)]
        r = oracle.diagnose(d=d, W=W, layout=None, beta1=0.9, mode=oracle.MODE_SIGN, nbits=1, flags=0, t=0,
                            grads=grads, m=m)[0]
        p = math.comb(W, W // 2) / 2 ** W
        assert abs(r["ties"] / d - p) < 5 * math.sqrt(p * (1 - p) / d)
        assert r["dropped"] == r["ties"]  # a tie is never a full-precision zero here
        assert r["match"] > r["flip"]     # the majority usually agrees with the sum


# ---------------------------------------------------------------------------
# Q_inf: max-norm scaling with stochastic rounding, the comparator of the
# diagnostics ("Lion Cub" page, "Core claim" and the Fig. 4 caption: Q_inf
# turns most of the heavy-tailed update into zero codes)
# ---------------------------------------------------------------------------

def test_splitmix64_published_outputs(oracle_lib):
    with open(os.path.join(GOLDEN, "splitmix64_vectors.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        want = case.get("outputs") or [int(h, 16) for h in case["outputs_hex"]]
        got = [oracle.splitmix64(case["seed"], k) for k in range(len(want))]
        assert got == want, case


def test_qinf_uniform_range_and_counter(oracle_lib):
    us = [oracle.qinf_uniform(5, 3, 2, e) for e in range(4000)]
    assert all(0.0 <= u < 1.0 for u in us)
    assert all(u * 16777216.0 == int(u * 16777216.0) for u in us)  # 24-bit grid
    assert abs(np.mean(us) - 0.5) < 5 * math.sqrt(1 / 12 / len(us))
    # step, worker and element each select another output of the generator
    base = oracle.qinf_uniform(5, 3, 2, 7)
    assert oracle.qinf_uniform(5, 3, 2, 7) == base
    assert len({base, oracle.qinf_uniform(5, 4, 2, 7), oracle.qinf_uniform(5, 3, 1, 7),
                oracle.qinf_uniform(5, 3, 2, 8), oracle.qinf_uniform(6, 3, 2, 7)}) == 5
    # the counter: (t mod 2^16) * 2^48 + worker * 2^40 + e, top 24 bits of the output
    k = (3 << 48) | (2 << 40) | 7
    assert base == (oracle.splitmix64(5, k) >> 40) / 16777216.0
    assert oracle.qinf_uniform(5, 3 + 65536, 2, 7) == base


def test_qinf_deterministic_cases(oracle_lib):
    # power-of-two max-norm: the scale qmax / M_inf is exact, so whole-number
    # y = qmax |c| / M_inf are exact and rounding has nothing to decide
    c = np.array([4.0, -4.0, 2.0, -1.0, 0.0, -0.0], np.float32)
    for seed in (0, 1, 99):
        q = oracle.qinf(c, 2, seed=seed, t=0, worker=0)        # qmax = 1, y = [1, 1, .5, .25, 0, 0]
        assert q[0] == 1 and q[1] == -1 and q[4] == 0 and q[5] == 0
        assert q[2] in (0, 1) and q[3] in (0, -1)
        q8 = oracle.qinf(np.array([8.0, -6.0, 2.0, 0.0], np.float32), 4, seed=seed, t=1, worker=3)  # inv = 7/8
        assert list(q8[[0, 3]]) == [7, 0] and q8[1] in (-5, -6) and q8[2] in (1, 2)
    # every |c| equal: each code is +-qmax whatever the draw
    c = np.where(np.arange(1000) % 3 == 0, -0.25, 0.25).astype(np.float32)
    for n in (2, 4, 8):
        q = oracle.qinf(c, n, seed=7, t=2, worker=1)
        qmax = (1 << (n - 1)) - 1
        assert np.array_equal(q, np.where(c < 0, -qmax, qmax))
    # an all-zero tensor (M_inf = 0) gives zero codes
    assert not oracle.qinf(np.zeros(64, np.float32), 4, seed=1, t=0, worker=0).any()
    assert oracle.maxabs(np.array([0.5, -3.0, 2.0], np.float32)) == 3.0


def test_qinf_is_unbiased_stochastic_rounding(oracle_lib):
    # 200,000 copies of 0.3 next to one 1.0: y = RN(0.3 * 7) = 2.1 (n = 4);
    # codes are 2 or 3, and their mean is y within the binomial error (a
    # floor, a round-to-nearest or a draw compared the wrong way fails)
    n = 200_001
    c = np.full(n, 0.3, np.float32)
    c[0] = 1.0
    q = oracle.qinf(c, 4, seed=11, t=0, worker=0)[1:].astype(np.float64)
    y = float(np.float32(np.float32(0.3) * np.float32(7.0)))
    frac = y - math.floor(y)
    assert set(np.unique(q)) <= {2.0, 3.0}
    assert abs(q.mean() - y) < 5 * math.sqrt(frac * (1 - frac) / q.size)
    # negative values mirror
    qn = oracle.qinf(-c, 4, seed=11, t=0, worker=0)[1:].astype(np.float64)
    assert abs(qn.mean() + y) < 5 * math.sqrt(frac * (1 - frac) / q.size)


def test_qinf_collapses_heavy_tails_where_q1_does_not(oracle_lib):
    # the pages' observation, on Student-t(3) values: most Q_inf codes are 0,
    # while most Eq. (1) codes are not
    rng = np.random.default_rng(3)
    x = (rng.standard_t(3.0, size=1 << 18) * 1e-3).astype(np.float32)
    for n in (2, 4):
        zq = np.mean(oracle.qinf(x, n, seed=2, t=0, worker=0) == 0)
        z1 = np.mean(oracle.q1(x, n) == 0)
        assert zq > 0.8 and z1 < zq, (n, zq, z1)
    assert np.mean(oracle.q1(x, 4) == 0) < 0.5


def test_diagnose_qinf_hand_case(oracle_lib):
    # beta1 = 0 so c = g; two workers, one tensor of 4 elements, n = 2
    # worker 0: [4, -4, 2, 0] (M_inf 4: codes 1, -1, 0 or 1, 0)
    # worker 1: [1, -1, -1, 0] (M_inf 1: codes 1, -1, -1, 0)
    g0 = np.array([4, -4, 2, 0], np.float32)
    g1 = np.array([1, -1, -1, 0], np.float32)
    m = [np.zeros(4, np.float32), np.zeros(4, np.float32)]
    for seed in range(8):
        r = oracle.diagnose_qinf(d=4, W=2, layout=None, beta1=0.0, nbits=2, flags=0, t=0, seed=seed, e_base=0,
                                 grads=[g0, g1], m=m)[0]
        q02 = oracle.qinf(g0, 2, seed=seed, t=0, worker=0)[2]
        # e0: 1 + 1 = 2, s = 5 -> match; e1: -2, s = -5 -> match; e3: 0, s = 0 -> match
        # e2: q02 - 1 (0 or -1) against s = 1 -> dropped or flip
        want = {"match": 3, "flip": 1 if q02 == 0 else 0, "dropped": 1 if q02 == 1 else 0, "spurious": 0}
        assert {f: r[f] for f in want} == want, (seed, r)
        assert r["zero_codes"] == 2 + (1 if q02 == 0 else 0)
    # the element index is global: the same tensor at another flat offset draws other numbers
    r_off = [oracle.diagnose_qinf(d=4, W=2, layout=None, beta1=0.0, nbits=2, flags=0, t=0, seed=s, e_base=1 << 20,
                                  grads=[g0, g1], m=m)[0]["flip"] for s in range(32)]
    r_0 = [oracle.diagnose_qinf(d=4, W=2, layout=None, beta1=0.0, nbits=2, flags=0, t=0, seed=s, e_base=0,
                                grads=[g0, g1], m=m)[0]["flip"] for s in range(32)]
    assert r_off != r_0


def test_diagnose_qinf_partitions_each_tensor(oracle_lib):
    rng = np.random.default_rng(4)
    d, W = 3000, 4
    layout = [(0, 1000, 0), (1000, 1968, 0), (2968, 32, 0)]
    grads = [(rng.standard_t(3.0, d) * 1e-3).astype(np.float32) for _ in range(W)]
    m = [(rng.standard_normal(d) * 1e-4).astype(np.float32) for _ in range(W)]
    recs = oracle.diagnose_qinf(d=d, W=W, layout=layout, beta1=0.9, nbits=4, flags=0, t=5, seed=9, e_base=0,
                                grads=grads, m=m)
    for (off, n, _), r in zip(layout, recs):
        assert r["match"] + r["flip"] + r["dropped"] + r["spurious"] == n
        assert 0 <= r["zero_codes"] <= W * n
        # a tensor on its own, given its flat offset, gives the same record
        one = oracle.diagnose_qinf(d=n, W=W, layout=None, beta1=0.9, nbits=4, flags=0, t=5, seed=9, e_base=off,
                                   grads=[g[off:off + n].copy() for g in grads],
                                   m=[x[off:off + n].copy() for x in m])[0]
        assert one == r
