"""Sensitivity of the oracle's pins: each case plants one plausible mistake
in a copy of the oracle's C source (on the CPU, in a temporary directory),
builds it, and runs the pin suite (tests/test_oracle_pins.py) against that
copy; at least one pin must fail.  The unmodified copy, built the same way,
must pass.  This checks that the pins constrain every step of the oracle --
a dropped term, a wrong sign, a swapped operand, an off-by-one -- and not
only the cases they were written for.

Not listed: computing omega = 1 - beta in double before rounding to fp32.
For beta in [0.5, 1] the fp32 subtraction is exact (Sterbenz), so that
change is equivalent, not a mistake.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "lioncub_oracle.c")
HDR = os.path.join(ROOT, "oracle", "lioncub_oracle.h")
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

# (name, original text, planted mistake); the original occurs exactly once.
MUTATIONS = [
    ("update_vector_operands_swapped", "float a = beta1 * m;\n    float b = omega1 * g;",
     "float a = omega1 * m;\n    float b = beta1 * g;"),
    ("momentum_from_m_not_g", "float b = omega2 * g;", "float b = omega2 * m;"),
    ("zero_sign_parity_flipped", "return (t % 2 == 0) ? 1 : 0;", "return (t % 2 == 0) ? 0 : 1;"),
    ("packing_msb_first", "words[e / 32] |= bit << (e % 32);", "words[e / 32] |= bit << (31 - e % 32);"),
    ("m1_without_abs", "s += fabs((double)c[e]);", "s += (double)c[e];"),
    ("m1_without_division", "return (float)(s / (double)n);", "return (float)s;"),
    ("q1_scale_inverted", "float inv = qmax / m1;", "float inv = m1 / qmax;"),
    ("q1_round_half_away", "float r = rintf(y);", "float r = roundf(y);"),
    ("q1_round_toward_zero", "float r = rintf(y);", "float r = truncf(y);"),
    ("q1_clamp_admits_minus_2_pow", "if (r < -qmax)\n            r = -qmax;",
     "if (r < -qmax - 1.0f)\n            r = -qmax - 1.0f;"),
    ("codes_field_mask_one_bit_short", "uint32_t field = (uint32_t)(int32_t)q[e] & mask;",
     "uint32_t field = (uint32_t)(int32_t)q[e] & (mask >> 1);"),
    ("vote_counts_zeros_as_nothing", "s += bit ? 1 : -1;", "s += bit ? 1 : 0;"),
    ("code_sum_sign_extension_wrong", "f -= 2 * half;", "f -= half;"),
    ("tie_gives_plus_one", "        return (t % 2 == 0) ? 1.0f : -1.0f;\n    return 0.0f;",
     "        return (t % 2 == 0) ? 1.0f : -1.0f;\n    return 1.0f;"),
    ("tie_alternation_flipped", "return (t % 2 == 0) ? 1.0f : -1.0f;", "return (t % 2 == 0) ? -1.0f : 1.0f;"),
    ("average_without_division", "return (float)agg / (float)W;", "return (float)agg;"),
    ("weight_decay_sign", "float b = u + a;", "float b = u - a;"),
    ("apply_adds_step", "return theta - c;", "return theta + c;"),
    ("sync_average_without_division", "float avg = s / (float)W;", "float avg = s;"),
    ("sync_average_skips_worker_0", "float s = m[0][e];\n        for (int j = 1; j < W; ++j)",
     "float s = 0.0f;\n        for (int j = 1; j < W; ++j)"),
    ("sync_one_step_early", "(t + 1) % sync_interval == 0", "t % sync_interval == 0"),
    ("bf16_widening_wrong", "uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;"),
    # the step's orchestration
    ("vote_skips_last_worker", "    for (int i = 0; i < W; ++i) {\n        uint32_t bit = (words[i][e / 32]",
     "    for (int i = 0; i < W - 1; ++i) {\n        uint32_t bit = (words[i][e / 32]"),
    ("code_sum_skips_last_worker", "    for (int i = 0; i < W; ++i) {\n        int32_t f =",
     "    for (int i = 0; i < W - 1; ++i) {\n        int32_t f ="),
    ("update_vector_from_worker_0_gradient", "float g = load_grad(grads[i], grad_dtype, off + e);",
     "float g = load_grad(grads[0], grad_dtype, off + e);"),
    ("momentum_from_worker_0_gradient", "m[i][e] = lco_momentum(m[i][e], load_grad(grads[i], grad_dtype, e),",
     "m[i][e] = lco_momentum(m[i][e], load_grad(grads[0], grad_dtype, e),"),
    ("m1_over_part_of_the_tensor", "float m1 = lco_m1(c, n);", "float m1 = lco_m1(c, (n + 1) / 2);"),
    # diagnostics
    ("worker_std_sample_variance", "return sqrtf(v / (float)W);", "return sqrtf(v / (float)(W - 1 > 0 ? W - 1 : 1));"),
    ("worker_std_mean_wrong", "float mean = s / (float)W;", "float mean = s / (float)(W + 1);"),
    ("classify_flip_dropped_swapped", "        return 1;\n    if (u_q == 0.0f)\n        return 2;",
     "        return 2;\n    if (u_q == 0.0f)\n        return 1;"),
    ("diagnose_full_sign_skips_worker_0", "s = (i == 0) ? ci : s + ci;", "s = (i == 0) ? 0.0f : s + ci;"),
    ("diagnose_max_std_keeps_first", "if (sd > r.max_std_m)", "if (r.max_std_m == 0.0f)"),
    # the Q_inf comparator
    ("splitmix_counter_off_by_one", "uint64_t z = seed + (k + 1u) * 0x9e3779b97f4a7c15ull;",
     "uint64_t z = seed + k * 0x9e3779b97f4a7c15ull;"),
    ("splitmix_shift_wrong", "z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;",
     "z = (z ^ (z >> 28)) * 0x94d049bb133111ebull;"),
    ("qinf_uniform_low_bits", "uint64_t bits = lco_splitmix64(seed, k) >> 40; /* 24 bits */",
     "uint64_t bits = lco_splitmix64(seed, k) & 0xffffffu; /* 24 bits */"),
    ("qinf_uniform_ignores_worker", "((uint64_t)(unsigned)worker << 40)", "((uint64_t)(unsigned)0 << 40)"),
    ("qinf_deterministic_floor", "int v = (int)fl + (u < frac ? 1 : 0);", "int v = (int)fl;"),
    ("qinf_round_up_when_draw_exceeds", "int v = (int)fl + (u < frac ? 1 : 0);", "int v = (int)fl + (u > frac ? 1 : 0);"),
    ("qinf_scale_by_first_element", "if (fabsf(c[e]) > mx)\n            mx = fabsf(c[e]);",
     "if (e == 0)\n            mx = fabsf(c[e]);"),
    ("qinf_sign_dropped", "q[e] = (int8_t)(c[e] < 0.0f ? -v : v);", "q[e] = (int8_t)v;"),
    ("qinf_local_element_index", "lco_qinf(c, n, nbits, lco_maxabs(c, n), seed, t, i, e_base + off,",
     "lco_qinf(c, n, nbits, lco_maxabs(c, n), seed, t, i, off,"),
]


def _build(tmp, text, name):
    src = os.path.join(tmp, f"{name}.c")
    with open(src, "w") as f:
        f.write(text)
    shutil.copy(HDR, os.path.join(tmp, "lioncub_oracle.h"))
    lib = os.path.join(tmp, f"lib{name}.so")
    r = subprocess.run(["gcc", *CFLAGS, "-o", lib, src, "-lm"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return lib


def _run_pins(lib):
    env = {**os.environ, "LIONCUB_ORACLE_LIB": lib}
    return subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
                           "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=600)


@pytest.fixture(scope="module")
def original():
    with open(SRC) as f:
        return f.read()


def test_unmodified_copy_passes(tmp_path, original):
    r = _run_pins(_build(str(tmp_path), original, "control"))
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,orig,mutant", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, original, name, orig, mutant):
    assert original.count(orig) == 1, f"{name}: the text to mutate must occur exactly once"
    r = _run_pins(_build(str(tmp_path), original.replace(orig, mutant), name))
    # pytest exits with 1 when tests ran and at least one failed (not 2-5:
    # interrupted, internal or usage error, nothing collected)
    assert r.returncode == 1, f"{name} survived the pins:\n{r.stdout[-1500:]}"
