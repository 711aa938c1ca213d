"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: values decoded or
computed by hand (``tests/golden``), torch's own E4M3 conversion, an exact integer dot,
a special case that collapses to one numpy matrix product, and invariants that the
formula of ROCm/aiter PR #7183 ("Motivation") implies.  The last test compiles
deliberately broken copies of the oracle and checks that these pins reject every one.
"""
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _hex(a):
    return np.array([[int(x, 16) for x in row] for row in a], dtype=np.uint8) \
        if isinstance(a[0], list) and not isinstance(a[0][0], list) else \
        np.array([[[int(x, 16) for x in r] for r in m] for m in a], dtype=np.uint8)


def _lib_arg(lib):
    return {} if lib is None else {"lib": lib}


# ---------------------------------------------------------------- E4M3 decode pins
def check_e4m3_vs_torch(lib=None):
    table = oracle.e4m3_table(lib)
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(table) & np.isnan(ref)
    assert np.all(both_nan | (table == ref))
    assert np.array_equal(np.signbit(table), np.signbit(ref))


def check_e4m3_hand_codes(lib=None):
    table = oracle.e4m3_table(lib)
    fx = json.load(open(os.path.join(GOLDEN, "e4m3_codes.json")))
    for code, val in fx["codes"]:
        got = table[int(code, 16)]
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val), (code, got, val)
            assert math.copysign(1.0, got) == math.copysign(1.0, float(val)), code


def test_e4m3_table_matches_torch():
    check_e4m3_vs_torch()


def test_e4m3_hand_decoded_codes():
    check_e4m3_hand_codes()


# ---------------------------------------------------------------- hand-computed cases
def _golden_cases():
    fx = json.load(open(os.path.join(GOLDEN, "hand_cases.json")))
    byname = {c["name"]: c for c in fx["cases"]}
    out = []
    for c in fx["cases"]:
        base = byname[c.get("same_inputs_as", c["name"])]
        merged = dict(base)
        merged.update({k: v for k, v in c.items() if k != "same_inputs_as"})
        out.append(merged)
    return out


def check_golden(lib=None):
    for c in _golden_cases():
        q = _hex(c["q"])
        k = _hex(c["k"])
        w = np.array(c["w"], np.float32)
        kv = np.array(c["kv_scale"], np.float32)
        ks = np.array(c["ks"], np.int32)
        ke = np.array(c["ke"], np.int32)
        poison = float("nan")
        init = np.full((c["M"], c["N"]), poison)
        got = oracle.fp8_mqa_logits(q, k, kv, w, ks, ke, c["clean_logits"], out=init,
                                    **_lib_arg(lib))
        for m, row in enumerate(c["expected"]):
            for n, e in enumerate(row):
                g = got[m, n]
                if e == "poison":
                    assert math.isnan(g), (c["name"], m, n, g)
                elif e == "-inf":
                    assert g == -math.inf, (c["name"], m, n, g)
                else:
                    assert g == float(e), (c["name"], m, n, g, e)


def test_golden_hand_cases():
    check_golden()


# ---------------------------------------------------------------- closed forms
ONE, MINUS_ONE = 0x38, 0xB8


def check_all_ones(lib=None):
    M, N, H, D = 5, 7, 3, 16
    rng = np.random.default_rng(1)
    q = np.full((M, H, D), ONE, np.uint8)
    k = np.full((N, D), ONE, np.uint8)
    w = rng.standard_normal((M, H)).astype(np.float32)
    kv = rng.uniform(0.5, 2, N).astype(np.float32)
    ks = np.zeros(M, np.int32)
    ke = np.full(M, N, np.int32)
    got = oracle.fp8_mqa_logits(q, k, kv, w, ks, ke, 1, **_lib_arg(lib))
    # every dot is D; relu(D) = D; out = D * sum_h w[m,h] * kv[n]
    want = D * w.astype(np.float64).sum(1)[:, None] * kv.astype(np.float64)[None, :]
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=0)


def check_negative_dots_vanish(lib=None):
    M, N, H, D = 3, 4, 2, 8
    q = np.full((M, H, D), MINUS_ONE, np.uint8)
    k = np.full((N, D), ONE, np.uint8)
    w = np.array([[1.0, -2.0], [3.0, 0.5], [-1.0, -1.0]], np.float32)
    kv = np.array([1.0, 2.0, 0.5, 1.5], np.float32)
    got = oracle.fp8_mqa_logits(q, k, kv, w, np.zeros(M, np.int32), np.full(M, N, np.int32),
                                1, **_lib_arg(lib))
    assert np.all(got == 0.0)


def check_one_hot(lib=None):
    # Q[m,h,:] is x at position a(m,h), K[n,:] is y at position b(n): the dot is x*y
    # when a == b, else 0.  Values chosen so every product is an exact binary fraction.
    M, N, H, D = 2, 3, 2, 8
    q = np.zeros((M, H, D), np.uint8)
    k = np.zeros((N, D), np.uint8)
    q[0, 0, 1] = 0x40  # 2
    q[0, 1, 5] = 0x3C  # 1.5
    q[1, 0, 5] = 0x30  # 0.5
    q[1, 1, 1] = 0xC4  # -3
    k[0, 1] = 0x38     # 1
    k[1, 5] = 0x40     # 2
    k[2, 3] = 0x7E     # 448 (no query touches d=3)
    w = np.array([[0.5, 2.0], [4.0, 1.0]], np.float32)
    kv = np.array([1.0, 0.25, 3.0], np.float32)
    got = oracle.fp8_mqa_logits(q, k, kv, w, np.zeros(M, np.int32), np.full(M, N, np.int32),
                                1, **_lib_arg(lib))
    want = np.array([
        [2 * 1 * 0.5 * 1.0, 1.5 * 2 * 2.0 * 0.25, 0.0],
        [0.0,               0.5 * 2 * 4.0 * 0.25, 0.0],  # head 1 of row 1: -3*1 -> relu 0
    ])
    assert np.array_equal(got, want), got


def test_all_ones_closed_form():
    check_all_ones()


def test_negative_dots_vanish():
    check_negative_dots_vanish()


def test_one_hot_products():
    check_one_hot()


# ---------------------------------------------------------------- exact integer dot
def _finite_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    return np.where((c & 0x7F) == 0x7F, c & 0xF8, c).astype(np.uint8)  # drop NaN codes


def check_exact_int_dot(lib=None):
    # H=1, w=1, kv=1: out = relu(dot) exactly, because the fp64 dot of E4M3 values is
    # exact.  The integer side decodes with torch (value * 2^9 is an integer) and sums
    # in int64, so it shares nothing with the oracle's arithmetic.
    rng = np.random.default_rng(7)
    M, N, D = 6, 9, 128
    q = _finite_codes(rng, (M, 1, D))
    k = _finite_codes(rng, (N, D))

    def ints(codes):
        v = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64) * 512.0
        iv = v.numpy()
        assert np.all(iv == np.round(iv))
        return iv.astype(np.int64)

    qi, ki = ints(q[:, 0, :]), ints(k)
    dot = qi @ ki.T  # int64, exact; true dot = dot * 2^-18
    want = np.maximum(dot, 0).astype(np.float64) * 2.0 ** -18
    got = oracle.fp8_mqa_logits(q, k, np.ones(N, np.float32), np.ones((M, 1), np.float32),
                                np.zeros(M, np.int32), np.full(M, N, np.int32), 1,
                                **_lib_arg(lib))
    assert np.array_equal(got, want)


def test_exact_integer_dot():
    check_exact_int_dot()


# ---------------------------------------------------------------- reduction to a matmul
def check_positive_is_matmul(lib=None):
    # With Q, K >= 0 every dot is >= 0, relu is the identity, and the formula collapses
    # to kv[n] * ((sum_h w[m,h] Q[m,h,:]) @ K[n,:]) -- one numpy matrix product with the
    # head sum moved inside.  A transposed operand, a wrong index or a dropped factor
    # changes this value.
    rng = np.random.default_rng(11)
    M, N, H, D = 7, 13, 5, 32
    q = _finite_codes(rng, (M, H, D)) & 0x7F
    k = _finite_codes(rng, (N, D)) & 0x7F
    w = rng.standard_normal((M, H)).astype(np.float32)
    kv = rng.uniform(0.5, 2, N).astype(np.float32)
    qf = torch.from_numpy(q.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    kf = torch.from_numpy(k.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    qw = np.einsum("mhd,mh->md", qf, w.astype(np.float64))
    want = (qw @ kf.T) * kv.astype(np.float64)[None, :]
    got = oracle.fp8_mqa_logits(q, k, kv, w, np.zeros(M, np.int32), np.full(M, N, np.int32),
                                1, **_lib_arg(lib))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_positive_inputs_reduce_to_matmul():
    check_positive_is_matmul()


# ---------------------------------------------------------------- invariants
def _rand_inputs(seed, M=6, N=40, H=4, D=16):
    rng = np.random.default_rng(seed)
    q = _finite_codes(rng, (M, H, D))
    k = _finite_codes(rng, (N, D))
    w = rng.standard_normal((M, H)).astype(np.float32)
    kv = rng.uniform(0.5, 2, N).astype(np.float32)
    ks = rng.integers(-3, N, M).astype(np.int32)
    ke = (ks + rng.integers(-2, N, M)).astype(np.int32)
    return q, k, kv, w, ks, ke


def check_mask_exact(lib=None):
    for seed in range(4):
        q, k, kv, w, ks, ke = _rand_inputs(seed)
        M, N = q.shape[0], k.shape[0]
        got = oracle.fp8_mqa_logits(q, k, kv, w, ks, ke, 1, **_lib_arg(lib))
        n = np.arange(N)[None, :]
        inside = (n >= np.clip(ks, 0, N)[:, None]) & (n < np.clip(ke, 0, N)[:, None])
        assert np.all(np.isneginf(got) == ~inside)
        assert np.all(np.isfinite(got[inside]))
        poison = np.full((M, N), 12345.5)
        got0 = oracle.fp8_mqa_logits(q, k, kv, w, ks, ke, 0, out=poison.copy(),
                                     **_lib_arg(lib))
        assert np.all(got0[~inside] == 12345.5)
        assert np.array_equal(got0[inside], got[inside])


def check_linear_in_w(lib=None):
    q, k, kv, _, ks, ke = _rand_inputs(21)
    M, H = q.shape[0], q.shape[1]
    rng = np.random.default_rng(5)
    w1 = rng.integers(-8, 9, (M, H)).astype(np.float32) / 4
    w2 = rng.integers(-8, 9, (M, H)).astype(np.float32) / 4
    a, b = 2.0, -0.5
    o1 = oracle.fp8_mqa_logits(q, k, kv, w1, ks, ke, 1, **_lib_arg(lib))
    o2 = oracle.fp8_mqa_logits(q, k, kv, w2, ks, ke, 1, **_lib_arg(lib))
    o12 = oracle.fp8_mqa_logits(q, k, kv, (a * w1 + b * w2).astype(np.float32), ks, ke, 1,
                                **_lib_arg(lib))
    fin = np.isfinite(o12)
    np.testing.assert_allclose(o12[fin], a * o1[fin] + b * o2[fin], rtol=1e-12, atol=1e-9)


def check_linear_in_kv(lib=None):
    q, k, kv, w, ks, ke = _rand_inputs(22)
    N = k.shape[0]
    scale = np.linspace(-2, 3, N).astype(np.float32)
    o1 = oracle.fp8_mqa_logits(q, k, kv, w, ks, ke, 1, **_lib_arg(lib))
    o2 = oracle.fp8_mqa_logits(q, k, (kv * scale).astype(np.float32), w, ks, ke, 1,
                               **_lib_arg(lib))
    fin = np.isfinite(o1)
    ratio = (kv * scale).astype(np.float64) / kv.astype(np.float64)
    np.testing.assert_allclose(o2[fin], (o1 * ratio[None, :])[fin], rtol=1e-12, atol=1e-9)


def check_nonneg(lib=None):
    q, k, kv, w, ks, ke = _rand_inputs(23)
    got = oracle.fp8_mqa_logits(q, k, kv, np.abs(w), ks, ke, 1, **_lib_arg(lib))
    fin = np.isfinite(got)
    assert np.all(got[fin] >= 0)
    assert np.any(got[fin] > 0)


def check_head_permutation(lib=None):
    q, k, kv, w, ks, ke = _rand_inputs(24)
    perm = np.random.default_rng(3).permutation(q.shape[1])
    o1 = oracle.fp8_mqa_logits(q, k, kv, w, ks, ke, 1, **_lib_arg(lib))
    o2 = oracle.fp8_mqa_logits(q[:, perm], k, kv, w[:, perm], ks, ke, 1, **_lib_arg(lib))
    fin = np.isfinite(o1)
    assert np.array_equal(np.isfinite(o2), fin)
    np.testing.assert_allclose(o2[fin], o1[fin], rtol=1e-13, atol=1e-12)


def check_independence(lib=None):
    # Rows are independent of other rows; keys outside a row's window do not change
    # in-window values; the row-subset entry point matches the full computation.
    q, k, kv, w, ks, ke = _rand_inputs(25)
    M, N = q.shape[0], k.shape[0]
    full = oracle.fp8_mqa_logits(q, k, kv, w, ks, ke, 1, **_lib_arg(lib))
    rows = np.array([4, 0, 5], np.int64)
    sub = oracle.fp8_mqa_logits(q, k, kv, w, ks, ke, 1, rows=rows, **_lib_arg(lib))
    assert np.array_equal(sub, full[rows], equal_nan=True)
    # append 9 random keys at the end: rows whose windows end before N are unchanged
    rng = np.random.default_rng(9)
    k2 = np.concatenate([k, _finite_codes(rng, (9, k.shape[1]))])
    kv2 = np.concatenate([kv, rng.uniform(0.5, 2, 9).astype(np.float32)])
    ke2 = np.minimum(ke, N).astype(np.int32)
    wide = oracle.fp8_mqa_logits(q, k2, kv2, w, ks, ke2, 1, **_lib_arg(lib))
    assert np.array_equal(wide[:, :N], full, equal_nan=True)
    assert np.all(np.isneginf(wide[:, N:]))
    # a single row computed alone equals that row of the batch
    one = oracle.fp8_mqa_logits(q[3:4], k, kv, w[3:4], ks[3:4], ke[3:4], 1, **_lib_arg(lib))
    assert np.array_equal(one[0], full[3], equal_nan=True)


def test_mask_exact_and_clean0_untouched():
    check_mask_exact()


def test_linear_in_w():
    check_linear_in_w()


def test_linear_in_kv_scale():
    check_linear_in_kv()


def test_nonnegative_for_nonnegative_w():
    check_nonneg()


def test_head_permutation_invariance():
    check_head_permutation()


def test_row_and_key_independence():
    check_independence()


def test_workload_windows_shapes():
    # the benchmark windows are the documented ones (pins the input recipe, not the oracle)
    ks, ke = workloads.windows("causal", 8192, 8192)
    assert ks[0] == 0 and ke[0] == 1 and ke[-1] == 8192
    ks, ke = workloads.windows("causal", 4096, 32768)
    assert ke[0] == 28672 + 1 and ke[-1] == 32768
    ks, ke = workloads.windows("causal", 1024, 131072)
    assert ke[0] == 130048 + 1
    ks, ke = workloads.windows("multi_req", 4096, 32768, 4)
    r, i = 2, 17
    assert ks[1024 * r + i] == 8192 * r and ke[1024 * r + i] == 8192 * r + 7168 + i + 1
    assert workloads.valid_pairs(*workloads.windows("causal", 8192, 8192), 8192) == 33558528


# ---------------------------------------------------------------- the pins have teeth
ALL_PINS = [check_e4m3_vs_torch, check_e4m3_hand_codes, check_golden, check_all_ones,
            check_negative_dots_vanish, check_one_hot, check_exact_int_dot,
            check_positive_is_matmul, check_mask_exact, check_linear_in_w,
            check_linear_in_kv, check_nonneg, check_head_permutation, check_independence]

# Plausible mistakes, planted into a temporary copy of the oracle source.
MUTANTS = {
    "no_relu": ("double r = dot > 0.0 ? dot : 0.0;", "double r = dot;"),
    "relu_after_w": ("acc += r * (double)j->w[(size_t)m * H + h];",
                     "acc += (dot * (double)j->w[(size_t)m * H + h] > 0.0 ? "
                     "dot * (double)j->w[(size_t)m * H + h] : 0.0);"),
    "w_transposed": ("(double)j->w[(size_t)m * H + h]", "(double)j->w[(size_t)h * j->M + m]"),
    "kv_by_row": ("acc * (double)j->kv_scale[n]", "acc * (double)j->kv_scale[m % N]"),
    "kv_dropped": ("out_row[n] = acc * (double)j->kv_scale[n];", "out_row[n] = acc;"),
    "k_transposed": ("const uint8_t* kv = j->k + (size_t)n * D;",
                     "const uint8_t* kv = j->k + (size_t)n;"),
    "q_head_index": ("const uint8_t* qv = j->q + ((size_t)m * H + h) * D;",
                     "const uint8_t* qv = j->q + ((size_t)h * j->M + m) * D;"),
    "window_closed": ("if (n < lo || n >= hi) {", "if (n < lo || n > hi) {"),
    "window_open_start": ("if (n < lo || n >= hi) {", "if (n <= lo || n >= hi) {"),
    "exp_bias_8": ("ldexp(1.0 + (double)man / 8.0, exp - 7)", "ldexp(1.0 + (double)man / 8.0, exp - 8)"),
    "subnormal_wrong": ("ldexp((double)man / 8.0, 1 - 7)", "ldexp((double)man / 8.0, -7)"),
    "last_head_dropped": ("for (int32_t h = 0; h < H; ++h) {", "for (int32_t h = 0; h < H - 1; ++h) {"),
    "clean0_writes": ("continue;                             /* clean = 0: untouched */",
                      "out_row[n] = 0.0; continue;"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.source_path()).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / f"libmutant_{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread", "-o", str(so),
                    str(mut), "-lm"], check=True)
    lib = oracle.bind(str(so))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
