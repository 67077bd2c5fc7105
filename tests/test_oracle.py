"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test is chosen so that a plausible slip in the oracle -- a wrong e4m3
exponent bias, a lost subnormal, transposed scales, a dropped bias, a wrong
k range -- fails at least one of them.  None of them re-types the oracle's
formula: they compare it with printed values, an independent decoder (torch),
exact rational arithmetic, or algebraic identities.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits_of(values):
    """bf16 bits of values that are exactly representable (checked)."""
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    back = t.float().numpy()
    assert np.array_equal(back, np.asarray(values, dtype=np.float32)), "not exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def _e4m3_code_of(v):
    """The e4m3 code of an exactly representable value, found with torch's cast."""
    t = torch.tensor(np.asarray(v, dtype=np.float32))
    c = t.to(torch.float8_e4m3fn)
    assert np.array_equal(c.float().numpy(), np.asarray(v, dtype=np.float32)), "not exact in e4m3"
    return c.view(torch.uint8).numpy()


# --------------------------------------------------------------------------- e4m3 table

def test_e4m3_anchor_values():
    """OCP E4M3FN: bias 7, 3 mantissa bits, S.1111.111 = NaN, max 448."""
    t = oracle.e4m3_table()
    anchors = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
               0x38: 1.0, 0x3F: 1.875, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0,
               0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9)}
    for code, val in anchors.items():
        assert t[code] == val, hex(code)
    assert math.copysign(1.0, t[0x00]) == 1.0
    assert t[0x80] == 0.0 and math.copysign(1.0, t[0x80]) == -1.0
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])


def test_e4m3_table_matches_independent_decoder():
    """All 256 codes against torch's float8_e4m3fn decoder."""
    t = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(t), nan)
    assert np.array_equal(t[~nan], ref[~nan])
    assert np.array_equal(np.signbit(t[~nan]), np.signbit(ref[~nan]))


def test_e4m3_table_structure():
    t = oracle.e4m3_table()
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0), "codes 0x00..0x7E must increase strictly"
    for c in range(0x7F):
        assert t[c | 0x80] == -t[c]
    # subnormal spacing 2^-9, and the first normal continues the spacing
    assert np.all(np.diff(pos[:9]) == 2.0 ** -9)
    assert len(set(t[np.isfinite(t)].tolist())) == 253  # +0 and -0 compare equal


# --------------------------------------------------------------------------- bf16

def test_bf16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_values(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_round_to_bf16_matches_torch_and_ties():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32),
        (rng.standard_normal(10_000) * 1e-39).astype(np.float32),   # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38, 1e-45], dtype=np.float32),
    ])
    got = oracle.round_to_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    # exact ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even (1.0)
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8], dtype=np.float32)
    assert list(oracle.round_to_bf16(ties)) == [0x3F80, 0x3F82]
    assert oracle.round_to_bf16(np.array([np.nan], dtype=np.float32))[0] & 0x7FC0 == 0x7FC0


# --------------------------------------------------------------------------- worked examples

def _column_split_inputs():
    g = json.load(open(os.path.join(GOLDEN, "column_split_example.json")))
    x = np.array(g["x"], dtype=np.float64)
    w_nk = np.array(g["w_inputs_by_outputs"], dtype=np.float64).T.copy()  # [N=6, K=4]
    return g, x, w_nk


def test_column_split_example_bf16():
    g, x, w = _column_split_inputs()
    y = oracle.linear(oracle.BF16, _bf16_bits_of(x), _bf16_bits_of(w), with_abs=False)
    assert np.array_equal(y, np.array(g["printed_one_device"], dtype=np.float64))
    # device halves = output columns 0..2 and 3..5 (an N split)
    y0 = oracle.linear(oracle.BF16, _bf16_bits_of(x), _bf16_bits_of(w), rows=[0, 1, 2], with_abs=False)
    y1 = oracle.linear(oracle.BF16, _bf16_bits_of(x), _bf16_bits_of(w), rows=[3, 4, 5], with_abs=False)
    assert np.array_equal(y0, np.array(g["printed_device0"], dtype=np.float64))
    assert np.array_equal(y1, np.array(g["printed_device1"], dtype=np.float64))


@pytest.mark.parametrize("pad_k", [4, 128, 256])
def test_column_split_example_fp8_scale_one(pad_k):
    g, x, w = _column_split_inputs()
    xp = np.zeros((2, pad_k)); xp[:, :4] = x
    wp = np.zeros((6, pad_k)); wp[:, :4] = w
    codes = _e4m3_code_of(wp)
    scales = np.ones((1, (pad_k + 127) // 128), dtype=np.float32)
    y = oracle.linear(oracle.FP8_B128, _bf16_bits_of(xp), codes, scales, with_abs=False)
    assert np.array_equal(y, np.array(g["printed_one_device"], dtype=np.float64))


def test_mlp_split_example_partials_are_k_ranges():
    g = json.load(open(os.path.join(GOLDEN, "mlp_split_example.json")))
    x = np.array(g["x"], dtype=np.float64)
    a = np.array(g["a"], dtype=np.float64)        # [4, 8] inputs x hidden
    b = np.array(g["b"], dtype=np.float64)        # [8, 4] hidden x outputs
    hpre = oracle.linear(oracle.BF16, _bf16_bits_of(x), _bf16_bits_of(a.T.copy()), with_abs=False)
    h = np.maximum(hpre, 0.0)                      # the example's ReLU, applied by the test
    hb, wb = _bf16_bits_of(h), _bf16_bits_of(b.T.copy())   # second linear: K = 8 hidden units
    p0 = oracle.linear(oracle.BF16, hb, wb, k_range=(0, 4), with_abs=False)
    p1 = oracle.linear(oracle.BF16, hb, wb, k_range=(4, 8), with_abs=False)
    full = oracle.linear(oracle.BF16, hb, wb, with_abs=False)
    assert np.array_equal(p0, np.array(g["printed_device0_partial"], dtype=np.float64))
    assert np.array_equal(p1, np.array(g["printed_device1_partial"], dtype=np.float64))
    assert np.array_equal(full, np.array(g["printed_all_reduce_sum"], dtype=np.float64))
    # the same split in the FP8 format (scale 1, K padded to two 128-blocks: hidden units
    # 0..3 in block 0 and 4..7 in block 1)
    hp = np.zeros((2, 256)); hp[:, 0:4] = h[:, 0:4]; hp[:, 128:132] = h[:, 4:8]
    wp = np.zeros((4, 256)); wp[:, 0:4] = b.T[:, 0:4]; wp[:, 128:132] = b.T[:, 4:8]
    sc = np.ones((1, 2), dtype=np.float32)
    q = _e4m3_code_of(wp)
    f0 = oracle.linear(oracle.FP8_B128, _bf16_bits_of(hp), q, sc, k_range=(0, 128), with_abs=False)
    f1 = oracle.linear(oracle.FP8_B128, _bf16_bits_of(hp), q, sc, k_range=(128, 256), with_abs=False)
    assert np.array_equal(f0, np.array(g["printed_device0_partial"], dtype=np.float64))
    assert np.array_equal(f1, np.array(g["printed_device1_partial"], dtype=np.float64))


# --------------------------------------------------------------------------- structure pins

def test_one_hot_selects_weight_column_bf16_with_bias():
    rng = np.random.default_rng(1)
    N, K = 37, 96
    w = torch.randn(N, K, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    bias = torch.randn(N, generator=torch.Generator().manual_seed(4)).mul(0.01).to(torch.bfloat16)
    wbits = w.view(torch.int16).numpy().view(np.uint16)
    bbits = bias.view(torch.int16).numpy().view(np.uint16)
    for k0 in [0, 1, 50, K - 1]:
        x = np.zeros((1, K)); x[0, k0] = 1.0
        y = oracle.linear(oracle.BF16, _bf16_bits_of(x), wbits, bias_bits=bbits, with_abs=False)
        exact = w[:, k0].double().numpy() + bias.double().numpy()
        assert np.array_equal(y[0], exact)
    assert rng is not None


def test_one_hot_fp8_all_codes_and_scale_orientation():
    """N = 256 rows take the 256 codes at k0; scales differ per (n-block, k-block)."""
    K = 256
    codes = np.zeros((256, K), dtype=np.uint8)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    scales = np.array([[2.0, 0.25], [8.0, 0.5]], dtype=np.float32)   # [n-block][k-block]
    for k0 in [0, 127, 128, 255]:
        codes[:] = 0
        codes[:, k0] = np.arange(256, dtype=np.uint8)
        x = np.zeros((1, K)); x[0, k0] = 1.0
        y = oracle.linear(oracle.FP8_B128, _bf16_bits_of(x), codes, scales, with_abs=False)[0]
        s = np.array([scales[n // 128, k0 // 128] for n in range(256)], dtype=np.float64)
        expect = ref * s
        nan = np.isnan(expect)
        assert np.array_equal(np.isnan(y), nan)
        assert np.array_equal(y[~nan], expect[~nan]), k0


def test_scale_one_blocks_give_integer_dot_products():
    rng = np.random.default_rng(5)
    M, N, K = 3, 129, 384
    wi = rng.integers(-16, 17, size=(N, K))
    xi = rng.integers(-8, 9, size=(M, K))
    q = _e4m3_code_of(wi.astype(np.float64))
    sc = np.ones(((N + 127) // 128, K // 128), dtype=np.float32)
    y = oracle.linear(oracle.FP8_B128, _bf16_bits_of(xi.astype(np.float64)), q, sc, with_abs=False)
    exact = np.array([[sum(int(a) * int(b) for a, b in zip(xi[m], wi[n])) for n in range(N)]
                      for m in range(M)], dtype=np.float64)
    assert np.array_equal(y, exact)


def test_linearity_exact_for_dyadic_inputs():
    rng = np.random.default_rng(9)
    M, N, K = 2, 40, 64
    w = rng.integers(-64, 65, size=(N, K)) / 64.0
    x1 = rng.integers(-8, 9, size=(M, K)) / 4.0       # alpha*x1 + x2 stays exact in bf16
    x2 = rng.integers(-8, 9, size=(M, K)) / 8.0
    bias = rng.integers(-16, 17, size=N) / 32.0
    alpha = 4.0
    wb, bb = _bf16_bits_of(w), _bf16_bits_of(bias)
    f = lambda xx: oracle.linear(oracle.BF16, _bf16_bits_of(xx), wb, bias_bits=bb, with_abs=False)  # noqa: E731
    lhs = f(alpha * x1 + x2) - bias
    rhs = alpha * (f(x1) - bias) + (f(x2) - bias)
    assert np.array_equal(lhs, rhs)


def test_abs_sum_is_sum_of_abs_products():
    x = np.array([[1.0, -2.0, 0.5, 0.0]])
    w = np.array([[3.0, 1.0, -4.0, 7.0], [-1.0, -1.0, -1.0, -1.0]])
    y, a = oracle.linear(oracle.BF16, _bf16_bits_of(x), _bf16_bits_of(w))
    assert y.tolist() == [[-1.0, 0.5]]
    assert a.tolist() == [[7.0, 3.5]]


# --------------------------------------------------------------------------- brute force

def _fraction_linear(x, w, bias=None):
    M, K = x.shape
    N = w.shape[0]
    out = []
    for m in range(M):
        row = []
        for n in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(float(x[m, k])) * Fraction(float(w[n, k]))
            if bias is not None:
                s += Fraction(float(bias[n]))
            row.append(s)
        out.append(row)
    return out


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (16, 2, 128), (3, 127, 128), (5, 129, 256),
                                   (2, 256, 256), (7, 128, 256)])
def test_brute_force_exact_rationals_dyadic(M, N, K):
    """Small dyadic values: every partial sum is exact in double -> equality."""
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    x = rng.integers(-8, 9, size=(M, K)) / 4.0
    codes = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38                      # no NaN codes
    wv = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()   # independent decode
    sexp = rng.integers(-3, 4, size=((N + 127) // 128, K // 128))
    scales = (2.0 ** sexp).astype(np.float32)
    wfull = wv * np.repeat(np.repeat(scales.astype(np.float64), 128, 0)[:N], 128, 1)
    bias = rng.integers(-8, 9, size=N) / 8.0
    y = oracle.linear(oracle.FP8_B128, _bf16_bits_of(x), codes, scales,
                      bias_bits=_bf16_bits_of(bias), with_abs=False)
    ref = _fraction_linear(x, wfull, bias)
    for m in range(M):
        for n in range(N):
            assert Fraction(y[m, n]) == ref[m][n], (m, n)


@pytest.mark.parametrize("M,N,K", [(1, 3, 128), (4, 5, 200), (16, 2, 256)])
def test_brute_force_gaussian_bf16_within_double_rounding(M, N, K):
    x = torch.randn(M, K, generator=torch.Generator().manual_seed(M + K)).to(torch.bfloat16)
    w = torch.randn(N, K, generator=torch.Generator().manual_seed(N + 7)).mul(0.02).to(torch.bfloat16)
    y, a = oracle.linear(oracle.BF16, x.view(torch.int16).numpy().view(np.uint16),
                         w.view(torch.int16).numpy().view(np.uint16))
    ref = _fraction_linear(x.double().numpy(), w.double().numpy())
    for m in range(M):
        for n in range(N):
            err = abs(Fraction(y[m, n]) - ref[m][n])
            assert err <= Fraction(K) * Fraction(2) ** -52 * Fraction(a[m, n])


def test_threads_do_not_change_results():
    x = torch.randn(4, 512, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    w = torch.randn(300, 512, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    wb = w.view(torch.int16).numpy().view(np.uint16)
    y1, a1 = oracle.linear(oracle.BF16, xb, wb, threads=1)
    y8, a8 = oracle.linear(oracle.BF16, xb, wb, threads=7)
    assert np.array_equal(y1, y8) and np.array_equal(a1, a8)
    rows = np.array([299, 0, 17])
    yr, _ = oracle.linear(oracle.BF16, xb, wb, rows=rows)
    assert np.array_equal(yr, y1[:, rows])


def test_rejects_bad_arguments():
    xb = np.zeros((1, 128), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.linear(oracle.FP8_B128, xb, np.zeros((2, 128), dtype=np.uint8))   # no scales
    with pytest.raises(ValueError):
        oracle.linear(oracle.BF16, xb, np.zeros((2, 64), dtype=np.uint16))       # K mismatch
    with pytest.raises(ValueError):
        oracle.linear(oracle.BF16, xb, np.zeros((2, 128), dtype=np.uint16), rows=[2])


# ------------------------------------------------------------------ SwiGLU epilogue

def test_silu_closed_forms():
    """sigma(ln 3) = 3/4 and sigma(-ln 3) = 1/4 exactly; silu(0) = 0; far from 0,
    silu(x) -> x (x > 0) and -> 0 from below (x < 0)."""
    ln3 = math.log(3.0)
    got = oracle.silu(np.array([ln3, -ln3, 0.0, 64.0, -64.0, -800.0]))
    assert got[0] == pytest.approx(0.75 * ln3, rel=1e-15)
    assert got[1] == pytest.approx(-0.25 * ln3, rel=1e-15)
    assert got[2] == 0.0
    assert got[3] == 64.0                       # sigma(64) rounds to 1 in double
    assert -1e-25 < got[4] < 0.0                # -64 e^-64 / (1 + e^-64)
    assert got[5] == 0.0 and math.copysign(1.0, got[5]) < 0   # e^800 overflows: -0


def test_silu_odd_part_identity():
    """silu(x) - silu(-x) = x (sigma(x) + sigma(-x) = 1): catches a sign slip."""
    x = np.linspace(-30.0, 30.0, 241)
    assert np.allclose(oracle.silu(x) - oracle.silu(-x), x, rtol=1e-14, atol=1e-13)


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP8_B128])
def test_swiglu_pairs_gate_and_up_rows(dtype):
    """x = e_0 selects column 0: g_j and u_j are exactly the values placed in
    the gate and up rows of output j; gates alternate 0 (silu = 0) and 64
    (silu = 64 exactly), ups are distinct integers, so y_j is 0 or 64 u_j and a
    swapped or shifted pairing shows."""
    I, K = 24, 128
    gate_vals = np.where(np.arange(I) % 2 == 0, 0.0, 64.0)
    # 24 distinct values exact in both bf16 and e4m3
    up_vals = np.array([1, 1.5, 2, 2.5, 3, 3.5, 4, 5, 6, 7, 8, 10, 12, 14, 16, 20, 24, 28, 32, 40,
                        48, 56, 64, 80], dtype=np.float64) * np.where(np.arange(I) % 3 == 0, -1, 1)
    gate_rows, up_rows = oracle.swiglu_rows(I)
    W = np.zeros((2 * I, K))
    W[gate_rows, 0] = gate_vals
    W[up_rows, 0] = up_vals
    x = np.zeros((1, K)); x[0, 0] = 1.0
    xb = _bf16_bits_of(x)
    if dtype == oracle.BF16:
        y, g, u, _, _ = oracle.swiglu(dtype, xb, _bf16_bits_of(W))
    else:
        y, g, u, _, _ = oracle.swiglu(dtype, xb, _e4m3_code_of(W), np.ones((1, 1), np.float32))
    assert np.array_equal(g[0], gate_vals) and np.array_equal(u[0], up_vals)
    assert np.array_equal(y[0], np.where(gate_vals == 64.0, 64.0 * up_vals, 0.0))


def test_swiglu_rows_match_the_binding_layout():
    """The oracle's pairing is the layout interleave_gate_up produces."""
    import torch
    import weight_streaming_skinny_gb300 as dl
    I = 40
    gate = torch.arange(I, dtype=torch.float64)[:, None]
    up = -1.0 - gate
    w = dl.interleave_gate_up(gate, up)[:, 0].numpy()
    gr, ur = oracle.swiglu_rows(I)
    assert np.array_equal(w[gr], gate[:, 0].numpy()) and np.array_equal(w[ur], up[:, 0].numpy())


# ------------------------------------------------------------------ argmax of the lm_head

def test_argmax_lowest_special_cases():
    """Ties go to the lowest index; the first NaN wins; -0 equals +0; -inf rows."""
    v = np.array([[1.0, 3.0, 3.0, 2.0],
                  [1.0, np.nan, 5.0, np.nan],
                  [-0.0, 0.0, -1.0, 0.0],
                  [-np.inf, -np.inf, -np.inf, -np.inf],
                  [np.nan, 9.0, 1.0, 2.0],
                  [-5.0, -2.0, -2.0, -7.0]])
    assert oracle.argmax_lowest(v).tolist() == [1, 1, 0, 0, 0, 1]


def test_argmax_lowest_matches_numpy_on_distinct_values():
    """Without ties or NaN it is numpy's argmax (an independent routine)."""
    rng = np.random.default_rng(5)
    v = rng.standard_normal((7, 513))
    assert np.array_equal(oracle.argmax_lowest(v), np.argmax(v, axis=1))
