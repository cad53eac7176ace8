"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something it does not compute itself:
a library conversion routine, exact integer arithmetic, a closed form, a
hand-derived worked step, finite differences or an invariant.  Together they
are chosen so that a dropped term, a flipped sign, a wrong index or a
transposed operand anywhere in the oracle breaks at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from persistent_step_megakernel_gb300 import synthetic as S
from persistent_step_megakernel_gb300.ir import Operation, Program, TensorSpec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
T = TensorSpec.contiguous


# --------------------------------------------------------------- rounding

def _fp32_sample(n_random=1 << 20):
    rng = np.random.default_rng(1234)
    rand = rng.integers(0, 1 << 32, size=n_random, dtype=np.uint64).astype(np.uint32)
    strided = (np.arange(0, 1 << 32, 4099, dtype=np.uint64)).astype(np.uint32)
    # every exponent x sign x {tie, tie +- 1 lsb, ...} of the bits bf16/fp16 drop
    exps = np.arange(256, dtype=np.uint32) << np.uint32(23)
    lows = np.array([0, 1, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x7FFF, 0x8000, 0x8001,
                     0xFFFF, 0x10000, 0x18000, 0x3FFFFF, 0x7FFFFF, 0x400000, 0x7F8000], dtype=np.uint32)
    edge = (exps[:, None] | lows[None, :]).reshape(-1)
    edge = np.concatenate([edge, edge | np.uint32(0x80000000)])
    bits = np.concatenate([rand, strided, edge])
    vals = bits.view(np.float32)
    return vals


def _same(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return both_nan | eq


def test_bfloat16_rounding_matches_library_conversion():
    v = _fp32_sample()
    with np.errstate(invalid="ignore", over="ignore"):
        ours = oracle.round_values(v.astype(np.float64), "bfloat16")
    lib = torch.from_numpy(v.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    bad = ~_same(ours, lib)
    assert not bad.any(), (v[bad][:8], ours[bad][:8], lib[bad][:8])


def test_float16_rounding_matches_library_conversion():
    v = _fp32_sample()
    with np.errstate(invalid="ignore", over="ignore"):
        ours = oracle.round_values(v.astype(np.float64), "float16")
        lib = v.astype(np.float16).astype(np.float64)
    bad = ~_same(ours, lib)
    assert not bad.any(), (v[bad][:8], ours[bad][:8], lib[bad][:8])


@pytest.mark.parametrize("dtype,value,expected", [
    ("bfloat16", 1 + 2 ** -8, 1.0),                         # tie -> even (down)
    ("bfloat16", 1 + 3 * 2 ** -8, 1 + 2 ** -6),              # tie -> even (up)
    ("bfloat16", 1 + 2 ** -8 + 2 ** -20, 1 + 2 ** -7),       # above tie
    ("bfloat16", 255 * 2.0 ** 120, 255 * 2.0 ** 120),        # largest finite
    ("bfloat16", 255.5 * 2.0 ** 120, math.inf),              # tie at the top -> inf
    ("bfloat16", -0.0, -0.0),
    ("bfloat16", 2.0 ** -133, 2.0 ** -133),                   # subnormal, exact
    ("float16", 65504.0, 65504.0),
    ("float16", 65519.0, 65504.0),
    ("float16", 65520.0, math.inf),
    ("float16", 2.0 ** -24, 2.0 ** -24),                      # smallest subnormal
    ("float16", 2.0 ** -25, 0.0),                             # tie -> even zero
    ("float16", 3 * 2.0 ** -25, 2.0 ** -23),                  # tie -> even (up)
    ("float16", 1 + 2 ** -11, 1.0),
    ("float32", 1 + 2 ** -24, 1.0),
    ("float32", 1 + 2 ** -23, 1 + 2 ** -23),
])
def test_rounding_textbook_cases(dtype, value, expected):
    got = oracle.round_values(np.array([value]), dtype)[0]
    assert got == expected and math.copysign(1, got) == math.copysign(1, expected)


def test_rounding_keeps_nan_and_inf():
    for dt in ("float32", "float16", "bfloat16"):
        r = oracle.round_values(np.array([np.nan, np.inf, -np.inf]), dt)
        assert np.isnan(r[0]) and r[1] == np.inf and r[2] == -np.inf


# ------------------------------------------------------------ single ops

def _run_single(op_kind, ins, out, values, attrs=None, dtype="float32", extra_inputs=()):
    inputs = [x for x in ins if isinstance(x, TensorSpec)] + list(extra_inputs)
    seen, uniq = set(), []
    for s in inputs:
        if s.buffer not in seen:
            seen.add(s.buffer)
            uniq.append(T(s.buffer, values[s.buffer].shape, s.dtype))
    prog = Program(uniq, [out], [Operation("o", op_kind, tuple(ins), out, dict(attrs or {}))])
    o = oracle.Oracle(prog)
    for s in uniq:
        o.set(s.buffer, values[s.buffer])
    o.run()
    return o.output(0)


def test_mm_integer_inputs_exact_including_transposed_views():
    rng = np.random.default_rng(7)
    A = rng.integers(-8, 9, size=(5, 7)).astype(np.float64)
    Bm = rng.integers(-8, 9, size=(6, 7)).astype(np.float64)    # stored [n, k]; used transposed
    a, b = T("A", (5, 7), "float32"), T("B", (6, 7), "float32")
    got = _run_single("mm", (a, b.T), T("C", (5, 6), "float32"), {"A": A, "B": Bm})
    np.testing.assert_array_equal(got, A @ Bm.T)
    # transposed A operand: C = A^T A  ([7,5] x [5,7])
    got2 = _run_single("mm", (a.T, a), T("C", (7, 7), "float32"), {"A": A})
    np.testing.assert_array_equal(got2, A.T @ A)
    # a mis-transposed operand would give a different (non-symmetric) product here
    assert not np.array_equal(A @ Bm.T, (Bm @ A.T).T[::-1])


@pytest.mark.parametrize("alpha,beta", [(1, 1), (2, -3), (0, 0), (0, 2), (3, 0)])
def test_addmm_alpha_beta_cases(alpha, beta):
    rng = np.random.default_rng(11)
    A = rng.integers(-4, 5, size=(3, 4)).astype(np.float64)
    W = rng.integers(-4, 5, size=(5, 4)).astype(np.float64)
    bias = rng.integers(-4, 5, size=(5,)).astype(np.float64)
    bias[0] = np.nan if (alpha, beta) == (3, 0) else bias[0]   # beta == 0 must not read bias
    a, w, b = T("A", (3, 4), "float32"), T("W", (5, 4), "float32"), T("bias", (5,), "float32")
    got = _run_single("addmm", (b, a, w.T), T("C", (3, 5), "float32"),
                      {"A": A, "W": W, "bias": bias}, {"alpha": alpha, "beta": beta})
    acc = A @ W.T
    if alpha == 0 and beta == 0:
        want = np.zeros_like(acc)
    elif beta == 0:
        want = alpha * acc
    elif alpha == 0:
        want = np.broadcast_to(beta * bias, acc.shape)
    else:
        want = alpha * acc + beta * bias
    np.testing.assert_array_equal(got, want)


def test_sum_closed_forms_and_dims():
    N = 4096
    v = np.arange(1, N + 1, dtype=np.float64)
    x = T("x", (N,), "float32")
    got = _run_single("sum", (x,), T("s", (), "float32"), {"x": v})
    assert got == N * (N + 1) // 2
    got = _run_single("mean", (x,), T("m", (), "float32"), {"x": v})
    assert got == np.float32(np.float32(N * (N + 1) // 2) / np.float32(N))
    M = np.arange(12, dtype=np.float64).reshape(3, 4)          # column sums 12,15,18,21
    m = T("M", (3, 4), "float32")
    np.testing.assert_array_equal(
        _run_single("sum", (m,), T("c", (4,), "float32"), {"M": M}, {"dims": (0,)}), [12, 15, 18, 21])
    np.testing.assert_array_equal(
        _run_single("sum", (m,), T("r", (3,), "float32"), {"M": M}, {"dims": (-1,)}), [6, 22, 38])
    # column sums over a transposed view equal row sums of the stored matrix
    np.testing.assert_array_equal(
        _run_single("sum", (m.T,), T("r2", (3,), "float32"), {"M": M}, {"dims": (0,)}), [6, 22, 38])
    e = T("e", (0, 3), "float32")
    got = _run_single("mean", (e,), T("me", (3,), "float32"), {"e": np.zeros(0)}, {"dims": (0,)})
    assert np.isnan(got).all()


def test_rank3_reductions_closed_forms():
    # x[i, j, k] = 100 i + 10 j + k: every sum below has a closed form
    A, Bd, C = 3, 4, 5
    i, j, k = np.meshgrid(np.arange(A), np.arange(Bd), np.arange(C), indexing="ij")
    xv = (100 * i + 10 * j + k).astype(np.float64)
    x = T("x", (A, Bd, C), "float32")
    tri = lambda n: n * (n - 1) // 2
    # over the middle dim: B (100 i + k) + 10 * (0 + 1 + ... + B-1)
    got = _run_single("sum", (x,), T("m", (A, C), "float32"), {"x": xv}, {"dims": (1,)})
    want = np.array([[Bd * (100 * a + c) + 10 * tri(Bd) for c in range(C)] for a in range(A)])
    np.testing.assert_array_equal(got, want)
    got = _run_single("sum", (x,), T("m2", (A, C), "float32"), {"x": xv}, {"dims": (-2,)})
    np.testing.assert_array_equal(got, want)
    # over the outer and inner dims: 100 C tri(A) + 10 A C j + A tri(C)
    got = _run_single("sum", (x,), T("o", (Bd,), "float32"), {"x": xv}, {"dims": (0, 2)})
    want = np.array([100 * C * tri(A) + 10 * A * C * b + A * tri(C) for b in range(Bd)])
    np.testing.assert_array_equal(got, want)
    got = _run_single("mean", (x,), T("om", (Bd,), "float32"), {"x": xv}, {"dims": (0, -1)})
    np.testing.assert_array_equal(got, (want.astype(np.float32) / np.float32(A * C)).astype(np.float32))
    # over the two leading dims, and over every dim
    got = _run_single("sum", (x,), T("l", (C,), "float32"), {"x": xv}, {"dims": (0, 1)})
    np.testing.assert_array_equal(got, [100 * Bd * tri(A) + 10 * A * tri(Bd) + A * Bd * c for c in range(C)])
    got = _run_single("sum", (x,), T("a", (), "float32"), {"x": xv})
    assert got == 100 * Bd * C * tri(A) + 10 * A * C * tri(Bd) + A * Bd * tri(C)
    # a permuted (non-contiguous) view: reducing its dim 0 is reducing the stored middle dim
    xt = TensorSpec("x", (Bd, A, C), (C, Bd * C, 1), 0, "float32")
    got = _run_single("sum", (xt,), T("p", (A, C), "float32"), {"x": xv}, {"dims": (0,)})
    np.testing.assert_array_equal(got, [[Bd * (100 * a + c) + 10 * tri(Bd) for c in range(C)] for a in range(A)])


def test_full_takes_the_value_attribute_over_an_operand():
    # page "trainkernel/codegen.py", point_expr: attrs["value"] when present,
    # else the first operand, else 0
    f = _run_single("full", (2.5,), T("f", (2,), "float32"), {}, {"value": 0.75})
    np.testing.assert_array_equal(f, [0.75, 0.75])
    f = _run_single("full", (2.5,), T("f", (2,), "float32"), {})
    np.testing.assert_array_equal(f, [2.5, 2.5])
    f = _run_single("full", (), T("f", (2,), "float32"), {})
    np.testing.assert_array_equal(f, [0.0, 0.0])


def test_pointwise_semantics_special_cases():
    x = T("x", (6,), "float32")
    v = np.array([-1.5, -0.0, 0.0, 2.0, np.nan, 3.0])
    r = _run_single("relu", (x,), T("r", (6,), "float32"), {"x": v})
    assert r[0] == 0 and math.copysign(1, r[1]) == -1 and r[3] == 2 and np.isnan(r[4])
    g = T("g", (6,), "float32")
    gv = np.array([1.0, 2.0, 3.0, 4.0, 5.0, 6.0])
    tb = _run_single("threshold_backward", (g, x), T("t", (6,), "float32"), {"g": gv, "x": v},
                     {"threshold": 0.0})
    np.testing.assert_array_equal(tb[[0, 1, 2, 3, 5]], [0, 0, 0, 4, 6])   # s <= 0 -> 0
    assert tb[4] == 5                                                      # NaN <= 0 is false
    a = _run_single("sub", (g, x), T("s", (6,), "float32"), {"g": gv, "x": np.ones(6)}, {"alpha": 0.5})
    np.testing.assert_array_equal(a, gv - 0.5)
    a = _run_single("add", (g, 0.25), T("s", (6,), "float32"), {"g": gv}, {"alpha": -2.0})
    np.testing.assert_array_equal(a, gv - 0.5)
    d = _run_single("div", (g, 4.0), T("q", (6,), "float32"), {"g": gv})
    np.testing.assert_array_equal(d, gv / 4)
    p = _run_single("pow", (g, 2), T("p", (6,), "float32"), {"g": gv})
    np.testing.assert_array_equal(p, gv ** 2)
    # general exponents: exact cases of the real power function
    p = _run_single("pow", (g, 3), T("p", (6,), "float32"), {"g": gv})
    np.testing.assert_array_equal(p, gv ** 3)
    sq = np.array([1.0, 4.0, 9.0, 16.0, 0.25, 2.0 ** 20])
    p = _run_single("pow", (g, 0.5), T("p", (6,), "float32"), {"g": sq})
    np.testing.assert_array_equal(p, np.sqrt(sq))
    p = _run_single("pow", (g, -1), T("p", (6,), "float32"), {"g": np.array([1.0, 2.0, 4.0, 0.5, -8.0, 1024.0])})
    np.testing.assert_array_equal(p, [1.0, 0.5, 0.25, 2.0, -0.125, 2.0 ** -10])
    p = _run_single("pow", (g, 0), T("p", (6,), "float32"), {"g": np.array([0.0, -3.0, 7.5, 1e30, -0.0, 2.0])})
    np.testing.assert_array_equal(p, np.ones(6))
    n = _run_single("neg", (g,), T("n", (6,), "float32"), {"g": gv})
    np.testing.assert_array_equal(n, -gv)
    f = _run_single("full", (), T("f", (2, 3), "bfloat16"), {}, {"value": 1 + 2 ** -8})
    np.testing.assert_array_equal(f, np.ones((2, 3)))                  # literal rounded to bf16
    c = _run_single("cast", (g,), T("c", (6,), "bfloat16"), {"g": gv + 2 ** -8})
    np.testing.assert_array_equal(c, gv)                               # ties to even


def test_float32_pointwise_rounds_each_operation():
    # sub with alpha: a - fl32(alpha*b); rounding the product first matters here.
    a_v, b_v, alpha = np.array([1.0]), np.array([1 + 2 ** -12]), 1 + 2 ** -12
    got = _run_single("sub", (T("a", (1,), "float32"), T("b", (1,), "float32")), T("s", (1,), "float32"),
                      {"a": a_v, "b": b_v}, {"alpha": alpha})
    prod = np.float32(np.float32(alpha) * np.float32(b_v[0]))
    assert got[0] == np.float32(np.float32(1.0) - prod)
    assert got[0] != np.float32(1.0 - alpha * b_v[0])  # an unrounded product would differ


def test_broadcast_right_aligned_and_errors():
    m = T("m", (2, 3), "float32")
    row = T("row", (3,), "float32")
    col = T("col", (2, 1), "float32")
    M = np.arange(6.0).reshape(2, 3)
    got = _run_single("add", (m, row), T("o", (2, 3), "float32"), {"m": M, "row": np.array([10., 20., 30.])})
    np.testing.assert_array_equal(got, M + [10, 20, 30])
    got = _run_single("mul", (m, col), T("o", (2, 3), "float32"), {"m": M, "col": np.array([[2.], [3.]])})
    np.testing.assert_array_equal(got, M * [[2], [3]])
    with pytest.raises(RuntimeError, match="broadcast"):
        _run_single("add", (m, T("bad", (2,), "float32")), T("o", (2, 3), "float32"),
                    {"m": M, "bad": np.ones(2)})
    with pytest.raises(RuntimeError, match="compatible rank-two"):
        _run_single("mm", (m, m), T("o", (2, 3), "float32"), {"m": M})


# --------------------------------------------------- whole-step worked example

def _golden():
    with open(os.path.join(GOLDEN, "two_layer_step.json")) as f:
        return json.load(f)


def _golden_program(dtype):
    g = _golden()
    cfg = S.scaled(S.CONFIGS["c1"], batch=2, dims=tuple(g["config"]["dims"]), lr=g["config"]["lr"], dtype=dtype)
    prog = S.mlp_step_program(cfg, export="all")
    vals = [np.array(g["inputs"][s.buffer], dtype=np.float64) for s in prog.inputs]
    return g, prog, vals


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "float16", "float64"])
def test_hand_computed_two_layer_step(dtype):
    g, prog, vals = _golden_program(dtype)
    outs = oracle.run_program(prog, vals)
    by_name = {s.buffer: o for s, o in zip(prog.outputs, outs)}
    for name, want in g["expected"].items():
        np.testing.assert_array_equal(by_name[name], np.array(want), err_msg=name)


def test_hand_computed_step_matches_exact_backprop():
    """The fixture itself against textbook backprop in exact rationals."""
    g = _golden()
    F = lambda a: [[Fraction(v) for v in r] for r in a]
    x, y = F(g["inputs"]["x"]), F(g["inputs"]["y"])
    W1, W2 = F(g["inputs"]["W1"]), F(g["inputs"]["W2"])
    b1, b2 = [Fraction(v) for v in g["inputs"]["b1"]], [Fraction(v) for v in g["inputs"]["b2"]]
    lr = Fraction(g["config"]["lr"])
    B = len(x)
    z1 = [[sum(W1[j][k] * x[n][k] for k in range(2)) + b1[j] for j in range(2)] for n in range(B)]
    a1 = [[max(v, 0) for v in r] for r in z1]
    z2 = [[sum(W2[0][j] * a1[n][j] for j in range(2)) + b2[0]] for n in range(B)]
    loss = sum((z2[n][0] - y[n][0]) ** 2 for n in range(B)) / B
    dz2 = [2 * (z2[n][0] - y[n][0]) / B for n in range(B)]
    gW2 = [sum(dz2[n] * a1[n][j] for n in range(B)) for j in range(2)]
    dz1 = [[dz2[n] * W2[0][j] * (1 if z1[n][j] > 0 else 0) for j in range(2)] for n in range(B)]
    gW1 = [[sum(dz1[n][j] * x[n][k] for n in range(B)) for k in range(2)] for j in range(2)]
    gb1 = [sum(dz1[n][j] for n in range(B)) for j in range(2)]
    e = g["expected"]
    assert loss == Fraction(e["loss"])
    assert [[W1[j][k] - lr * gW1[j][k] for k in range(2)] for j in range(2)] == F(e["W1_new"])
    assert [W2[0][j] - lr * gW2[j] for j in range(2)] == F(e["W2_new"])[0]
    assert [b1[j] - lr * gb1[j] for j in range(2)] == [Fraction(v) for v in e["b1_new"]]
    assert b2[0] - lr * sum(dz2) == Fraction(e["b2_new"][0])


def _golden_momentum():
    with open(os.path.join(GOLDEN, "two_layer_momentum_step.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("dtype,master", [("float32", None), ("bfloat16", None), ("float16", None),
                                          ("float64", None), ("bfloat16", "float32")])
def test_hand_computed_momentum_step(dtype, master):
    # the momentum wiring (v' = mu v + g, W' = W - lr v', in place) and, with a
    # float32 master copy, the mixed-precision wiring (bf16 GEMM copies of the
    # weights, float32 loss, gradients of the weights and updates)
    g = _golden_momentum()
    c = g["config"]
    cfg = S.scaled(S.CONFIGS["c1"], batch=c["batch"], dims=tuple(c["dims"]), lr=c["lr"], momentum=c["momentum"],
                   dtype=dtype, master=master)
    prog = S.mlp_step_program(cfg, export="grads")
    if master:
        assert any(op.op == "cast" for op in prog.operations)
        assert {s.dtype for s in prog.inputs if s.buffer.startswith(("W", "b", "v"))} == {master}
    vals = [np.array(g["inputs"][s.buffer], dtype=np.float64) for s in prog.inputs]
    outs = oracle.run_program(prog, vals)
    by_name = {s.buffer: o for s, o in zip(prog.outputs, outs)}
    assert set(g["expected"]) == set(by_name)
    for name, want in g["expected"].items():
        np.testing.assert_array_equal(by_name[name], np.array(want), err_msg=name)


def test_hand_computed_momentum_step_matches_exact_momentum_sgd():
    """The momentum fixture against textbook backprop and momentum SGD in exact rationals."""
    g = _golden_momentum()
    F = lambda a: [[Fraction(v) for v in r] for r in a]
    F1 = lambda a: [Fraction(v) for v in a]
    inp = g["inputs"]
    x, y, W1, W2 = F(inp["x"]), F(inp["y"]), F(inp["W1"]), F(inp["W2"])
    b1, b2 = F1(inp["b1"]), F1(inp["b2"])
    vW1, vW2, vb1, vb2 = F(inp["vW1"]), F(inp["vW2"]), F1(inp["vb1"]), F1(inp["vb2"])
    lr, mu, B = Fraction(g["config"]["lr"]), Fraction(g["config"]["momentum"]), len(x)
    z1 = [[sum(W1[j][k] * x[n][k] for k in range(2)) + b1[j] for j in range(2)] for n in range(B)]
    a1 = [[max(v, 0) for v in r] for r in z1]
    z2 = [sum(W2[0][j] * a1[n][j] for j in range(2)) + b2[0] for n in range(B)]
    dz2 = [2 * (z2[n] - y[n][0]) / B for n in range(B)]
    gW2 = [sum(dz2[n] * a1[n][j] for n in range(B)) for j in range(2)]
    dz1 = [[dz2[n] * W2[0][j] * (1 if z1[n][j] > 0 else 0) for j in range(2)] for n in range(B)]
    gW1 = [[sum(dz1[n][j] * x[n][k] for n in range(B)) for k in range(2)] for j in range(2)]
    gb1 = [sum(dz1[n][j] for n in range(B)) for j in range(2)]
    gb2 = sum(dz2)
    e = g["expected"]
    vW1n = [[mu * vW1[j][k] + gW1[j][k] for k in range(2)] for j in range(2)]
    vW2n = [mu * vW2[0][j] + gW2[j] for j in range(2)]
    vb1n = [mu * vb1[j] + gb1[j] for j in range(2)]
    vb2n = mu * vb2[0] + gb2
    assert vW1n == F(e["vW1_new"]) and [vW2n] == F(e["vW2_new"])
    assert vb1n == F1(e["vb1_new"]) and [vb2n] == F1(e["vb2_new"])
    assert [[W1[j][k] - lr * vW1n[j][k] for k in range(2)] for j in range(2)] == F(e["W1_new"])
    assert [[W2[0][j] - lr * vW2n[j] for j in range(2)]] == F(e["W2_new"])
    assert [b1[j] - lr * vb1n[j] for j in range(2)] == F1(e["b1_new"])
    assert [b2[0] - lr * vb2n] == F1(e["b2_new"])
    assert sum((z2[n] - y[n][0]) ** 2 for n in range(B)) / B == Fraction(e["loss"])


# ------------------------------------------------------ finite differences

def _fd_inputs(cfg, prog, seed):
    """float64 inputs whose pre-activations all keep |z| > 1e-2 (no ReLU kink)."""
    for s in range(seed, seed + 200):
        vals = S.mlp_inputs(cfg, prog, seed=s, dtype="float64")
        o = oracle.Oracle(S.mlp_step_program(cfg, export="all", dtype="float64"))
        o.set_inputs(vals)
        o.run()
        zs = [o.get(f"z{i}") for i in range(1, cfg.layers)]
        if all(np.abs(z).min() > 1e-2 for z in zs):
            return vals
    raise RuntimeError("no kink-free inputs found")


@pytest.mark.parametrize("key,changes", [
    ("c1", {}),
    ("c3", {"batch": 3, "dims": (4, 6, 4)}),
    ("c2", {"batch": 4, "dims": (5, 7, 6, 3)}),
    ("c2m", {"batch": 4, "dims": (5, 7, 6, 3)}),                  # the cast-to-compute-copy wiring
    ("c2m", {"batch": 3, "dims": (4, 6, 3), "momentum": 0.9}),
    ("lsq", {"batch": 5, "dims": (6, 3)}),                        # one-hot targets, one layer
])
def test_gradients_match_central_finite_differences(key, changes):
    cfg = S.scaled(S.CONFIGS[key], **changes)
    prog = S.mlp_step_program(cfg, export="grads", dtype="float64")
    vals = _fd_inputs(cfg, prog, 0)
    o = oracle.Oracle(prog)
    o.set_inputs(vals)
    o.run()
    loss_prog = Program(prog.inputs, [prog.outputs[0]], prog.operations)
    names = [s.buffer for s in prog.inputs]

    def loss_at(vs):
        return oracle.run_program(loss_prog, vs)[0].item()

    h = 1e-6
    for i in range(1, cfg.layers + 1):
        for pname, gname in ((f"W{i}", f"gW{i}"), (f"b{i}", f"gb{i}")):
            grad = o.get(gname)
            k = names.index(pname)
            base = np.array(vals[k], dtype=np.float64)
            fd = np.empty(base.size)
            for j in range(base.size):
                vp, vm = base.copy().reshape(-1), base.copy().reshape(-1)
                vp[j] += h
                vm[j] -= h
                vs_p = list(vals); vs_p[k] = vp.reshape(base.shape)
                vs_m = list(vals); vs_m[k] = vm.reshape(base.shape)
                fd[j] = (loss_at(vs_p) - loss_at(vs_m)) / (2 * h)
            scale = max(np.abs(fd).max(), 1e-3)
            assert np.abs(fd - grad).max() <= 1e-6 * scale + 1e-9, (pname, np.abs(fd - grad).max(), scale)


# ----------------------------------------------------------- invariants

def test_zero_learning_rate_leaves_parameters_unchanged():
    for key, ch in (("c2", {}), ("c3", {"batch": 4, "dims": (16, 32, 16)})):
        cfg = S.scaled(S.CONFIGS[key], lr=0.0, **ch)
        prog = S.mlp_step_program(cfg, export="state")
        ins = S.mlp_inputs(cfg, prog)
        vals = [S.storage_to_float64(a, s.dtype) for a, s in zip(ins, prog.inputs)]
        outs = oracle.run_program(prog, vals)
        for slot, idx in prog.inplace.items():
            if prog.inputs[idx].buffer.startswith("v"):
                continue                                                   # momentum buffers do move
            np.testing.assert_array_equal(outs[slot] == vals[idx], True)   # by value (-0 == +0)


def test_relu_masks_follow_preactivation_sign():
    cfg = S.CONFIGS["c2"]
    prog = S.mlp_step_program(cfg, export="all")
    ins = S.mlp_inputs(cfg, prog)
    o = oracle.Oracle(prog)
    o.set_inputs([S.storage_to_float64(a, s.dtype) for a, s in zip(ins, prog.inputs)])
    o.run()
    for i in range(1, cfg.layers):
        z, g = o.get(f"z{i}"), o.get(f"g{i}")
        assert np.all(g[z <= 0] == 0)
        ga = o.get(f"ga{i}")
        np.testing.assert_array_equal(g[z > 0], ga[z > 0])
        assert (z > 0).any() and (z <= 0).any()


def test_one_hot_least_squares_head_closed_form_at_zero_weights():
    # logits = 0: loss = mean(onehot^2) = 1/C; g = -2/(B C) onehot, so
    # gb[c] = -2/(B C) * count(c) and gW[c] = -2/(B C) * sum of the rows of x labelled c
    cfg = S.scaled(S.CONFIGS["lsq"], dtype="float32", batch=12, dims=(7, 4))
    prog = S.mlp_step_program(cfg, export="grads")
    ins = S.mlp_inputs(cfg, prog)
    vals = [S.storage_to_float64(a, s.dtype) for a, s in zip(ins, prog.inputs)]
    names = [s.buffer for s in prog.inputs]
    for p in ("W1", "b1"):
        vals[names.index(p)] = np.zeros_like(vals[names.index(p)])
    outs = {s.buffer: o for s, o in zip(prog.outputs, oracle.run_program(prog, vals))}
    x, y = vals[names.index("x")], vals[names.index("y")]
    B, C = y.shape
    assert (y.sum(1) == 1).all() and set(np.unique(y)) == {0.0, 1.0}
    assert outs["loss"] == np.float32(1.0 / C)
    scale = -2.0 / (B * C)
    np.testing.assert_allclose(outs["gb1"], scale * y.sum(0), rtol=1e-6)
    np.testing.assert_allclose(outs["gW1"], scale * (y.T @ x), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(outs["W1_new"], -cfg.lr * outs["gW1"], rtol=1e-6, atol=1e-9)


def test_residual_loss_closed_form_with_zero_second_layer():
    cfg = S.scaled(S.CONFIGS["c3"], batch=4, dims=(8, 16, 8))
    prog = S.mlp_step_program(cfg, export="state")
    ins = S.mlp_inputs(cfg, prog)
    vals = [S.storage_to_float64(a, s.dtype) for a, s in zip(ins, prog.inputs)]
    names = [s.buffer for s in prog.inputs]
    vals[names.index("W2")] = np.zeros_like(vals[names.index("W2")])
    vals[names.index("b2")] = np.zeros_like(vals[names.index("b2")])
    loss = oracle.run_program(prog, vals)[0].item()
    x = vals[names.index("x")]
    sq = (x * x).astype(np.float16).astype(np.float64)           # pow rounds to fp16
    want = np.float16(np.float32(np.float32(sq.sum()) / np.float32(sq.size)))
    assert loss == float(want)
