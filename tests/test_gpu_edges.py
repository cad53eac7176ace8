"""Edge values through the CUDA path: rounding ties, signed zeros, NaN, +-inf,
subnormals and overflow, bit for bit against the oracle.

Pointwise ops round one fully specified float32 expression once to the output
dtype, so results must match exactly -- including the sign of zero -- with NaN
in the same places (NaN payloads are not compared).  The GEMM programs use
small integer operands, whose float32 accumulators are exact in any summation
order, so their epilogues (bias, ReLU, the target difference with the loss
gradient as a side output, the ReLU mask) are fully specified too; they run
through the staged tensor-core epilogue at every tile width and through the
generic-chain and instruction forms.
"""
import numpy as np
import pytest

import oracle
from persistent_step_megakernel_gb300 import synthetic as S
from persistent_step_megakernel_gb300.build import build
from persistent_step_megakernel_gb300.ir import Operation, Program, TensorSpec
from tests._gpu import run_step
from tests._util import values

pytestmark = pytest.mark.gpu
T = TensorSpec.contiguous


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def bits(v, dtype):
    """Bit patterns of values exactly representable in dtype (NaN -> -1)."""
    v = np.asarray(v, dtype=np.float64).reshape(-1)
    if dtype == "float16":
        b = v.astype(np.float16).view(np.uint16).astype(np.int64)
    else:
        b = v.astype(np.float32).view(np.uint32).astype(np.int64)
    return np.where(np.isnan(v), -1, b)


def assert_bit_exact(got, want, dtype, name):
    g, w = bits(got, dtype), bits(want, dtype)
    bad = g != w
    assert not bad.any(), (name, np.asarray(got).reshape(-1)[bad][:6], np.asarray(want).reshape(-1)[bad][:6])


def edge_pairs():
    """(x, y) float32 pairs aimed at the rounding and special cases of each op."""
    inf, nan = np.inf, np.nan
    p = [(nan, 1.0), (1.0, nan), (inf, 1.0), (-inf, 1.0), (inf, -inf), (inf, inf), (-inf, -inf),
         (0.0, -0.0), (-0.0, -0.0), (-0.0, 0.0), (0.0, 0.0), (1.0, 0.0), (-1.0, 0.0), (1.0, -0.0),
         (-0.0, 1.0), (0.0, -1.0), (3.0e38, 3.0e38), (-3.0e38, 3.0e38), (65504.0, 16.0), (65519.0, 1.0),
         (65520.0, 0.0), (-65520.0, 0.0), (2.0 ** -149, 1.0), (2.0 ** -140, 2.0 ** -3), (-(2.0 ** -130), 3.0),
         (1.0 + 2.0 ** -4, 1.0 + 2.0 ** -4), (1.0 + 3 * 2.0 ** -5, 1.0 + 2.0 ** -3), (2.0 ** -12, 2.0 ** -13)]
    # exact ties of the float32 result at 16-bit precision, both parities
    for k in range(16):
        p.append((1.0 + k * 2.0 ** -7, 2.0 ** -8))        # bfloat16 ulp at 1 is 2^-7
        p.append((-(1.0 + k * 2.0 ** -7), -(2.0 ** -8)))
        p.append((1.0 + k * 2.0 ** -10, 2.0 ** -11))      # float16 ulp at 1 is 2^-10
        p.append((256.0 + 2 * k + 1, 0.0))                # bfloat16 ulp at 256 is 2
        p.append(((2 * k + 1) * 2.0 ** -25, 0.0))         # float16 subnormal ties (spacing 2^-24)
        p.append(((2 * k + 1) * 2.0 ** -134, 0.0))        # bfloat16 subnormal ties (spacing 2^-133)
        p.append((2048.0 + 2 * k + 1, 0.0))               # float16 ulp at 2048 is 2
    # the largest finite bfloat16 plus half an ulp (ties to even: overflows)
    p.append((float(np.float32((2 - 2.0 ** -7) * 2.0 ** 127)), float(np.float32(2.0 ** 119))))
    return p


def edge_inputs(shape, dtype, seed):
    n = int(np.prod(shape))
    pairs = edge_pairs()
    rnd = S.normal(S.stream_seed(seed, 0), 2 * n).reshape(n, 2)
    xy = np.concatenate([np.asarray(pairs, dtype=np.float64), rnd])[:n]
    xs = S.to_storage(xy[:, 0], "float32") if dtype == "float32" else None
    if dtype == "float32":
        return xs.reshape(shape), S.to_storage(xy[:, 1], "float32").reshape(shape)
    # 16-bit inputs: the pair values rounded once by numpy / truncated (exact in the dtype)
    return S.to_storage(xy[:, 0], dtype).reshape(shape), S.to_storage(xy[:, 1], dtype).reshape(shape)


def pointwise_program(in_dt):
    shape = (4, 256)
    x, y = T("x", shape, in_dt), T("y", shape, in_dt)
    V = lambda n, dt: T(n, shape, dt)
    ops = [
        Operation("a", "add", (x, y), V("a", "bfloat16")),
        Operation("a16", "add", (x, y), V("a16", "float16")),
        Operation("s", "sub", (x, y), V("s", "float16"), {"alpha": 0.5}),
        Operation("m", "mul", (x, y), V("m", "bfloat16")),
        Operation("m16", "mul", (x, y), V("m16", "float16")),
        Operation("q", "div", (x, y), V("q", "float16")),
        Operation("n", "neg", (x,), V("n", "bfloat16")),
        Operation("r", "relu", (x,), V("r", "float16")),
        Operation("t", "threshold_backward", (x, y), V("t", "bfloat16"), {"threshold": 0.0}),
        Operation("cb", "cast", (x,), V("cb", "bfloat16")),
        Operation("ch", "cast", (x,), V("ch", "float16")),
        Operation("p", "pow", (x, 2), V("p", "bfloat16")),
        Operation("f", "full", (), V("f", "bfloat16"), {"value": 1.0 + 2.0 ** -8}),
        Operation("f2", "full", (2.5,), V("f2", "float16"), {"value": 1.0 + 2.0 ** -11}),  # the attribute wins
        Operation("f3", "full", (0.75,), V("f3", "bfloat16")),
        # chains: inlined single-use values (the loss-gradient and update shapes)
        Operation("d", "sub", (x, y), V("d", "bfloat16")),
        Operation("g", "mul", (V("d", "bfloat16"), 0.125), V("g", "bfloat16")),
        Operation("u", "sub", (x, V("g", "bfloat16")), V("u", "bfloat16"), {"alpha": 3.0}),
        Operation("e", "add", (V("a", "bfloat16"), y), V("e", "float16"), {"alpha": -1.0}),
        Operation("w", "mul", (x, 0.75), V("w", in_dt)),
        Operation("ws", "sub", (V("w", in_dt), y), V("ws", in_dt), {"alpha": 0.25}),
    ]
    outs = [V(o.name, o.output.dtype) for o in ops if o.name not in ("d", "g", "w")]
    return Program([x, y], outs, ops)


@pytest.mark.parametrize("forms", [0, 1, 2])
@pytest.mark.parametrize("fuse", [0, 1])
@pytest.mark.parametrize("in_dt", ["float32", "bfloat16", "float16"])
def test_pointwise_edge_values_bit_exact(in_dt, fuse, forms):
    prog = pointwise_program(in_dt)
    arrays = list(edge_inputs((4, 256), in_dt, seed=23))
    gpu, st = run_step(prog, arrays, fuse_pointwise=fuse, expr_forms=forms)
    if fuse:
        assert st.stats["inlined_ops"] > 0
    want = oracle.run_program(prog, values(arrays, prog))
    for spec, g, w in zip(prog.outputs, gpu, want):
        assert_bit_exact(g, w, spec.dtype, (spec.buffer, in_dt, fuse, forms))


def gemm_program(dt):
    """Integer-valued GEMMs (exact accumulators) whose epilogues meet edge values."""
    M, N, K = 256, 256, 64
    a, W, e = T("a", (M, K), dt), T("W", (N, K), dt), T("e", (M, N), dt)
    b, y, mask = T("b", (N,), dt), T("y", (M, N), dt), T("mask", (M, K), dt)
    ops = [
        # forward layer: bias + ReLU (NaN passes ReLU)
        Operation("z", "addmm", (b, a, W.T), T("z", (M, N), dt)),
        Operation("h", "relu", (T("z", (M, N), dt),), T("h", (M, N), dt)),
        # output layer: bias, minus the target, the loss gradient as a side output
        Operation("z2", "addmm", (b, a, W.T), T("z2", (M, N), dt)),
        Operation("d", "sub", (T("z2", (M, N), dt), y), T("d", (M, N), dt)),
        Operation("g", "mul", (T("d", (M, N), dt), 0.125), T("g", (M, N), dt)),
        # input gradient with the ReLU mask
        Operation("ga", "mm", (e, W), T("ga", (M, K), dt)),
        Operation("gz", "threshold_backward", (T("ga", (M, K), dt), mask), T("gz", (M, K), dt), {"threshold": 0.0}),
        # a returned GEMM result and an update loading another input next to it
        # (a loaded side output): u = y - 0.5 q
        Operation("q", "mm", (a, W.T), T("q", (M, N), dt)),
        Operation("u", "sub", (y, T("q", (M, N), dt)), T("u", (M, N), dt), {"alpha": 0.5}),
    ]
    outs = [T("h", (M, N), dt), T("d", (M, N), dt), T("g", (M, N), dt), T("gz", (M, K), dt), T("q", (M, N), dt),
            T("u", (M, N), dt)]
    return Program([a, W, e, b, y, mask], outs, ops)


def gemm_inputs(prog, dt, seed):
    rng = np.random.default_rng(seed)
    shapes = {s.buffer: s.shape for s in prog.inputs}
    ints = lambda name, lo, hi: rng.integers(lo, hi + 1, size=shapes[name]).astype(np.float64)
    a, W, e = ints("a", -3, 3), ints("W", -3, 3), ints("e", -3, 3)
    special = np.array([np.nan, np.inf, -np.inf, 0.0, -0.0, 0.5, -0.5, 0.25, 2.0 ** -9, 2.0 ** -12, 1.0, 3.0])
    b = special[rng.integers(0, special.size, size=shapes["b"])]
    # the target: integers (exact differences and ties) and specials
    y = ints("y", -300, 300)
    pick = rng.random(shapes["y"]) < 0.05
    y[pick] = special[rng.integers(0, special.size, size=int(pick.sum()))]
    mask = rng.integers(-2, 3, size=shapes["mask"]).astype(np.float64)
    mask[rng.random(shapes["mask"]) < 0.05] = np.nan
    mask[rng.random(shapes["mask"]) < 0.05] = -0.0
    arrays = []
    for spec, v in zip(prog.inputs, (a, W, e, b, y, mask)):
        arrays.append(S.to_storage(v, dt).reshape(spec.shape))
    return arrays


@pytest.mark.parametrize("forms,bn", [(0, 64), (0, 128), (0, 224), (0, 256), (1, 256), (2, 64)])
@pytest.mark.parametrize("dt", ["bfloat16", "float16"])
def test_gemm_epilogue_edge_values_bit_exact(dt, forms, bn):
    prog = gemm_program(dt)
    arrays = gemm_inputs(prog, dt, seed=29)
    gpu, st = run_step(prog, arrays, expr_forms=forms, tile_n=bn)
    tiles = [t for t in st.tasks() if t["kind"] == "gemm_tc"]
    # 224-wide tiles where B is K-major (ragged: 224 + 32 columns); the input
    # gradient's MN-major B takes 256
    mn_major_b = {"ga"}
    assert len(tiles) == 4
    assert all(t["tile_n"] == (256 if bn == 224 and t["op"] in mn_major_b else bn) for t in tiles)
    assert sum(t["side_output"] for t in tiles) == 2
    if forms == 0:
        # with 256-wide tiles in the launch the ring leaves no room to stage
        # the loaded side's operand: that tile keeps direct accesses
        assert all(t["staged_epilogue"] for t in tiles[:3])
        assert tiles[3]["staged_epilogue"] == (bn <= 128)
    want = oracle.run_program(prog, values(arrays, prog))
    for spec, g, w in zip(prog.outputs, gpu, want):
        assert_bit_exact(g, w, spec.dtype, (spec.buffer, dt, forms, bn))
