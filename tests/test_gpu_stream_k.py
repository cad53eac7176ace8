"""Stream-K stages: equal ranges of k blocks per block, a tile cut in two
finished by adding the next block's fp32 partial sum.

The cut points follow the grid size, so a stream-K GEMM adds its products in
another order than whole tiles do; it must still meet the per-op parity with
the oracle (teacher-forced), stay within the same bound of the whole-tile
result, and give the same bits on every run with the same grid.
"""
import numpy as np
import pytest

from persistent_step_megakernel_gb300 import synthetic as S
from persistent_step_megakernel_gb300.build import build
from persistent_step_megakernel_gb300.ir import Operation, Program, TensorSpec
from tests._gpu import run_step, teacher_forced
from tests._util import ulp_distance, ulp_of, values

pytestmark = pytest.mark.gpu
T = TensorSpec.contiguous


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def sk_tasks(step):
    return [t for t in step.tasks() if t["kind"] == "gemm_tc" and t["stream_k"]]


def gemm_program(m, n, k, dt="bfloat16"):
    """A forward layer (bias + ReLU) and a second GEMM on its result."""
    a, w, b, w2 = T("a", (m, k), dt), T("W", (n, k), dt), T("b", (n,), dt), T("W2", (n, n), dt)
    ops = [Operation("z", "addmm", (b, a, w.T), T("z", (m, n), dt)),
           Operation("h", "relu", (T("z", (m, n), dt),), T("h", (m, n), dt)),
           Operation("o", "mm", (T("h", (m, n), dt), w2.T), T("o", (m, n), dt))]
    return Program([a, w, b, w2], [T("h", (m, n), dt), T("o", (m, n), dt)], ops)


def inputs(prog, seed):
    return [S.to_storage(S.normal(S.stream_seed(seed, i), int(np.prod(s.shape)), 0.0, 0.5), s.dtype).reshape(s.shape)
            for i, s in enumerate(prog.inputs)]


@pytest.mark.parametrize("grid", [24, 37, 61])
def test_stream_k_gemm_matches_oracle_and_whole_tiles(grid):
    # 1024^3 in 128 x 128 tiles: 64 tiles of 16 k blocks over `grid` blocks
    # leave a partly idle last wave, so both GEMMs run stream-K; the three grid
    # sizes move the cut points (tiles cut at different k blocks)
    prog = gemm_program(1024, 1024, 1024)
    arrays = inputs(prog, 41)
    sk, st = run_step(prog, arrays, tile_n=128, max_blocks=grid, split_k=0)
    assert len(sk_tasks(st)) == 2 and st.stats["grid_blocks"] == grid
    again, _ = run_step(prog, arrays, tile_n=128, max_blocks=grid, split_k=0)
    for x, y in zip(sk, again):
        np.testing.assert_array_equal(x, y)                         # deterministic for a grid
    whole, sw = run_step(prog, arrays, tile_n=128, max_blocks=grid, split_k=0, stream_k=0)
    assert not sk_tasks(sw)
    # the first GEMM's output differs only by its float32 summation order: each
    # is within the float32 summation bound K 2^-24 sum|a w| (plus the final
    # rounding) of the exact value, so the two are within twice that; sums
    # that nearly cancel may differ by many ulp of their small value
    av, wv, bv = (np.abs(v) for v in values(arrays, prog)[:3])
    bound = 2 * 1.01 * 1024 * 2.0 ** -24 * (av @ wv.T + bv) + 2 * ulp_of(whole[0], "bfloat16")
    assert (np.abs(sk[0] - whole[0]) <= bound).all()
    u = ulp_distance(sk[0], whole[0], "bfloat16")
    assert (u <= 2).mean() >= 0.999
    all_prog = Program(prog.inputs, [T("z", (1024, 1024), "bfloat16")] + list(prog.outputs), prog.operations)
    outs, sa = run_step(all_prog, arrays, tile_n=128, max_blocks=grid, split_k=0)
    assert sk_tasks(sa)
    teacher_forced(all_prog, arrays, outs)


def test_stream_k_in_the_gemm_bound_step():
    # the bf16 GEMM-bound step on two layers of the full width: the forward
    # stages (tensor-core tiles only) run stream-K; every op against the oracle
    cfg = S.scaled(S.CONFIGS["c5"], dims=(4096, 4096, 4096))
    prog = S.mlp_step_program(cfg, export="all")
    arrays = S.mlp_inputs(cfg, prog)
    outs, st = run_step(prog, arrays)
    names = {prog.operations[t["op_index"]].name for t in sk_tasks(st)}
    assert "z1" in names
    teacher_forced(prog, arrays, outs, sample=2048)
    # the timed program: stream-K against whole tiles, state after a step
    state = S.mlp_step_program(S.CONFIGS["c5"], export="state")
    arrays = S.mlp_inputs(S.CONFIGS["c5"], state)
    a, sa = run_step(state, arrays)
    b, _ = run_step(state, arrays, stream_k=0)
    assert sk_tasks(sa)
    assert abs(a[0] - b[0]) <= 1e-2 * abs(b[0])                    # loss
    # not teacher-forced: the forward GEMMs' other summation order carries
    # through the layers into the gradients' cancelling column sums, so this
    # is the end-to-end tracking bound (per-op parity is checked above)
    for slot in state.inplace:
        name = state.outputs[slot].buffer
        if name.startswith("W"):
            u = ulp_distance(a[slot], b[slot], "bfloat16")
            assert (u <= 2).mean() >= 0.99 and u.max() <= 64, (name, (u <= 2).mean(), u.max())
        else:
            # the biases start at 0 and move by lr times a cancelling column
            # sum: compare on the scale of the update, not in ulps
            assert np.abs(a[slot] - b[slot]).max() <= 0.02 * np.abs(b[slot]).max(), name
