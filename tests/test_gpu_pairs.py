"""Pair-tile launches: clusters of two blocks, every tensor-core GEMM on
256-row tiles, each block loading its 128 rows of A and half of B's columns;
`cta_pairs=1` runs cta_group::2 MMAs over both blocks' shared memory,
`cta_pairs=2` each block's own 128-row MMAs on B tiles whose halves are
multicast to both blocks.

  * a single GEMM with 128-wide tiles (the smallest tensor-memory allocation),
    then ragged shapes at every tile width, each op against the oracle;
  * the fused program bit-identical to the unfused one, both on pairs;
  * the full-size GEMM-bound layers on pairs, against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from persistent_step_megakernel_gb300 import synthetic as S
from persistent_step_megakernel_gb300.build import build
from persistent_step_megakernel_gb300.ir import Operation, Program, TensorSpec
from tests._gpu import run_step, teacher_forced
from tests._util import values
from tests.test_gpu_tiles import C5_TWO, WIDE, run_on_device, tc_tasks

pytestmark = pytest.mark.gpu
T = TensorSpec.contiguous


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def one_gemm(M, N, K, dt="bfloat16"):
    a, W = T("a", (M, K), dt), T("W", (N, K), dt)
    ops = [Operation("z", "mm", (a, W.T), T("z", (M, N), dt))]
    return Program([a, W], [T("z", (M, N), dt)], ops)


MODES = [1, 2]


@pytest.mark.parametrize("mode", MODES)
def test_single_pair_gemm_matches_oracle(mode):
    prog = one_gemm(256, 256, 128)
    rng = np.random.default_rng(5)
    # small integers: float32 accumulators exact in any order, so the result
    # is fully specified
    arrays = [S.to_storage(rng.integers(-3, 4, size=s.shape).astype(np.float64), s.dtype).reshape(s.shape)
              for s in prog.inputs]
    outs, step = run_step(prog, arrays, cta_pairs=mode, tile_n=128, barrier_timeout_s=1.0)
    assert step.stats["cta_pairs"] == mode and step.stats["grid_blocks"] % 2 == 0
    (t,) = tc_tasks(step)
    assert (t["tile_m"], t["tile_n"], t["n_items"]) == (256, 128, 2)
    want = oracle.run_program(prog, values(arrays, prog))
    np.testing.assert_array_equal(outs[0], want[0])


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("bn", [128, 224, 256])
@pytest.mark.parametrize("key", list(WIDE))
def test_pair_tiles_each_op_matches_oracle_teacher_forced(key, bn, mode):
    cfg = WIDE[key]
    prog = S.mlp_step_program(cfg, export="all")
    arrays = S.mlp_inputs(cfg, prog)
    outs, step = run_step(prog, arrays, cta_pairs=mode, tile_n=bn)
    tiles = tc_tasks(step)
    assert step.stats["cta_pairs"] == mode and all(t["tile_m"] == 256 for t in tiles)
    teacher_forced(prog, arrays, outs)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("key", list(WIDE))
def test_pair_tiles_fused_bit_identical_to_unfused(key, mode):
    cfg = WIDE[key]
    fused = S.mlp_step_program(cfg, export="grads")
    unfused = S.mlp_step_program(cfg, export="all")
    arrays = S.mlp_inputs(cfg, fused)
    a, _ = run_step(fused, arrays, cta_pairs=mode, tile_n=256)
    b, _ = run_step(unfused, arrays, cta_pairs=mode, tile_n=256, fuse_epilogues=0)
    names_b = {s.buffer: v for s, v in zip(unfused.outputs, b)}
    for s, v in zip(fused.outputs, a):
        np.testing.assert_array_equal(v, names_b[s.buffer], err_msg=s.buffer)


@pytest.mark.parametrize("mode", MODES)
def test_pair_tiles_state_program_over_steps_matches_its_unfused_plan(mode):
    cfg = WIDE["wide_f16_mom"]
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    fused, _ = run_step(prog, arrays, steps=2, cta_pairs=mode)
    plain, _ = run_step(prog, arrays, steps=2, cta_pairs=mode, fuse_epilogues=0, fuse_pointwise=0)
    for spec, x, y in zip(prog.outputs, fused, plain):
        np.testing.assert_array_equal(x, y, err_msg=spec.buffer)


@pytest.mark.parametrize("mode", MODES)
def test_full_gemm_bound_layers_on_pairs_match_oracle_teacher_forced(mode):
    prog = S.mlp_step_program(C5_TWO, export="all")
    arrays = S.mlp_inputs(C5_TWO, prog)
    outs, step = run_step(prog, arrays, cta_pairs=mode)
    assert step.stats["cta_pairs"] == mode
    assert {t["tile_n"] for t in tc_tasks(step)} == {224, 256}
    teacher_forced(prog, arrays, outs, sample=2048)


@pytest.mark.parametrize("mode", MODES)
def test_full_timed_program_on_pairs_fused_matches_unfused_over_steps(mode):
    cfg = S.CONFIGS["c5"]
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    fused, sf = run_on_device(prog, arrays, steps=2, cta_pairs=mode)
    plain, _ = run_on_device(prog, arrays, steps=2, cta_pairs=mode, fuse_epilogues=0, fuse_pointwise=0)
    assert sf.stats["cta_pairs"] == mode
    for spec, x, y in zip(prog.outputs, fused, plain):
        assert torch.equal(x, y), spec.buffer
