"""Parity of the tensor-core tile widths and of the full-size workloads.

The planner picks a 64-, 128- or 256-wide N tile per GEMM from its tile count
and the SM count, so small parity shapes only reach the 64-wide path.  Here
`tile_n` forces each width on moderate shapes (ragged M, N and K tails,
K-major and MN-major operands in one-box-per-slab and slab-box form, the
staged epilogue with a side output), and the full-size fp16 FFN block and
bf16 GEMM-bound step run with the tiles the planner picks for them:
  * teacher-forced per-op parity with the oracle (all-outputs program);
  * the fused program bit-identical to the unfused one at the same tiles;
  * the timed (state) program bit-identical to its unfused plan over steps.
"""
import numpy as np
import pytest
import torch

from persistent_step_megakernel_gb300 import synthetic as S
from persistent_step_megakernel_gb300.build import build
from persistent_step_megakernel_gb300.runtime import TrainStep
from tests._gpu import run_step, teacher_forced
from tests._util import to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


WIDE = {
    # 3 M tiles; N = 768 / 640 / 320 (ragged at 256); every width divides by 64 (slab boxes)
    "wide_bf16": S.scaled(S.CONFIGS["c2"], batch=384, dims=(512, 768, 640, 320)),
    # ragged M (200) and a ragged last k block in the weight gradients (K = 200);
    # N = 136 is not a multiple of 64, so MN-major operands load one box per slab
    "wide_bf16_ragged": S.scaled(S.CONFIGS["c2"], batch=200, dims=(256, 384, 136)),
    # fp16, residual loss and momentum
    "wide_f16_mom": S.scaled(S.CONFIGS["c3"], batch=256, dims=(512, 1024, 512)),
}


def tc_tasks(step):
    return [t for t in step.tasks() if t["kind"] == "gemm_tc"]


def widths_ok(tiles, bn):
    # forcing 224 gives 224-wide tiles where B is K-major (the forward GEMMs)
    # and 256 elsewhere (the backward GEMMs read B along its rows)
    if bn != 224:
        return all(t["tile_n"] == bn for t in tiles)
    fwd = [t for t in tiles if t["op"].startswith("z")]
    return fwd and all(t["tile_n"] == 224 for t in fwd) and all(t["tile_n"] in (224, 256) for t in tiles)


@pytest.mark.parametrize("bn", [128, 224, 256])
@pytest.mark.parametrize("key", list(WIDE))
def test_wide_tiles_each_op_matches_oracle_teacher_forced(key, bn):
    cfg = WIDE[key]
    prog = S.mlp_step_program(cfg, export="all")
    arrays = S.mlp_inputs(cfg, prog)
    outs, step = run_step(prog, arrays, tile_n=bn)
    tiles = tc_tasks(step)
    assert tiles and widths_ok(tiles, bn)
    report = []
    teacher_forced(prog, arrays, outs, report=report)
    assert any(op.startswith("gW") for op, _, _ in report)


@pytest.mark.parametrize("bn", [128, 224, 256])
@pytest.mark.parametrize("key", list(WIDE))
def test_wide_tiles_fused_bit_identical_to_unfused(key, bn):
    # the fused plan runs the staged epilogue (with the loss gradient as a
    # side output of the output layer's GEMM); the unfused one stores every op
    cfg = WIDE[key]
    fused = S.mlp_step_program(cfg, export="grads")
    unfused = S.mlp_step_program(cfg, export="all")
    arrays = S.mlp_inputs(cfg, fused)
    a, sa = run_step(fused, arrays, tile_n=bn)
    b, _ = run_step(unfused, arrays, tile_n=bn, fuse_epilogues=0)
    tiles = tc_tasks(sa)
    assert widths_ok(tiles, bn)
    assert any(t["staged_epilogue"] for t in tiles)
    if cfg.loss == "mse":
        assert any(t["staged_epilogue"] and t["side_output"] for t in tiles)
    names_b = {s.buffer: v for s, v in zip(unfused.outputs, b)}
    for s, v in zip(fused.outputs, a):
        np.testing.assert_array_equal(v, names_b[s.buffer], err_msg=s.buffer)


@pytest.mark.parametrize("bn", [128, 224, 256])
@pytest.mark.parametrize("key", list(WIDE))
def test_wide_tiles_state_program_fused_matches_unfused_over_steps(key, bn):
    cfg = WIDE[key]
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    fused, _ = run_step(prog, arrays, steps=2, tile_n=bn)
    plain, _ = run_step(prog, arrays, steps=2, tile_n=bn, fuse_epilogues=0, fuse_pointwise=0)
    for spec, x, y in zip(prog.outputs, fused, plain):
        np.testing.assert_array_equal(x, y, err_msg=spec.buffer)


@pytest.mark.parametrize("key", ["wide_f16_mom", "wide_bf16"])
def test_staging_ring_depths_bit_identical(key):
    # the deepest staging rings (all chunks of a momentum tile in flight, the
    # loss gradient in buffers of its own) against depth 2 with the side values
    # written in place, over two steps of the timed program and the grads one
    cfg = WIDE[key]
    for export, steps in (("state", 2), ("grads", 1)):
        prog = S.mlp_step_program(cfg, export=export)
        arrays = S.mlp_inputs(cfg, prog)
        deep, sd = run_step(prog, arrays, steps=steps, tile_n=128)
        flat, sf = run_step(prog, arrays, steps=steps, tile_n=128, epi_stage_bytes=8192)
        deep_d = [t["staged_depth"] for t in tc_tasks(sd)]
        flat_d = [t["staged_depth"] for t in tc_tasks(sf)]
        assert all(f & 15 <= d & 15 for d, f in zip(deep_d, flat_d))
        assert any(f & 15 < d & 15 for d, f in zip(deep_d, flat_d)), (deep_d, flat_d)
        # with the cap, staged side outputs (the momentum step's W', the loss
        # gradient) run at depth 2, the unary one in place
        assert all(t["staged_depth"] in (0, 2) for t in tc_tasks(sf) if t["side_output"])
        for spec, x, y in zip(prog.outputs, deep, flat):
            np.testing.assert_array_equal(x, y, err_msg=(export, spec.buffer))


# ------------------------------------------------------------ full sizes

def run_on_device(program, arrays, steps=1, **opts):
    """Like run_step, but the outputs stay on the device (large programs)."""
    step = TrainStep(program, 0, **opts)
    ins = [to_torch(a, s.dtype, "cuda") for a, s in zip(arrays, program.inputs)]
    outs, ws = step.allocate(ins)
    for _ in range(steps):
        step.run(ins, outs, ws)
    torch.cuda.synchronize()
    status, stage = step.status(ws)
    assert status == 0, f"device status {status} at stage {stage}"
    return outs, step


def test_full_ffn_block_each_op_matches_oracle_teacher_forced():
    cfg = S.CONFIGS["c3"]
    prog = S.mlp_step_program(cfg, export="all")
    arrays = S.mlp_inputs(cfg, prog)
    outs, step = run_step(prog, arrays)
    assert tc_tasks(step)
    teacher_forced(prog, arrays, outs)


def test_full_ffn_block_fused_bit_identical_to_unfused():
    cfg = S.CONFIGS["c3"]
    fused = S.mlp_step_program(cfg, export="grads")
    unfused = S.mlp_step_program(cfg, export="all")
    arrays = S.mlp_inputs(cfg, fused)
    a, _ = run_step(fused, arrays)
    b, _ = run_step(unfused, arrays, fuse_epilogues=0)
    names_b = {s.buffer: v for s, v in zip(unfused.outputs, b)}
    for s, v in zip(fused.outputs, a):
        np.testing.assert_array_equal(v, names_b[s.buffer], err_msg=s.buffer)


@pytest.mark.parametrize("key", ["c3", "c5"])
def test_full_timed_program_fused_matches_unfused_over_steps(key):
    # the program the benchmark times, against its plan with no fusion at all
    cfg = S.CONFIGS[key]
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    fused, sf = run_on_device(prog, arrays, steps=2)
    plain, sp = run_on_device(prog, arrays, steps=2, fuse_epilogues=0, fuse_pointwise=0)
    widths = {t["op"]: t["tile_n"] for t in tc_tasks(sf)}
    assert widths == {t["op"]: t["tile_n"] for t in tc_tasks(sp)}
    if key == "c5":
        # forward GEMMs 4 full waves of 224-wide tiles, backward 256-wide
        assert {t["tile_n"] for t in tc_tasks(sf) if t["op"].startswith("z")} == {224}
        assert {t["tile_n"] for t in tc_tasks(sf) if not t["op"].startswith("z")} == {256}
    for spec, x, y in zip(prog.outputs, fused, plain):
        assert torch.equal(x, y), spec.buffer


# Two layers of the GEMM-bound step: every GEMM has the full 4096 x 4096 x 4096
# shape and the planner's tiles (128 x 224 forward: 19 column tiles, the last
# with 64 live columns; 128 x 256 backward): forward with ReLU, the output
# layer with the MSE epilogue and its side output, weight and input gradients
# with the ReLU mask, the fused SGD updates.
C5_TWO = S.scaled(S.CONFIGS["c5"], dims=(4096, 4096, 4096))


def test_full_gemm_bound_each_op_matches_oracle_teacher_forced():
    prog = S.mlp_step_program(C5_TWO, export="all")
    arrays = S.mlp_inputs(C5_TWO, prog)
    outs, step = run_step(prog, arrays)
    assert {t["tile_n"] for t in tc_tasks(step)} == {224, 256}
    teacher_forced(prog, arrays, outs, sample=2048)


def test_full_gemm_bound_fused_bit_identical_to_unfused():
    fused = S.mlp_step_program(C5_TWO, export="grads")
    unfused = S.mlp_step_program(C5_TWO, export="all")
    arrays = S.mlp_inputs(C5_TWO, fused)
    a, sa = run_on_device(fused, arrays)
    b, _ = run_on_device(unfused, arrays, fuse_epilogues=0)
    tiles = tc_tasks(sa)
    assert any(t["staged_epilogue"] and t["side_output"] and t["tile_n"] == 224 for t in tiles)
    names_b = {s.buffer: v for s, v in zip(unfused.outputs, b)}
    for s, v in zip(fused.outputs, a):
        assert torch.equal(v, names_b[s.buffer]), s.buffer
