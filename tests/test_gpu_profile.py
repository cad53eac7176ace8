"""The kernel's per-stage %globaltimer stamps (programs created with profile=1):
every stage's events are ordered as the pipeline orders them, and profiling
changes no result."""
import numpy as np
import pytest
import torch

from persistent_step_megakernel_gb300 import synthetic as S
from persistent_step_megakernel_gb300.build import build
from persistent_step_megakernel_gb300.runtime import TrainStep
from tests._gpu import run_step
from tests._util import to_f64, to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def test_stage_stamps_follow_the_pipeline_order():
    cfg = S.CONFIGS["c2"]
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    plain, _ = run_step(prog, arrays)
    step = TrainStep(prog, 0, profile=1)
    ins = [to_torch(a, s.dtype, "cuda") for a, s in zip(arrays, prog.inputs)]
    outs, ws = step.allocate(ins)
    step.run(ins, outs, ws)
    torch.cuda.synchronize()
    assert step.status(ws)[0] == 0
    for spec, x, y in zip(prog.outputs, plain, outs):
        np.testing.assert_array_equal(x, to_f64(y), err_msg=spec.buffer)

    st = step.stats
    prof = step.profile(ws)
    stamps = prof["stamps"]
    assert st["stages"] > 1
    assert len(stamps) == st["stages"] and all(len(row) == st["grid_blocks"] for row in stamps)
    tiles = 0
    for s, row in enumerate(stamps):
        for r in row:
            assert len(r) == 9
            begin, arrive = r[0], r[1]
            assert 0 < begin <= arrive
            if r[3] > 0:  # a block with tensor-core tiles in this stage
                tiles += 1
                # first operand tile, first accumulator, last store issued,
                # stores complete: in that order, inside the stage
                assert begin <= r[3] <= r[5] <= r[8] <= r[6] <= arrive
                assert begin <= r[2] <= arrive and begin <= r[4] <= arrive
        if s + 1 < len(stamps):
            # every block reaches barrier s before any block starts stage s + 1
            assert max(r[1] for r in row) <= min(r[0] for r in stamps[s + 1])
    assert tiles > 0
    assert all(w > 0 for w in prof["work_us"]) and all(b >= 0 for b in prof["barrier_us"])
