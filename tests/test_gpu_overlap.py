"""Reductions run beside the tensor-core tiles (`overlap_reductions`: 1 where
the planner estimates they fit in the tiles' time, the default; 2 for every
eligible one): warps 2 and 3 of each block take a stage's compiled row and
column reductions while the tiles run, emulating the eight warps of the
routines that otherwise run after the tiles.  Every output must be
bit-identical either way: split and unsplit losses and bias gradients, the
SGD and momentum updates fused after them, bf16 and fp16."""
import numpy as np
import pytest
import torch

from persistent_step_megakernel_gb300 import synthetic as S
from persistent_step_megakernel_gb300.build import build
from tests._gpu import run_step
from tests.test_gpu_tiles import WIDE, run_on_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


CASES = {
    "c2": S.CONFIGS["c2"],
    "c4": S.CONFIGS["c4"],            # unsplit reductions with the SGD update fused after them
    "c2b1": S.CONFIGS["c2b1"],
    "wide_bf16": WIDE["wide_bf16"],
    "wide_f16_mom": WIDE["wide_f16_mom"],  # fp16, momentum on the bias gradients
    "c3": S.CONFIGS["c3"],
}


@pytest.mark.parametrize("export,steps", [("state", 2), ("grads", 1)])
@pytest.mark.parametrize("key", list(CASES))
def test_reductions_beside_tiles_bit_identical(key, export, steps):
    cfg = CASES[key]
    prog = S.mlp_step_program(cfg, export=export)
    arrays = S.mlp_inputs(cfg, prog)
    beside, sb = run_step(prog, arrays, steps=steps, overlap_reductions=2)
    after, sa = run_step(prog, arrays, steps=steps, overlap_reductions=0)
    assert any(t["beside_tiles"] for t in sb.tasks())
    assert not any(t["beside_tiles"] for t in sa.tasks())
    for spec, x, y in zip(prog.outputs, beside, after):
        np.testing.assert_array_equal(x, y, err_msg=(key, export, spec.buffer))


def test_full_gemm_bound_step_reductions_beside_tiles_bit_identical():
    # the split loss (304 parts) and the split bias gradients of the 4096-wide
    # layers, each beside a stage of 4096^3 GEMM tiles
    cfg = S.CONFIGS["c5"]
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    beside, sb = run_on_device(prog, arrays, steps=2)      # the default plan
    after, _ = run_on_device(prog, arrays, steps=2, overlap_reductions=0)
    assert sum(t["beside_tiles"] for t in sb.tasks()) == 4
    for spec, x, y in zip(prog.outputs, beside, after):
        assert torch.equal(x, y), spec.buffer


def test_every_reduction_beside_the_tiles_with_folded_finals_bit_identical():
    # forced: gb4 beside the tiles too; the finals of gb4, gb3 and gb2 fold
    # into their partials' stages (48 of the 59 chunk counters), gb1's does
    # not fit and keeps a stage of its own
    cfg = S.CONFIGS["c5"]
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    forced, sf = run_on_device(prog, arrays, steps=3, overlap_reductions=2)
    after, _ = run_on_device(prog, arrays, steps=3, overlap_reductions=0)
    folded = sorted(prog.operations[t["op_index"]].name for t in sf.tasks() if t["folded"])
    assert folded == ["gb2", "gb3", "gb4"]
    for spec, x, y in zip(prog.outputs, forced, after):
        assert torch.equal(x, y), spec.buffer
