"""tk_run_static: the entry point with a built-in workspace, for callers that
cannot allocate device memory where they run a step (inside a stream capture,
under a runtime whose memory another allocator owns, or when a host framework
hands over only input/output pointers).

It must give the same bits as tk_run with a caller-allocated workspace -- the
kernel is deterministic (fixed summation orders everywhere), so any difference
means a stale read -- on two calls in a row, with the built-in array left full
of another program's values in between (the array keeps the previous call's
contents).  It must refuse a program whose workspace does not fit its 8 MiB.
The file is named so that pytest collects it last; it needs no other test to
run first.
"""
import numpy as np
import pytest
import torch

from persistent_step_megakernel_gb300 import binding as B
from persistent_step_megakernel_gb300 import synthetic as S
from persistent_step_megakernel_gb300.build import build
from persistent_step_megakernel_gb300.runtime import TrainStep
from tests._util import to_f64, to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def _static_run(step, ins, outs):
    B.tk_run_static(step.handle, [t.data_ptr() for t in ins], [o.data_ptr() for o in outs],
                    torch.cuda.current_stream().cuda_stream)


def _fill_array_with_another_program(key):
    """Run a different workload through the built-in array (fresh buffers)."""
    cfg = S.CONFIGS[key]
    prog = S.mlp_step_program(cfg, export="all")
    step = TrainStep(prog, 0)
    ins = [to_torch(a, s.dtype, "cuda") for a, s in zip(S.mlp_inputs(cfg, prog, seed=5), prog.inputs)]
    outs, _ = step.allocate(ins)
    _static_run(step, ins, outs)


@pytest.mark.parametrize("key,other", [("c1", "c2"), ("c2", "c4"), ("c4", "c2"), ("c2b1", "c1")])
def test_static_workspace_matches_caller_workspace_on_two_calls(key, other):
    cfg = S.CONFIGS[key]
    prog = S.mlp_step_program(cfg, export="grads")
    arrays = S.mlp_inputs(cfg, prog)
    step = TrainStep(prog, 0)
    assert step.workspace_elements <= B.STATIC_WORKSPACE_ELEMENTS
    # two independent copies of the state: one per entry point
    ins_a = [to_torch(a, s.dtype, "cuda") for a, s in zip(arrays, prog.inputs)]
    ins_b = [to_torch(a, s.dtype, "cuda") for a, s in zip(arrays, prog.inputs)]
    outs_a, ws = step.allocate(ins_a)
    outs_b, _ = step.allocate(ins_b)
    for call in range(2):
        step.run(ins_a, outs_a, ws)
        _static_run(step, ins_b, outs_b)
        torch.cuda.synchronize()
        assert step.status(ws) == (0, 0)
        for spec, a, b in zip(prog.outputs, outs_a, outs_b):
            np.testing.assert_array_equal(to_f64(b), to_f64(a), err_msg=f"call {call}: {spec.buffer}")
        _fill_array_with_another_program(other)


def test_static_workspace_rejects_programs_that_do_not_fit():
    cfg = S.scaled(S.CONFIGS["c3"], batch=1024)  # needs ~21 MB of workspace
    prog = S.mlp_step_program(cfg, export="state")
    step = TrainStep(prog, 0)
    assert step.workspace_elements > B.STATIC_WORKSPACE_ELEMENTS
    arrays = S.mlp_inputs(cfg, prog)
    ins = [to_torch(a, s.dtype, "cuda") for a, s in zip(arrays, prog.inputs)]
    outs, _ = step.allocate(ins)
    with pytest.raises(B.TkError, match="built-in one holds 2097152") as e:
        _static_run(step, ins, outs)
    assert e.value.status == 3
