"""tk_run_static: the entry point with a built-in workspace, for callers that
cannot allocate device memory where they run a step (inside a stream capture,
under a runtime whose memory another allocator owns, or when a host framework
hands over only input/output pointers).

It must give the same results as tk_run with a caller-allocated workspace, on
two calls in a row (the built-in array keeps the previous call's contents), and
must refuse a program whose workspace does not fit its 8 MiB.  This file is
named to run last.
"""
import numpy as np
import pytest
import torch

from persistent_step_megakernel_gb300 import binding as B
from persistent_step_megakernel_gb300 import synthetic as S
from persistent_step_megakernel_gb300.build import build
from persistent_step_megakernel_gb300.runtime import TrainStep
from tests._util import to_f64, to_torch, ulp_distance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


@pytest.mark.parametrize("key", ["c1", "c2", "c4"])
def test_static_workspace_matches_caller_workspace_on_two_calls(key):
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
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        step.run(ins_a, outs_a, ws)
        B.tk_run_static(step.handle, [t.data_ptr() for t in ins_b], [o.data_ptr() for o in outs_b], stream)
        torch.cuda.synchronize()
        for spec, a, b in zip(prog.outputs, outs_a, outs_b):
            ga, gb = to_f64(a), to_f64(b)
            if cfg.dtype == "float32":
                np.testing.assert_allclose(gb, ga, rtol=1e-4, atol=1e-5, err_msg=f"call {call}: {spec.buffer}")
            else:
                assert ulp_distance(gb, ga, cfg.dtype).max() <= 2, (call, spec.buffer)


def test_static_workspace_rejects_programs_that_do_not_fit():
    cfg = S.scaled(S.CONFIGS["c3"], batch=1024)  # needs ~21 MB of workspace
    prog = S.mlp_step_program(cfg, export="state")
    step = TrainStep(prog, 0)
    assert step.workspace_elements > B.STATIC_WORKSPACE_ELEMENTS
    arrays = S.mlp_inputs(cfg, prog)
    ins = [to_torch(a, s.dtype, "cuda") for a, s in zip(arrays, prog.inputs)]
    outs, _ = step.allocate(ins)
    with pytest.raises(B.TkError, match="built-in one holds 2097152") as e:
        B.tk_run_static(step.handle, [t.data_ptr() for t in ins], [o.data_ptr() for o in outs],
                        torch.cuda.current_stream().cuda_stream)
    assert e.value.status == 3
