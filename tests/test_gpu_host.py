"""Steps fed from host memory (tk_run_host): each step's batch (x, y) is
copied from page-locked host memory on the library's copy stream, into two
device buffers used alternately, while the previous step computes; the loss
of every step is copied back.  The final state and every step's loss must be
bit-identical to the same steps run one by one (tk_run) with the batches
copied in by the caller, and the host-side checks must reject bad calls
before anything is enqueued."""
import numpy as np
import pytest
import torch

from persistent_step_megakernel_gb300 import binding as B
from persistent_step_megakernel_gb300 import synthetic as S
from persistent_step_megakernel_gb300.build import build
from persistent_step_megakernel_gb300.runtime import TrainStep
from tests._util import to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def batches(prog, arrays, n, seed):
    """n different (x, y) batches: the workload's own scaled by per-step factors."""
    names = [s.buffer for s in prog.inputs]
    idx = [names.index("x")] + ([names.index("y")] if "y" in names else [])
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        f = rng.uniform(0.5, 1.5)
        out.append([to_torch(arrays[i], prog.inputs[i].dtype, "cpu").mul_(f).contiguous() for i in idx])
    return idx, out


@pytest.mark.parametrize("key,n", [("c2", 5), ("c3", 4), ("c4", 3), ("c5", 3)])
def test_host_fed_steps_bit_identical_to_steps_one_by_one(key, n):
    cfg = S.CONFIGS[key]
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    idx, host = batches(prog, arrays, n, seed=7)

    # one by one: the caller copies each batch in, runs the step, reads the loss
    step = TrainStep(prog, 0)
    ins = [to_torch(a, s.dtype, "cuda") for a, s in zip(arrays, prog.inputs)]
    outs, ws = step.allocate(ins)
    want_loss = []
    for s in range(n):
        for b, i in enumerate(idx):
            ins[i].copy_(host[s][b])
        step.run(ins, outs, ws)
        want_loss.append(outs[0].clone())
    torch.cuda.synchronize()
    assert step.status(ws)[0] == 0
    want_state = [o.clone() for o in outs]

    # fed from page-locked host memory through tk_run_host
    step2 = TrainStep(prog, 0)
    ins2 = [to_torch(a, s.dtype, "cuda") for a, s in zip(arrays, prog.inputs)]
    outs2, ws2 = step2.allocate(ins2)
    pinned = [[t.pin_memory() for t in hb] for hb in host]
    alt = [torch.empty_like(ins2[i]) for i in idx]
    loss_host = torch.empty((n,) + tuple(outs2[0].shape), dtype=outs2[0].dtype).pin_memory()
    step2.run_host(ins2, outs2, ws2, idx, alt, pinned, [0], [[loss_host[s]] for s in range(n)])
    torch.cuda.synchronize()
    assert step2.status(ws2)[0] == 0
    for s in range(n):
        assert torch.equal(loss_host[s], want_loss[s].cpu()), s
    for spec, x, y in zip(prog.outputs, outs2, want_state):
        assert torch.equal(x, y), spec.buffer
    # a second call continues from the state the first one left
    step2.run_host(ins2, outs2, ws2, idx, alt, pinned[:1], [0], [[loss_host[0]]])
    for b, i in enumerate(idx):
        ins[i].copy_(host[0][b])
    step.run(ins, outs, ws)
    torch.cuda.synchronize()
    assert torch.equal(loss_host[0], outs[0].cpu())
    for spec, x, y in zip(prog.outputs, outs2, outs):
        assert torch.equal(x, y), spec.buffer


def test_host_fed_steps_reject_bad_calls_before_enqueueing():
    cfg = S.CONFIGS["c2"]
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    step = TrainStep(prog, 0)
    ins = [to_torch(a, s.dtype, "cuda") for a, s in zip(arrays, prog.inputs)]
    outs, ws = step.allocate(ins)
    names = [s.buffer for s in prog.inputs]
    x = names.index("x")
    inplace_target = sorted(prog.inplace.values())[0]      # a parameter updated in place
    hx = ins[x].cpu().pin_memory()
    P = lambda ts: [t.data_ptr() for t in ts]

    def call(batch, alt, host, n=1):
        B.tk_run_host(step.handle, n, P(ins), P(outs), batch, alt, host, [], [], ws.data_ptr(), ws.numel(),
                      torch.cuda.current_stream().cuda_stream)

    alt = torch.empty_like(ins[x])
    with pytest.raises(B.TkError) as e:          # the alternate buffer is another input
        call([x], [ins[inplace_target].data_ptr()], [hx.data_ptr()])
    assert B.STATUS[e.value.status] in ("TK_ERR_ALIAS", "TK_ERR_INVALID")
    with pytest.raises(B.TkError) as e:          # an in-place target cannot be a batch input
        call([inplace_target], [alt.data_ptr()], [hx.data_ptr()])
    assert B.STATUS[e.value.status] == "TK_ERR_INVALID"
    with pytest.raises(B.TkError) as e:          # NULL host batch
        call([x], [alt.data_ptr()], [0])
    assert B.STATUS[e.value.status] == "TK_ERR_INVALID"
    with pytest.raises(B.TkError) as e:          # input index out of range
        call([len(ins)], [alt.data_ptr()], [hx.data_ptr()])
    assert B.STATUS[e.value.status] == "TK_ERR_INVALID"
    # nothing ran: the workspace header is still clean and the state unchanged
    torch.cuda.synchronize()
    assert step.status(ws)[0] == 0
    for a, t, s in zip(arrays, ins, prog.inputs):
        assert torch.equal(t, to_torch(a, s.dtype, "cuda")), s.buffer


def test_host_fed_steps_without_batch_inputs_only_read_results_back():
    # no batch input: the steps run on the resident inputs and only the loss
    # of every step comes back; zero steps enqueue nothing
    cfg = S.CONFIGS["c2"]
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    step = TrainStep(prog, 0)
    ins = [to_torch(a, s.dtype, "cuda") for a, s in zip(arrays, prog.inputs)]
    outs, ws = step.allocate(ins)
    want = []
    for _ in range(3):
        step.run(ins, outs, ws)
        want.append(outs[0].cpu())
    step2 = TrainStep(prog, 0)
    ins2 = [to_torch(a, s.dtype, "cuda") for a, s in zip(arrays, prog.inputs)]
    outs2, ws2 = step2.allocate(ins2)
    loss_host = torch.empty((3,) + tuple(outs2[0].shape), dtype=outs2[0].dtype).pin_memory()
    step2.run_host(ins2, outs2, ws2, [], [], [], [0], [[loss_host[s]] for s in range(3)])
    step2.run_host(ins2, outs2, ws2, [], [], [], [], [])
    torch.cuda.synchronize()
    assert step2.status(ws2)[0] == 0
    for s in range(3):
        assert torch.equal(loss_host[s], want[s]), s
    for spec, x, y in zip(prog.outputs, outs2, outs):
        assert torch.equal(x, y), spec.buffer
