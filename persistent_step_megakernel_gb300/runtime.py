"""Torch-facing wrapper over the C ABI: device memory, streams and checks.

PyTorch provides the allocations and the stream; the step itself runs in the
kernel behind ``tk_run``.  The checks mirror trainkernel's runtime boundary
(page "trainkernel 0.1.0 -- trainkernel/runtime.py", `_validate_inputs`,
`allocate`, `run_into`): inputs must match the program's device, shape,
strides and dtype; outputs are fresh contiguous tensors except in-place slots,
which bind their declared input; the workspace is float32.
"""
from __future__ import annotations

import torch

from . import binding as B
from .ir import Program

TORCH_DTYPE = {"float32": torch.float32, "float16": torch.float16, "bfloat16": torch.bfloat16}


class TrainStep:
    """One planned program on one CUDA device."""

    def __init__(self, program: Program, device: int = 0, **options):
        self.program = program
        self.device = torch.device("cuda", device)
        self.options = B.options(**options)
        self.handle = B.tk_program_create(program, self.options, device)
        self.workspace_elements = B.tk_allocate(self.handle)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            B.tk_program_destroy(h)
            self.handle = None

    @property
    def stats(self) -> dict:
        return B.tk_plan_stats_get(self.handle)

    def tasks(self) -> list:
        """The plan's device tasks in stage order, each with the op name it computes."""
        out = []
        for i in range(self.stats["tasks"]):
            t = B.tk_plan_task(self.handle, i)
            t["op"] = self.program.operations[t["op_index"]].name if t["op_index"] >= 0 else None
            out.append(t)
        return out

    def resource_usage(self) -> dict:
        return B.tk_resource_usage(self.handle)

    def _stream(self, stream) -> int:
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return int(s.cuda_stream)

    def validate_inputs(self, inputs) -> None:
        if len(inputs) != len(self.program.inputs):
            raise ValueError(f"tk: expected {len(self.program.inputs)} inputs, got {len(inputs)}")
        for i, (t, spec) in enumerate(zip(inputs, self.program.inputs)):
            if not isinstance(t, torch.Tensor):
                raise TypeError(f"tk: input {i} must be a tensor")
            if (t.device != self.device or tuple(t.shape) != tuple(spec.shape)
                    or tuple(t.stride()) != tuple(spec.strides) or t.dtype != TORCH_DTYPE[spec.dtype]):
                raise ValueError(f"tk: input {i} does not match compiled device, shape, stride, or dtype")

    def allocate(self, inputs, stream=None):
        """Output tensors (in-place slots bind their input) and an initialised workspace."""
        self.validate_inputs(inputs)
        outs = []
        for j, spec in enumerate(self.program.outputs):
            if j in self.program.inplace:
                outs.append(inputs[self.program.inplace[j]])
            else:
                outs.append(torch.empty(spec.shape, dtype=TORCH_DTYPE[spec.dtype], device=self.device))
        ws = torch.empty(self.workspace_elements, dtype=torch.float32, device=self.device)
        B.tk_workspace_init(self.handle, ws.data_ptr(), ws.numel(), self._stream(stream))
        return outs, ws

    def run(self, inputs, outputs, workspace, stream=None):
        self.validate_inputs(inputs)
        for j, (o, spec) in enumerate(zip(outputs, self.program.outputs)):
            if (o.device != self.device or tuple(o.shape) != tuple(spec.shape)
                    or o.dtype != TORCH_DTYPE[spec.dtype] or not o.is_contiguous()):
                raise ValueError(f"tk: output {j} does not match compiled requirements")
        if workspace.dtype != torch.float32 or not workspace.is_contiguous() or workspace.device != self.device:
            raise ValueError("tk: workspace does not match compiled requirements")
        B.tk_run(self.handle, [t.data_ptr() for t in inputs], [o.data_ptr() for o in outputs],
                 workspace.data_ptr(), workspace.numel(), self._stream(stream))
        return outputs

    def run_host(self, inputs, outputs, workspace, batch, batch_alt, host_batches, results=(), host_results=(),
                 stream=None):
        """len(host_batches) steps fed from host memory: step s copies
        host_batches[s][b] (a host tensor, page-locked for overlap) into the
        device input named by batch[b] (an input index), alternating with
        batch_alt[b] (a second device buffer like it), and copies output
        results[r] to host_results[s][r] after the step.  The copy of step
        s+1's batch overlaps step s (tk_run_host).  Asynchronous on `stream`:
        every host tensor must stay alive until it completes."""
        self.validate_inputs(inputs)
        for j, (o, spec) in enumerate(zip(outputs, self.program.outputs)):
            if (o.device != self.device or tuple(o.shape) != tuple(spec.shape)
                    or o.dtype != TORCH_DTYPE[spec.dtype] or not o.is_contiguous()):
                raise ValueError(f"tk: output {j} does not match compiled requirements")
        if workspace.dtype != torch.float32 or not workspace.is_contiguous() or workspace.device != self.device:
            raise ValueError("tk: workspace does not match compiled requirements")
        batch, results = list(batch), list(results)
        for b, i in enumerate(batch):
            ref = inputs[i]
            for t, where in [(batch_alt[b], ref.device)] + [(hb[b], torch.device("cpu")) for hb in host_batches]:
                if (t.device != where or t.dtype != ref.dtype or tuple(t.shape) != tuple(ref.shape)
                        or not t.is_contiguous()):
                    raise ValueError(f"tk: batch buffer of input {i} does not match it")
        for s, hr in enumerate(host_results):
            for r, j in enumerate(results):
                o = outputs[j]
                if hr[r].device.type != "cpu" or hr[r].dtype != o.dtype or hr[r].numel() != o.numel():
                    raise ValueError(f"tk: host result of output {j} at step {s} does not match it")
        n_steps = len(host_batches) if batch else len(host_results)
        if results and len(host_results) != n_steps:
            raise ValueError("tk: one host result list per step")
        B.tk_run_host(self.handle, n_steps, [t.data_ptr() for t in inputs], [o.data_ptr() for o in outputs], batch,
                      [t.data_ptr() for t in batch_alt], [t.data_ptr() for hb in host_batches for t in hb], results,
                      [t.data_ptr() for hr in host_results for t in hr], workspace.data_ptr(), workspace.numel(),
                      self._stream(stream))
        return outputs

    def launcher(self, inputs, outputs, workspace, stream=None):
        """A callable that runs one step on these buffers per call, with the
        checks of run() done once here (the buffers must stay alive)."""
        self.validate_inputs(inputs)
        for j, (o, spec) in enumerate(zip(outputs, self.program.outputs)):
            if (o.device != self.device or tuple(o.shape) != tuple(spec.shape)
                    or o.dtype != TORCH_DTYPE[spec.dtype] or not o.is_contiguous()):
                raise ValueError(f"tk: output {j} does not match compiled requirements")
        if workspace.dtype != torch.float32 or not workspace.is_contiguous() or workspace.device != self.device:
            raise ValueError("tk: workspace does not match compiled requirements")
        return B.tk_run_prepared(self.handle, [t.data_ptr() for t in inputs], [o.data_ptr() for o in outputs],
                                 workspace.data_ptr(), workspace.numel(), self._stream(stream))

    def profile(self, workspace, stream=None) -> dict:
        """Per-stage timing of the last run (program created with profile=1).

        work_us[s]: first block starting stage s -> last block reaching the
        barrier after it; barrier_us[s]: last arrival at barrier s -> first
        block starting stage s+1.
        """
        st = self.stats
        stamps = B.tk_profile_read(self.handle, workspace.data_ptr(), st["stages"], st["grid_blocks"],
                                   self._stream(stream))
        begin = [min(r[0] for r in row) for row in stamps]
        arrive = [max(r[1] for r in row) for row in stamps]
        work = [(a - b) / 1e3 for b, a in zip(begin, arrive)]
        barrier = [(begin[s + 1] - arrive[s]) / 1e3 for s in range(len(stamps) - 1)]
        entry = min(r[7] for r in stamps[0])
        return {"work_us": work, "barrier_us": barrier, "total_us": (arrive[-1] - begin[0]) / 1e3,
                "prologue_us": (begin[0] - entry) / 1e3, "stamps": stamps}

    def status(self, workspace, stream=None):
        return B.tk_run_status(self.handle, workspace.data_ptr(), self._stream(stream))

    def __call__(self, *inputs):
        outs, ws = self.allocate(inputs)
        return self.run(inputs, outs, ws)
