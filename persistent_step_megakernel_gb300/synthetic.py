"""Seeded synthetic workloads: MLP training-step programs and their inputs.

This module is shared by the CPU oracle's tests and the CUDA path's tests and
benchmark.  It holds the workload only -- a counter-based random generator, the
initialisation recipes and the op list of one functional MLP training step --
and none of the method's arithmetic (no rounding, no matmul, no reduction).

Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): output k of a stream with seed s is mix(s + k*gamma)
with gamma = 0x9E3779B97F4A7C15.  Uniforms take the top 53 bits; normals use
the Box-Muller transform on consecutive pairs.

Low-precision inputs: values are drawn in float64, converted to float32, and
then stored as float16 by numpy's conversion or as bfloat16 by keeping the upper
16 bits of the float32 pattern (truncation).  Either way the stored value is
exactly representable in its dtype, which is all the step requires.
"""
from __future__ import annotations

from dataclasses import dataclass
import math

import numpy as np

from .ir import Operation, Program, TensorSpec

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start..start+n-1 of the SplitMix64 stream with the given seed."""
    with np.errstate(over="ignore"):
        k = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + k * _GAMMA)


def stream_seed(seed: int, index: int) -> int:
    """Seed of the index-th independent tensor stream of a workload seed."""
    return int(splitmix64((seed * 0x100000001B3 + index) & 0xFFFFFFFFFFFFFFFF, 1)[0])


def uniform01(seed: int, n: int) -> np.ndarray:
    """n doubles in [0, 1) from the top 53 bits of each SplitMix64 output."""
    return (splitmix64(seed, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """Box-Muller normals: pair j uses outputs 2j (radius) and 2j+1 (angle)."""
    pairs = (n + 1) // 2
    u = uniform01(seed, 2 * pairs).reshape(pairs, 2)
    r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))          # 1-u in (0, 1]
    theta = 2.0 * math.pi * u[:, 1]
    z = np.stack([r * np.cos(theta), r * np.sin(theta)], axis=1).reshape(-1)[:n]
    return mean + std * z


def uniform(seed: int, n: int, bound: float) -> np.ndarray:
    return (2.0 * uniform01(seed, n) - 1.0) * bound


def to_storage(values: np.ndarray, dtype: str) -> np.ndarray:
    """float64 draws -> the array a caller would hand the step in that dtype.

    float32 -> np.float32, float16 -> np.float16, bfloat16 -> np.uint16 bit
    patterns (upper half of the float32 pattern).
    """
    f32 = np.asarray(values, dtype=np.float64).astype(np.float32)
    if dtype == "float32":
        return f32
    if dtype == "float16":
        return f32.astype(np.float16)
    if dtype == "bfloat16":
        return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    raise ValueError(f"unsupported dtype {dtype}")


def storage_to_float64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of a stored array back to float64 values."""
    if dtype == "bfloat16":
        return (arr.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return arr.astype(np.float64)


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class MLPConfig:
    key: str
    description: str
    dtype: str
    batch: int
    dims: tuple            # d0 -> d1 -> ... -> dL
    lr: float
    init: str              # "torch_default" | "kaiming_uniform" | "normal002"
    loss: str = "mse"      # "mse" (targets y) | "mean_square_residual"
    momentum: float = 0.0  # > 0: SGD with a momentum buffer per parameter
    seed: int = 0
    master: str | None = None  # e.g. "float32": parameters kept in this type, GEMMs in dtype
    targets: str = "normal"    # "normal": y ~ N(0, 1); "onehot": y one-hot rows of seeded class labels

    @property
    def layers(self) -> int:
        return len(self.dims) - 1

    def flops(self) -> int:
        """Forward + weight-grad + input-grad GEMM flops (layer 1 has no input grad)."""
        per = [2 * self.batch * a * b for a, b in zip(self.dims[:-1], self.dims[1:])]
        return 2 * sum(per) + sum(per[1:])

    def compulsory_bytes(self) -> int:
        """Parameters read+written, x (+y) read, momentum read+written, loss written."""
        sizes = {"float32": 4, "float16": 2, "bfloat16": 2}
        e = sizes[self.dtype]
        pe = sizes[self.master or self.dtype]
        params = sum(a * b + b for a, b in zip(self.dims[:-1], self.dims[1:]))
        total = 2 * params * pe + self.batch * self.dims[0] * e + (4 if self.master else e)
        if self.loss == "mse":
            total += self.batch * self.dims[-1] * e
        if self.momentum:
            total += 2 * params * pe
        return total


CONFIGS = {
    "c1": MLPConfig("c1", "fp32 MLP step: batch 8, Linear(16->32)+ReLU+Linear(32->4), MSE, SGD lr=0.01",
                    "float32", 8, (16, 32, 4), 0.01, "torch_default"),
    "c2": MLPConfig("c2", "bf16 MLP step: batch 64, 256->512->512->128, ReLU, MSE, SGD lr=1e-3",
                    "bfloat16", 64, (256, 512, 512, 128), 1e-3, "kaiming_uniform"),
    "c3": MLPConfig("c3", "fp16 FFN-block step: batch 256, 1024->4096->1024 + residual, loss=mean(out^2), SGD momentum 0.9",
                    "float16", 256, (1024, 4096, 1024), 1e-3, "torch_default",
                    loss="mean_square_residual", momentum=0.9),
    "c4": MLPConfig("c4", "deep-narrow bf16 MLP step: batch 32, 16 layers of width 128, ReLU, MSE, SGD lr=1e-3",
                    "bfloat16", 32, (128,) * 17, 1e-3, "kaiming_uniform"),
    "c5": MLPConfig("c5", "GEMM-bound bf16 MLP step: batch 4096, 4 layers 4096->4096, ReLU, MSE, SGD lr=1e-4",
                    "bfloat16", 4096, (4096,) * 5, 1e-4, "normal002"),
    # the online (batch-1) step on the C2 shapes
    "c2b1": MLPConfig("c2b1", "online bf16 MLP step: batch 1, 256->512->512->128, ReLU, MSE, SGD lr=1e-3",
                      "bfloat16", 1, (256, 512, 512, 128), 1e-3, "kaiming_uniform"),
    # the mixed-precision method of the pages' harness on the C2 shapes
    "c2m": MLPConfig("c2m", "mixed-precision MLP step: fp32 master weights, bf16 GEMMs, fp32 loss and SGD; "
                     "batch 64, 256->512->512->128", "bfloat16", 64, (256, 512, 512, 128), 1e-3,
                     "kaiming_uniform", master="float32"),
    # a linear classification head trained by least squares against one-hot
    # targets, updated in place (the pages name the workload; these shapes are
    # this build's own choice)
    "lsq": MLPConfig("lsq", "one-hot least-squares classification head: bf16, batch 128, 1024 features -> "
                     "10 classes, MSE against one-hot targets, SGD lr=1e-2, in place", "bfloat16", 128, (1024, 10),
                     1e-2, "torch_default", targets="onehot"),
}


def scaled(cfg: MLPConfig, **changes) -> MLPConfig:
    """A copy of a config with some fields replaced (small parity cases)."""
    fields = dict(cfg.__dict__)
    fields.update(changes)
    return MLPConfig(**fields)


def mlp_step_program(cfg: MLPConfig, export: str = "state", dtype: str | None = None) -> Program:
    """The op list of one functional training step, in topological order.

    export: "state" -> loss and updated parameters (+ momentum buffers);
            "grads" -> additionally every weight and bias gradient;
            "all"   -> every operation's result is a program output, which
                       disables fusion and inlining (each op is materialised).
    dtype overrides the config dtype (e.g. "float64" for the oracle's
    finite-difference instantiation).
    """
    dt = dtype or cfg.dtype
    # mixed precision (the pages' harness): parameters, momentum, loss and
    # updates in the master type; GEMM operands and activations in dt
    pt = (dtype or cfg.master) if cfg.master else dt
    B, dims, L = cfg.batch, cfg.dims, cfg.layers
    T = TensorSpec.contiguous
    x = T("x", (B, dims[0]), dt)
    inputs = [x]
    y = None
    if cfg.loss == "mse":
        y = T("y", (B, dims[-1]), dt)
        inputs.append(y)
    W, b, vW, vb = {}, {}, {}, {}
    for i in range(1, L + 1):
        W[i] = T(f"W{i}", (dims[i], dims[i - 1]), pt)
        b[i] = T(f"b{i}", (dims[i],), pt)
        inputs += [W[i], b[i]]
        if cfg.momentum:
            vW[i] = T(f"vW{i}", (dims[i], dims[i - 1]), pt)
            vb[i] = T(f"vb{i}", (dims[i],), pt)
            inputs += [vW[i], vb[i]]
    ops: list[Operation] = []

    def emit(name, op, ins, shape, attrs=None, out_dtype=None):
        out = T(name, shape, out_dtype or dt)
        ops.append(Operation(name, op, tuple(ins), out, dict(attrs or {})))
        return out

    # GEMM copies of the master weights
    Wc = dict(W)
    if pt != dt:
        for i in range(1, L + 1):
            Wc[i] = emit(f"Wc{i}", "cast", (W[i],), W[i].shape)

    # forward: z_i = b_i + a_{i-1} W_i^T ; a_i = relu(z_i) between layers
    a = {0: x}
    for i in range(1, L + 1):
        z = emit(f"z{i}", "addmm", (b[i], a[i - 1], Wc[i].T), (B, dims[i]))
        a[i] = emit(f"a{i}", "relu", (z,), (B, dims[i])) if i < L else z
    out = a[L]
    n_out = B * dims[-1]
    if cfg.loss == "mse":
        d = emit("d", "sub", (out, y), (B, dims[-1]), out_dtype=pt)
        sq = emit("sq", "pow", (d, 2), (B, dims[-1]), out_dtype=pt)
        loss = emit("loss", "mean", (sq,), (), out_dtype=pt)
        g = emit(f"g{L}", "mul", (d, 2.0 / n_out if n_out else 0.0), (B, dims[-1]))
    elif cfg.loss == "mean_square_residual":
        r = emit("out", "add", (out, x), (B, dims[-1]), out_dtype=pt)
        sq = emit("sq", "pow", (r, 2), (B, dims[-1]), out_dtype=pt)
        loss = emit("loss", "mean", (sq,), (), out_dtype=pt)
        g = emit(f"g{L}", "mul", (r, 2.0 / n_out if n_out else 0.0), (B, dims[-1]))
    else:
        raise ValueError(cfg.loss)

    grads_w, grads_b, new_state = {}, {}, []
    for i in range(L, 0, -1):
        grads_w[i] = emit(f"gW{i}", "mm", (g.T, a[i - 1]), (dims[i], dims[i - 1]), out_dtype=pt)
        grads_b[i] = emit(f"gb{i}", "sum", (g,), (dims[i],), {"dims": (0,)}, out_dtype=pt)
        if i > 1:
            ga = emit(f"ga{i - 1}", "mm", (g, Wc[i]), (B, dims[i - 1]))
            g_prev = emit(f"g{i - 1}", "threshold_backward", (ga, a[i - 1]), (B, dims[i - 1]),
                          {"threshold": 0.0})
        for p, gp, v, tag in ((W[i], grads_w[i], vW.get(i), "W"), (b[i], grads_b[i], vb.get(i), "b")):
            if cfg.momentum:
                mv = emit(f"m{tag}{i}", "mul", (v, cfg.momentum), v.shape, out_dtype=pt)
                v_new = emit(f"v{tag}{i}_new", "add", (mv, gp), v.shape, out_dtype=pt)
                p_new = emit(f"{tag}{i}_new", "sub", (p, v_new), p.shape, {"alpha": cfg.lr}, out_dtype=pt)
                new_state += [(p_new, p), (v_new, v)]
            else:
                p_new = emit(f"{tag}{i}_new", "sub", (p, gp), p.shape, {"alpha": cfg.lr}, out_dtype=pt)
                new_state.append((p_new, p))
        if i > 1:
            g = g_prev

    outputs = [loss]
    inplace = {}
    for new, old in new_state:
        inplace[len(outputs)] = inputs.index(old)
        outputs.append(new)
    if export in ("grads", "all"):
        for i in range(1, L + 1):
            outputs += [grads_w[i], grads_b[i]]
    if export == "all":
        have = {o.buffer for o in outputs}
        for op in ops:
            if op.output.buffer not in have:
                outputs.append(op.output)
                have.add(op.output.buffer)
    return Program(inputs, outputs, ops, inplace)


def mlp_inputs(cfg: MLPConfig, program: Program, seed: int | None = None, dtype: str | None = None) -> list:
    """Seeded input arrays in program-input order (storage form, see to_storage).

    x ~ N(0, 1); y ~ N(0, 1), or one-hot rows of class labels drawn uniformly
    from the stream (label = floor(u * classes)); weights and biases per
    cfg.init; momentum buffers ~ N(0, 0.01^2).
    """
    seed = cfg.seed if seed is None else seed
    arrays = []
    for idx, spec in enumerate(program.inputs):
        n = int(np.prod(spec.shape)) if spec.shape else 1
        s = stream_seed(seed, idx)
        name = spec.buffer
        if name == "y" and cfg.targets == "onehot":
            classes = spec.shape[-1]
            rows = n // classes if classes else 0
            labels = np.minimum((uniform01(s, rows) * classes).astype(np.int64), classes - 1)
            vals = np.zeros((rows, classes))
            vals[np.arange(rows), labels] = 1.0
            vals = vals.reshape(-1)
        elif name in ("x", "y"):
            vals = normal(s, n)
        elif name.startswith("vW") or name.startswith("vb"):
            vals = normal(s, n, 0.0, 0.01)
        elif name.startswith("W") or name.startswith("b"):
            fan_in = program.inputs[program.inputs.index(
                next(p for p in program.inputs if p.buffer == "W" + name[1:]))].shape[1]
            if cfg.init == "torch_default":
                vals = uniform(s, n, 1.0 / math.sqrt(fan_in))
            elif cfg.init == "kaiming_uniform":
                vals = uniform(s, n, math.sqrt(6.0 / fan_in) if name[0] == "W" else 1.0 / math.sqrt(fan_in))
            elif cfg.init == "normal002":
                vals = normal(s, n, 0.0, 0.02) if name[0] == "W" else np.zeros(n)
            else:
                raise ValueError(cfg.init)
        else:
            vals = normal(s, n)
        dt = dtype or spec.dtype
        if dt == "float64":
            arrays.append(vals.reshape(spec.shape))
        else:
            arrays.append(to_storage(vals, dt).reshape(spec.shape))
    return arrays
