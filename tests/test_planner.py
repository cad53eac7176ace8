"""Golden planner tests (no GPU): hand-built programs whose inlining, epilogue
fusion, arena reuse and barrier placement follow from the planning rules of
trainkernel/codegen.py (`_Generator`), and the boundary's error cases."""
import pytest

from persistent_step_megakernel_gb300 import binding as B
from persistent_step_megakernel_gb300 import synthetic as S
from persistent_step_megakernel_gb300.build import build
from persistent_step_megakernel_gb300.ir import Operation, Program, TensorSpec

T = TensorSpec.contiguous


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def plan(prog, **opts):
    h = B.tk_program_create(prog, B.options(sm_count=152, **opts), device=-1)
    try:
        return B.tk_plan_stats_get(h)
    finally:
        B.tk_program_destroy(h)


def f32(name, shape):
    return T(name, shape, "float32")


def test_independent_ops_share_one_stage():
    x, y = f32("x", (4, 8)), f32("y", (4, 8))
    prog = Program([x, y], [f32("a", (4, 8)), f32("b", (4, 8))],
                   [Operation("a", "add", (x, y), f32("a", (4, 8))),
                    Operation("b", "mul", (x, y), f32("b", (4, 8)))])
    s = plan(prog)
    assert (s["materialized_ops"], s["inlined_ops"], s["stages"], s["direct_outputs"], s["output_copies"]) == (2, 0, 1, 2, 0)


def test_single_use_pointwise_is_inlined():
    x, y = f32("x", (4, 8)), f32("y", (4, 8))
    prog = Program([x, y], [f32("b", (4, 8))],
                   [Operation("a", "add", (x, y), f32("a", (4, 8))),
                    Operation("b", "mul", (f32("a", (4, 8)), 2.0), f32("b", (4, 8)))])
    s = plan(prog)
    assert (s["materialized_ops"], s["inlined_ops"], s["stages"]) == (1, 1, 1)
    s = plan(prog, fuse_pointwise=0)
    assert (s["materialized_ops"], s["inlined_ops"], s["stages"]) == (2, 0, 2)


def _gemm_relu_sum(relu_is_output):
    x, w = f32("x", (4, 8)), f32("W", (16, 8))
    ops = [Operation("t", "mm", (x, w.T), f32("t", (4, 16))),
           Operation("u", "relu", (f32("t", (4, 16)),), f32("u", (4, 16))),
           Operation("s", "sum", (f32("u", (4, 16)),), f32("s", ()))]
    outs = [f32("s", ())] + ([f32("u", (4, 16))] if relu_is_output else [])
    return Program([x, w], outs, ops)


def test_gemm_epilogue_chain_fusion():
    s = plan(_gemm_relu_sum(False))
    assert (s["fused_epilogues"], s["materialized_ops"], s["inlined_ops"], s["stages"]) == (1, 2, 0, 2)
    s = plan(_gemm_relu_sum(False), fuse_epilogues=0)           # relu then inlines into the sum
    assert (s["fused_epilogues"], s["materialized_ops"], s["inlined_ops"], s["stages"]) == (0, 2, 1, 2)


def test_chain_ends_at_a_program_output():
    # the relu output is returned: the epilogue stores it straight from the tile
    s = plan(_gemm_relu_sum(True))
    assert (s["fused_epilogues"], s["materialized_ops"], s["inlined_ops"], s["stages"]) == (1, 2, 0, 2)


def test_chain_does_not_pass_through_a_program_output():
    x, w = f32("x", (4, 8)), f32("W", (16, 8))
    v = lambda n: f32(n, (4, 16))
    ops = [Operation("t", "mm", (x, w.T), v("t")),
           Operation("u", "relu", (v("t"),), v("u")),
           Operation("n", "neg", (v("u"),), v("n")),
           Operation("s", "sum", (v("n"),), f32("s", ()))]
    s = plan(Program([x, w], [f32("s", ()), v("u")], ops))
    # mm+relu fused (ends at the output u); neg inlines into the sum
    assert (s["fused_epilogues"], s["materialized_ops"], s["inlined_ops"], s["stages"]) == (1, 2, 1, 2)


def _update(read_after):
    w, g = f32("W", (8,)), f32("g", (8,))
    upd = Operation("Wn", "sub", (w, g), f32("Wn", (8,)), {"alpha": 0.5})
    use = Operation("c", "mul", (w, 2.0), f32("c", (8,)))
    ops = [upd, use] if read_after else [use, upd]
    return Program([w, g], [f32("Wn", (8,)), f32("c", (8,))], ops, {0: 0})


def test_inplace_update_direct_when_no_later_reader():
    s = plan(_update(read_after=False))
    assert (s["direct_state_commits"], s["output_copies"], s["stages"], s["direct_outputs"]) == (1, 0, 2, 2)


def test_inplace_update_committed_after_a_later_reader():
    s = plan(_update(read_after=True))
    assert (s["direct_state_commits"], s["output_copies"], s["stages"], s["direct_outputs"]) == (0, 1, 2, 1)


def test_arena_reuse_never_adds_a_barrier():
    x = f32("x", (64,))
    v = lambda n: f32(n, (64,))
    ops = [Operation("a", "neg", (x,), v("a")),
           Operation("b", "mul", (v("a"), 2.0), v("b")),
           Operation("c", "add", (v("a"), 1.0), v("c")),
           Operation("d", "mul", (x, 3.0), v("d")),
           Operation("e", "add", (v("d"), v("d")), v("e"))]
    # d (stage 0) may not take a's slot while a is still read in stage 1
    s = plan(Program([x], [v("b"), v("c"), v("e")], ops))
    assert (s["materialized_ops"], s["stages"], s["arena_elements"]) == (5, 3, 128)


def test_arena_reuses_slots_across_stages():
    x = f32("x", (64,))
    v = lambda n: f32(n, (64,))
    ops = [Operation("a", "neg", (x,), v("a")),
           Operation("b", "mul", (v("a"), 2.0), v("b")),
           Operation("c", "add", (v("b"), 1.0), v("c")),
           Operation("e", "mul", (v("c"), 3.0), v("e"))]
    # c (stage 2) takes a's slot: a was last read in stage 1
    s = plan(Program([x], [v("e")], ops), fuse_pointwise=0)
    assert (s["materialized_ops"], s["stages"], s["arena_elements"]) == (4, 4, 128)


def test_large_mean_is_split():
    x = f32("x", (1024, 1024))
    s = plan(Program([x], [f32("m", ())], [Operation("m", "mean", (x,), f32("m", ()))]))
    assert (s["split_reductions"], s["stages"], s["max_work_items"]) == (1, 2, 128)


def test_mlp_step_plan_counts():
    s = plan(S.mlp_step_program(S.CONFIGS["c2"], export="state"))
    # fused: 3 forward addmm(+relu/+sub, the last also writing the loss gradient
    # 2/N*d as a side output), 2 input-grad mm(+threshold_backward), 3 weight-grad
    # mm(+SGD update, written in place) and 3 bias-grad sums (+SGD update);
    # inlined: pow
    assert (s["fused_epilogues"], s["inlined_ops"], s["materialized_ops"]) == (11, 1, 12)
    assert (s["direct_state_commits"], s["direct_outputs"], s["output_copies"]) == (6, 7, 0)
    # forward 3, then loss, ga2, gb3+update | gW3+update, ga1, gb2+update |
    # gW2+update, gW1+update, gb1+update
    assert s["stages"] == 6


def test_weight_update_gemm_runs_after_the_input_grad_gemm_that_reads_w():
    prog = S.mlp_step_program(S.CONFIGS["c2"], export="state")
    h = B.tk_program_create(prog, B.options(sm_count=152), device=-1)
    try:
        tasks = [B.tk_plan_task(h, i) for i in range(B.tk_plan_stats_get(h)["tasks"])]
    finally:
        B.tk_program_destroy(h)
    stage = {prog.operations[t["op_index"]].name: t["stage"] for t in tasks if t["op_index"] >= 0}
    for i in (2, 3):  # gW_i (fused with W_i's update) after ga_{i-1}, which reads W_i
        assert stage[f"gW{i}"] > stage[f"ga{i-1}"]


# ------------------------------------------------------------ errors

def _err(prog, match, status=None, **opts):
    with pytest.raises(B.TkError, match=match) as e:
        plan(prog, **opts)
    if status is not None:
        assert e.value.status == status


def test_rejects_malformed_programs():
    x, w = f32("x", (4, 8)), f32("W", (16, 8))
    _err(Program([x, w], [f32("t", (4, 16))], [Operation("t", "mm", (x, w), f32("t", (4, 16)))]),
         "compatible rank-two")
    _err(Program([x, f32("r", (3,))], [f32("a", (4, 8))],
                 [Operation("a", "add", (x, f32("r", (3,))), f32("a", (4, 8)))]), "incompatible broadcast")
    _err(Program([x], [f32("a", (4, 8))], [Operation("a", "mul", (x, float("inf")), f32("a", (4, 8)))]),
         "non-finite", 2)
    _err(Program([x], [f32("a", (4, 8))],
                 [Operation("a", "neg", (x,), TensorSpec("a", (4, 8), (1, 4), 0, "float32"))]), "contiguous")
    _err(Program([x], [f32("b", (4, 8))],
                 [Operation("b", "neg", (f32("a", (4, 8)),), f32("b", (4, 8))),
                  Operation("a", "neg", (x,), f32("a", (4, 8)))]), "topological")
    _err(Program([T("x", (4, 8), "float64")], [], []), "unsupported dtype", 2)
    _err(Program([TensorSpec("x", (-1, 8), (8, 1), 0, "float32")], [], []), "invalid static shape")
    _err(Program([x], [f32("s", (4,))], [Operation("s", "sum", (x,), f32("s", (4,)), {"dims": (2,)})]),
         "reduction dims")
    _err(Program([x], [f32("s", (3,))], [Operation("s", "sum", (x,), f32("s", (3,)), {"dims": (1,)})]),
         "reduction output shape")
    _err(Program([x], [f32("p", (4, 8))], [Operation("p", "pow", (x, x), f32("p", (4, 8)))]), "exponent")
    _err(Program([x], [f32("a", (4, 8))], [Operation("a", "neg", (x,), f32("a", (4, 8)))]), "blocks_per_sm",
         blocks_per_sm=9)
    neg = Program([x], [f32("a", (4, 8))], [Operation("a", "neg", (x,), f32("a", (4, 8)))])
    _err(neg, "tile_n", tile_n=192)
    _err(neg, "cta_pairs", cta_pairs=3)
    _err(neg, "epi_stage_bytes", epi_stage_bytes=-4)


def test_rejects_bad_inplace_mappings():
    x, y = f32("x", (4, 8)), f32("y", (4, 4))
    neg = Operation("a", "neg", (x,), f32("a", (4, 8)))
    _err(Program([x, y], [f32("a", (4, 8))], [neg], {0: 1}), "match a contiguous input")
    _err(Program([x], [x], [], {0: 0}), "computed values")
    _err(Program([x, f32("z", (4, 8))], [f32("a", (4, 8)), f32("b", (4, 8))],
                 [neg, Operation("b", "neg", (x,), f32("b", (4, 8)))], {0: 0, 1: 0}), "distinct inputs")
    _err(Program([x], [f32("a", (4, 8))], [neg], {0: 5}), "invalid inplace")


def test_plan_only_program_cannot_run():
    prog = S.mlp_step_program(S.CONFIGS["c1"])
    h = B.tk_program_create(prog, B.options(sm_count=8), device=-1)
    try:
        assert B.tk_allocate(h) >= 64
        with pytest.raises(B.TkError, match="plan-only") as e:
            B.tk_run(h, [16] * len(prog.inputs), [16] * len(prog.outputs), 256, 1 << 20)
        assert e.value.status == 6
    finally:
        B.tk_program_destroy(h)


@pytest.mark.parametrize("name", ["c2", "c3", "c5"])
def test_mlp_step_tasks_take_compiled_loops(name):
    # Every expression of the bf16 MLP step has one of the fixed shapes: bias
    # (+ReLU) and bias-minus-target GEMM epilogues, the ReLU-mask epilogue,
    # squares and scaled sums, SGD and momentum updates.
    s = plan(S.mlp_step_program(S.CONFIGS[name], export="state"))
    # C3's second layer (32 tiles, K = 4096) is split over K: its partial
    # products and their sum + epilogue evaluate the generic chain
    split = 1 if name == "c3" else 0
    assert s["compiled_tasks"] == s["materialized_ops"] - split and s["chain_tasks"] == 2 * split


def test_strided_operand_falls_back_to_generic_chain():
    x = f32("x", (8, 16))
    xt = TensorSpec("x", (16, 8), (1, 16), 0, "float32")
    prog = Program([x], [f32("y", (16, 8))], [Operation("y", "mul", (xt, 3.0), f32("y", (16, 8)))])
    s = plan(prog)
    assert (s["compiled_tasks"], s["chain_tasks"]) == (0, 1)
    s = plan(Program([x], [f32("y", (8, 16))], [Operation("y", "mul", (x, 3.0), f32("y", (8, 16)))]))
    assert (s["compiled_tasks"], s["chain_tasks"]) == (1, 0)


def test_expr_forms_option_restricts_evaluators():
    prog = S.mlp_step_program(S.CONFIGS["c2"], export="state")
    s0, s1, s2 = (plan(prog, expr_forms=f) for f in (0, 1, 2))
    assert s0["compiled_tasks"] > 0
    assert s1["compiled_tasks"] == 0 and s1["chain_tasks"] == s0["compiled_tasks"] + s0["chain_tasks"]
    assert s2["compiled_tasks"] == 0 and s2["chain_tasks"] == 0
    with pytest.raises(B.TkError):
        plan(prog, expr_forms=3)


@pytest.mark.parametrize("name", ["c2", "c5"])
def test_tensor_core_epilogues_are_staged(name):
    # 16-bit GEMM epilogues move their tiles through shared memory; with
    # 256-wide tiles (C5) the 192 KB ring leaves room for a per-row operand
    # (the target) and a bias row per epilogue warp.
    prog = S.mlp_step_program(S.CONFIGS[name], export="state")
    h = B.tk_program_create(prog, B.options(sm_count=152), device=-1)
    try:
        tasks = [B.tk_plan_task(h, i) for i in range(B.tk_plan_stats_get(h)["tasks"])]
    finally:
        B.tk_program_destroy(h)
    tc = [t for t in tasks if t["kind"] == "gemm_tc"]
    direct = [prog.operations[t["op_index"]].name for t in tc if not t["staged_epilogue"]]
    assert tc and direct == []


def _tc_tasks(prog, **opts):
    h = B.tk_program_create(prog, B.options(sm_count=152, **opts), device=-1)
    try:
        tasks = [B.tk_plan_task(h, i) for i in range(B.tk_plan_stats_get(h)["tasks"])]
    finally:
        B.tk_program_destroy(h)
    return {prog.operations[t["op_index"]].name: t for t in tasks if t["kind"] == "gemm_tc"}


def test_staging_ring_depth_follows_the_shared_memory_left():
    # C3's momentum GEMMs (128-wide tiles, a 128 KB ring): v and W of all four
    # 32-column chunks of a tile fit at once (depth 4); C2's output layer gets
    # buffers of its own for the loss gradient (depth 2 + 16); C5's 192 KB ring
    # leaves room for depth 2 only, with the side values written in place
    c3 = _tc_tasks(S.mlp_step_program(S.CONFIGS["c3"], export="state"))
    assert c3["gW1"]["staged_depth"] == c3["gW2"]["staged_depth"] == 4
    assert c3["z1"]["staged_depth"] == 2                     # 64-wide tiles: two chunks
    c2 = _tc_tasks(S.mlp_step_program(S.CONFIGS["c2"], export="state"))
    assert c2["z3"]["side_output"] and c2["z3"]["staged_depth"] == 2 + 16
    c5 = _tc_tasks(S.mlp_step_program(S.CONFIGS["c5"], export="state"))
    assert {t["staged_depth"] for t in c5.values()} == {2}
    # a cap on the staging bytes of each epilogue warp gives shallower rings
    capped = _tc_tasks(S.mlp_step_program(S.CONFIGS["c3"], export="state"), epi_stage_bytes=8192)
    assert capped["gW1"]["staged_depth"] == 2
    capped = _tc_tasks(S.mlp_step_program(S.CONFIGS["c2"], export="state"), epi_stage_bytes=8192)
    assert capped["z3"]["staged_depth"] == 2
    assert not _tc_tasks(S.mlp_step_program(S.CONFIGS["c2"], export="state"), epi_stage_bytes=1024)["z3"]["staged_epilogue"]
    with pytest.raises(B.TkError):
        plan(S.mlp_step_program(S.CONFIGS["c2"], export="state"), epi_stage_bytes=-1)


def test_reduction_epilogue_fuses_the_bias_update():
    g, b = f32("g", (16, 8)), f32("b", (8,))
    ops = [Operation("gb", "sum", (g,), f32("gb", (8,)), {"dims": (0,)}),
           Operation("bn", "sub", (b, f32("gb", (8,))), f32("bn", (8,)), {"alpha": 0.5})]
    s = plan(Program([g, b], [f32("bn", (8,))], ops, {0: 1}))
    assert (s["fused_epilogues"], s["materialized_ops"], s["stages"], s["direct_state_commits"]) == (1, 1, 1, 1)
    # a returned gradient is stored, and the update is written next to it as
    # a side output of the same reduction (one op, one stage); without
    # epilogue fusion it is a second pass behind a barrier
    s = plan(Program([g, b], [f32("bn", (8,)), f32("gb", (8,))], ops, {0: 1}))
    assert (s["fused_epilogues"], s["materialized_ops"], s["stages"], s["direct_state_commits"]) == (1, 1, 1, 1)
    s = plan(Program([g, b], [f32("bn", (8,)), f32("gb", (8,))], ops, {0: 1}), fuse_epilogues=0)
    assert (s["fused_epilogues"], s["materialized_ops"], s["stages"]) == (0, 2, 2)


def test_loaded_side_outputs_write_the_momentum_step_from_the_tile():
    # momentum: the weight-gradient GEMM writes v' = 0.9 v + gW (its chain) and
    # W' = W - lr v' (a side output loading W); both in place, both direct,
    # after the input-gradient GEMM that reads the old W
    prog = S.mlp_step_program(S.CONFIGS["c3"], export="state")
    h = B.tk_program_create(prog, B.options(sm_count=152), device=-1)
    try:
        st = B.tk_plan_stats_get(h)
        tasks = [B.tk_plan_task(h, i) for i in range(st["tasks"])]
    finally:
        B.tk_program_destroy(h)
    name = lambda t: prog.operations[t["op_index"]].name if t["op_index"] >= 0 else None
    assert not any(name(t) in ("W1_new", "W2_new", "b1_new", "b2_new") for t in tasks)
    gw = {name(t): t for t in tasks if name(t) in ("gW1", "gW2")}
    assert all(t["side_output"] for t in gw.values())
    ga1 = next(t for t in tasks if name(t) == "ga1")
    assert gw["gW2"]["stage"] > ga1["stage"]
    assert st["output_copies"] == 0 and st["direct_state_commits"] == 8
    assert sum(t["side_output"] for t in tasks if t["kind"] in ("reduce_col", "reduce_final")) == 2


def test_side_output_written_from_the_gemm_tile():
    x, w, y = f32("x", (4, 8)), f32("W", (16, 8)), f32("y", (4, 16))
    v = lambda n: f32(n, (4, 16))
    ops = [Operation("z", "mm", (x, w.T), v("z")),
           Operation("d", "sub", (v("z"), y), v("d")),
           Operation("g", "mul", (v("d"), 0.5), v("g")),
           Operation("s", "sum", (v("d"),), f32("s", ())),
           Operation("h", "mm", (v("g"), f32("V", (16, 3))), f32("h", (4, 3)))]
    prog = Program([x, w, y, f32("V", (16, 3))], [f32("s", ()), f32("h", (4, 3))], ops)
    s = plan(prog)
    # mm -> d fused; g comes from the same tile; s and h run in the next stage
    assert (s["fused_epilogues"], s["materialized_ops"], s["stages"]) == (1, 3, 2)
    s = plan(prog, fuse_epilogues=0)
    assert (s["materialized_ops"], s["stages"]) == (5, 4)


def test_under_filled_gemm_is_split_over_k():
    prog = S.mlp_step_program(S.CONFIGS["c3"], export="state")
    h = B.tk_program_create(prog, B.options(sm_count=152), device=-1)
    try:
        tasks = [B.tk_plan_task(h, i) for i in range(B.tk_plan_stats_get(h)["tasks"])]
    finally:
        B.tk_program_destroy(h)
    z2 = [t for t in tasks if t["op_index"] >= 0 and prog.operations[t["op_index"]].name == "z2"]
    assert [t["kind"] for t in z2] == ["gemm_tc", "splitk_final"]
    assert z2[0]["n_items"] == 4 * 32 and z2[1]["stage"] == z2[0]["stage"] + 1
    s = plan(prog, split_k=0)
    assert s["tasks"] == len(tasks) - 1


def test_pair_tiles_plan_256_row_tiles_without_split_k():
    # cta_pairs: every tensor-core GEMM on 256-row tiles dealt to pairs of
    # SMs, 128-wide at least (each block stages half of B's columns), no
    # split-K; the C5 forward GEMMs still take 224 columns (16 x 19 = 304 pair
    # tiles = 4 waves of 76 pairs), the backward ones (MN-major B) 256
    c5 = S.mlp_step_program(S.CONFIGS["c5"], export="state")
    st = plan(c5, cta_pairs=1)
    assert st["cta_pairs"] == 1
    tasks = _tc_tasks(c5, cta_pairs=1)
    assert all(t["tile_m"] == 256 for t in tasks.values())
    assert (tasks["z1"]["tile_n"], tasks["z1"]["n_items"]) == (224, 304)
    assert (tasks["gW1"]["tile_n"], tasks["gW1"]["n_items"]) == (256, 256)
    c3 = S.mlp_step_program(S.CONFIGS["c3"], export="state")
    assert plan(c3)["split_reductions"] >= 1
    single = _tc_tasks(c3)
    paired = _tc_tasks(c3, cta_pairs=1)
    assert single["z2"]["n_items"] == 128                  # 32 tiles x 4 k splits
    assert paired["z2"]["n_items"] == 8 and paired["z2"]["tile_n"] == 128
    assert plan(c3, cta_pairs=0)["cta_pairs"] == 0
    # a program without tensor-core GEMMs ignores the option
    assert plan(S.mlp_step_program(S.CONFIGS["c1"], export="state"), cta_pairs=1)["cta_pairs"] == 0


def test_forward_gemms_take_224_wide_tiles_where_they_fill_whole_waves():
    c5 = _tc_tasks(S.mlp_step_program(S.CONFIGS["c5"], export="state"))
    assert {n: t["tile_n"] for n, t in c5.items() if n.startswith("z")} == {f"z{i}": 224 for i in range(1, 5)}
    assert c5["z1"]["n_items"] == 608 == 4 * 152
    # MN-major B (the input-gradient and weight-gradient GEMMs) stays at 256
    assert {t["tile_n"] for n, t in c5.items() if not n.startswith("z")} == {256}
    # forced: 224 where B is K-major, 256 elsewhere
    forced = _tc_tasks(S.mlp_step_program(S.CONFIGS["c2"], export="state"), tile_n=224)
    assert {t["tile_n"] for n, t in forced.items() if n.startswith("z")} == {224}
    assert {t["tile_n"] for n, t in forced.items() if not n.startswith("z")} == {256}


def test_reductions_run_beside_long_tiles_where_they_fit():
    # C5: the loss and three bias gradients run on warps 2-3 beside the
    # 4096^3 GEMM tiles; C2's short tiles keep theirs after the tiles unless
    # forced; option 0 keeps every reduction after the tiles
    def beside(name, **opts):
        prog = S.mlp_step_program(S.CONFIGS[name], export="state")
        h = B.tk_program_create(prog, B.options(sm_count=152, **opts), device=-1)
        try:
            tasks = [B.tk_plan_task(h, i) for i in range(B.tk_plan_stats_get(h)["tasks"])]
        finally:
            B.tk_program_destroy(h)
        return sorted(prog.operations[t["op_index"]].name for t in tasks if t["beside_tiles"])
    assert beside("c5") == ["gb1", "gb2", "gb3", "loss"]      # gb4 would not fit beside the loss
    assert beside("c5", overlap_reductions=0) == []
    assert beside("c2") == []
    assert beside("c2", overlap_reductions=2) == ["gb1", "gb2", "gb3", "loss"]
    assert beside("c1", overlap_reductions=2) == []          # no tensor-core stage


def test_split_bias_gradient_finals_fold_into_their_partials_stage():
    # C5: gb1..gb3 are split column sums beside the tiles; each one's final
    # pass (the sum of its 19 parts and the SGD update of the bias) is run by
    # the warp that adds a 256-column chunk's last part, in the same stage, so
    # the stage that held only gb1's final pass goes; the loss (one output,
    # a block-wide final) and gb4 (after the tiles) keep their final passes
    def plan(**opts):
        prog = S.mlp_step_program(S.CONFIGS["c5"], export="state")
        h = B.tk_program_create(prog, B.options(sm_count=152, **opts), device=-1)
        try:
            stats = B.tk_plan_stats_get(h)
            tasks = [B.tk_plan_task(h, i) for i in range(stats["tasks"])]
        finally:
            B.tk_program_destroy(h)
        for t in tasks:
            t["op"] = prog.operations[t["op_index"]].name
        return stats, tasks
    stats, tasks = plan()
    assert stats["stages"] == 8 and stats["grid_barriers"] == 7
    folded = {t["op"]: t for t in tasks if t["folded"]}
    assert sorted(folded) == ["gb1", "gb2", "gb3"]
    for name, f in folded.items():
        (part,) = [t for t in tasks if t["op"] == name and t["kind"] == "reduce_col"]
        assert f["kind"] == "reduce_final" and f["n_items"] == 0 and f["stage"] == part["stage"] and part["beside_tiles"]
        assert part["n_items"] == 16 * part["parts"]
    finals = sorted(t["op"] for t in tasks if t["kind"] == "reduce_final" and not t["folded"])
    assert finals == ["gb4", "loss"]
    # with every reduction after the tiles nothing folds
    stats0, tasks0 = plan(overlap_reductions=0)
    assert stats0["stages"] == 9 and not any(t["folded"] for t in tasks0)
    # with every reduction beside the tiles gb4 folds too, and gb1's 16
    # chunks no longer fit the 59 counters: it keeps its own final stage
    stats2, tasks2 = plan(overlap_reductions=2)
    assert sorted(t["op"] for t in tasks2 if t["folded"]) == ["gb2", "gb3", "gb4"]
    assert stats2["stages"] == 9
