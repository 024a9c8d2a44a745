"""Tuner host logic: the representative shapes fall in the classes they
stand for (checked against the library's own classifier), winners are the
least total time, and the generated table names real configurations."""
import re

from dense_fp32_gemm_gb300 import binding, tune


def test_representative_shapes_classify_as_their_class():
    for cls, shapes in tune.CLASS_SHAPES.items():
        for M, N, K, _, _ in shapes:
            assert binding.sgemm_choose_config(M, N, K)[1] == cls, (cls, M, N, K)


def test_pick_winners_least_total_time():
    t = {"square_large": {"A_x": [1.0, 3.0], "B_x": [2.0, 1.5], "C_x": [None, 0.1]}}
    assert tune.pick_winners(t) == {"square_large": "B_x"}


def test_generated_table_names_compiled_configs():
    names = [binding.sgemm_config_info(i)[0] for i in range(binding.sgemm_config_count())]
    winners = {c: names[i % len(names)] for i, c in enumerate(tune.CLASS_TOKENS)}
    text = tune.table_text(winners, "GPU", 152)
    rows = re.findall(r"X\((\w+), (\w+)\)", text)
    assert [r[0] for r in rows] == list(tune.CLASS_TOKENS.values())
    tokens = {n.split("_", 1)[0] for n in names}
    assert all(r[1] in tokens for r in rows)


def test_committed_table_is_well_formed():
    import os
    text = open(os.path.join(os.path.dirname(tune.__file__), "csrc", "tuned_table.inc")).read()
    rows = re.findall(r"X\((\w+), (\w+)\)", text)
    assert sorted(r[0] for r in rows) == sorted(tune.CLASS_TOKENS.values())


def test_pick_winners_only_among_eligible():
    t = {"k_dominant": {"A_x": [1.0], "B_x": [2.0]}}
    assert tune.pick_winners(t, eligible={"B_x"}) == {"k_dominant": "B_x"}


def test_every_class_dispatches_to_an_all_layout_configuration():
    # the dispatcher's choice also serves sgemm_ex and sgemm_strided_batched
    # with transposed operands, so it must be built for every layout
    for cls, shapes in tune.CLASS_SHAPES.items():
        for M, N, K, _, _ in shapes:
            cid, _ = binding.sgemm_choose_config(M, N, K)
            assert binding.sgemm_config_layouts(cid) == 1, (cls, binding.sgemm_config_info(cid)[0])
    assert binding.sgemm_config_layouts(binding.sgemm_config_count()) == binding.SGEMM_ERR_INVALID_VALUE
