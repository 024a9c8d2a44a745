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


def test_tune_classes_saves_after_each_class_and_resumes():
    names = ["A_x", "B_x"]
    calls, saved = [], []

    def measure(cls, ci, si, cid):
        calls.append((cls, si, cid))
        if cid == 1 and si == 0:
            raise RuntimeError("cannot run")
        return 1.0 + cid
    classes = ["tiny", "skinny_n"]
    t = tune.tune_classes(names, classes, measure, save=lambda x: saved.append(dict(x)),
                          log=lambda *_: None)
    assert [list(s) for s in saved] == [["tiny"], ["tiny", "skinny_n"]]
    assert t["tiny"]["B_x"][0] is None and t["tiny"]["A_x"] == [1.0] * len(tune.CLASS_SHAPES["tiny"])
    # an interrupted run saved "tiny": resuming measures only "skinny_n"
    calls.clear()
    t2 = tune.tune_classes(names, classes, measure, done={"tiny": t["tiny"]}, log=lambda *_: None)
    assert t2["tiny"] == t["tiny"] and {c[0] for c in calls} == {"skinny_n"}


def test_load_partial_matches_gpu_sms_configs_and_shapes(tmp_path):
    import json
    names = ["A_x", "B_x"]
    rec = {"gpu": "GPU", "sms": 152, "config_names": names,
           "shapes": {"tiny": [list(x) for x in tune.CLASS_SHAPES["tiny"]],
                      "skinny_n": [[1, 2, 3, 1.0, 0.0]]},
           "timings_ms": {"tiny": {"A_x": [1.0]}, "skinny_n": {"A_x": [2.0]}}}
    p = tmp_path / "tuned_table.json"
    p.write_text(json.dumps(rec))
    # skinny_n was timed on other shapes: only tiny resumes
    assert tune.load_partial(str(p), "GPU", 152, names) == {"tiny": {"A_x": [1.0]}}
    assert tune.load_partial(str(p), "GPU", 148, names) == {}
    assert tune.load_partial(str(p), "OTHER", 152, names) == {}
    assert tune.load_partial(str(p), "GPU", 152, names + ["C_x"]) == {}
    assert tune.load_partial(str(tmp_path / "missing.json"), "GPU", 152, names) == {}
