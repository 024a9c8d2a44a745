"""Tuner and configuration-generator host logic (no GPU): the representative
shapes fall in the classes they stand for (the library's own classifier),
the generated candidates are legal, the pruning rules hold, names round-trip,
the scoring picks the least geometric-mean relative time, the two-stage
search keeps the best configurations and tries every policy on them, and the
written configuration list and table name real, legal configurations."""
import os
import re

import pytest

from dense_fp32_gemm_gb300 import binding, configgen, tune


def test_representative_shapes_classify_as_their_class():
    for cls, shapes in tune.CLASS_SHAPES.items():
        for M, N, K, _, _ in shapes:
            assert binding.sgemm_choose_config(M, N, K)[1] == cls, (cls, M, N, K)
    assert set(tune.CLASS_TOKENS) == set(binding.SHAPE_CLASSES) == set(tune.CLASS_SHAPES)


def test_candidates_are_legal_and_obey_the_pruning_rules():
    cands = configgen.candidates()
    assert 20 <= len(cands) <= 64
    assert len(set(cands)) == len(cands)
    for t in cands:
        rule, d = binding.sgemm_cfg_check(list(t))       # the library's checker agrees
        assert rule == 0, t
        BM, BN, BK, WM, WN, WNI, TM, TN, NT, ST, MINB, KU, ORD = t
        assert (TM, TN, ORD, KU) == (4, 4, 2, BK) and BK in (16, 24, 32)      # P1-P3
        assert (NT // 32) * MINB >= 8 and d["acc"] >= 64                        # P5, P6
        # P4: the next larger residency of the searched range would not fit
        larger = [m for m in configgen.SPACE["MINB"] if m > MINB]
        if larger:
            more = list(t)
            more[10] = min(larger)
            assert all(binding.sgemm_cfg_check(more[:9] + [st, more[10]] + more[11:])[0] != 0
                       for st in configgen.SPACE["STAGES"]), t
    # the measured square-large winner of the first hand-picked sweep is generated
    assert (128, 256, 32, 64, 64, 2, 4, 4, 256, 4, 1, 32, 2) in cands
    # every tile shape of the space that has a legal pruned tuple is represented
    shapes = {t[:3] for t in cands}
    assert {(128, 256, 32), (256, 64, 16), (64, 256, 24), (128, 64, 32), (128, 128, 32)} <= shapes


def test_generated_names_round_trip():
    for t in configgen.candidates() + [tune.PAGES_WINNER]:
        name = configgen.config_name(t)
        assert re.fullmatch(r"[A-Za-z_]\w*", name)
        assert configgen.parse_name(name) == t
        assert configgen.parse_name(name + "_suffix") == t
    with pytest.raises(ValueError):
        configgen.parse_name("WideBk32F2Ku32")


def test_checker_rejects_what_the_kernel_forbids():
    # the host copy of the checker is the kernel's own constexpr function
    assert configgen.check((128, 512, 8, 64, 64, 2, 4, 4, 512, 3, 1, 8, 2))[0] == 13
    assert configgen.check((128, 64, 16, 64, 32, 2, 4, 4, 128, 2, 1, 16, 2))[0] == 16
    for t in configgen.candidates()[:5]:
        assert configgen.check(t)[0] == binding.sgemm_cfg_check(list(t))[0] == 0


def test_relative_scores_and_pick():
    t = {"A": [1.0, 4.0], "B": [2.0, 2.0], "C": [None, 0.1]}
    sc = tune.relative_scores(t)
    assert set(sc) == {"A", "B"}                       # C failed on a shape
    assert sc["A"] == pytest.approx((1.0 * 2.0) ** 0.5)  # 1/1 and 4/2
    assert sc["B"] == pytest.approx((2.0 * 1.0) ** 0.5)
    assert tune.pick_best(t) == "A"                    # tie: the smaller key
    assert tune.pick_best({"A": [3.0], "B": [2.0]}) == "B"
    with pytest.raises(RuntimeError):
        tune.pick_best({"A": [None]})


def test_search_class_two_stages():
    names = ["c0", "c1", "c2", "c3", "c4"]
    calls = []

    def measure(si, cid, pol):
        calls.append((cid, pol))
        if cid == 4:
            raise RuntimeError("cannot run")
        base = [5.0, 1.0, 3.0, 2.0][cid]
        bonus = 1.5 if (cid == 3 and pol == (tune.SPK, 8, 4, 4)) else 0.0
        return base - bonus
    win, st1, st2 = tune.search_class("skinny_n", names, measure, top=2, log=lambda *_: None)
    assert win == (3, (tune.SPK, 8, 4, 4))
    assert st1[4] == [None] * len(tune.CLASS_SHAPES["skinny_n"])
    kept = {c for c, _ in st2}
    assert kept == {1, 3}                              # the two best of stage 1
    assert {p for c, p in st2 if c == 3} == set(tune.POLICIES)


def test_table_and_product_list_name_real_configurations(tmp_path):
    cands = configgen.candidates()
    winners = {c: (configgen.config_name(cands[i % len(cands)]), tune.POLICIES[i % len(tune.POLICIES)])
               for i, c in enumerate(tune.CLASS_TOKENS)}
    text = tune.table_text(winners, "GPU", 152)
    rows = re.findall(r"X\((\w+), (\w+), (\d+), (\d+), (\d+), (\d+)\)", text)
    assert [r[0] for r in rows] == list(tune.CLASS_TOKENS.values())
    tuples = [configgen.parse_name(winners[c][0]) for c in tune.CLASS_TOKENS]
    entries = tune.product_entries(tuples + tuples[:1])
    assert [t for t, a in entries if a] == list(dict.fromkeys(tuples))
    assert entries[-1] == (tune.PAGES_WINNER, False)
    path = tmp_path / "configs.inc"
    configgen.write_configs_inc(entries, tuples[0], "test.", path=str(path))
    back, fb = configgen.read_configs_inc(str(path))
    assert back == entries and fb == tuples[0]


def test_configs_inc_refuses_bad_lists():
    good = (128, 256, 32, 64, 64, 2, 4, 4, 256, 4, 1, 32, 2)
    bad = (128, 64, 16, 64, 32, 2, 4, 4, 128, 2, 1, 16, 2)       # two stages
    with pytest.raises(ValueError):
        configgen.configs_inc_text([(good, True), (bad, False)], good, "x")
    with pytest.raises(ValueError):
        configgen.configs_inc_text([(good, False)], good, "x")  # fallback not all-layout
    with pytest.raises(ValueError):
        configgen.configs_inc_text([(good, True), (good, True)], good, "x")


def test_committed_list_and_table_are_consistent():
    entries, fb = configgen.read_configs_inc()
    names = [configgen.config_name(t) for t, _ in entries]
    assert names == [binding.sgemm_config_info(i)[0] for i in range(binding.sgemm_config_count())]
    text = open(os.path.join(os.path.dirname(tune.__file__), "csrc", "tuned_table.inc")).read()
    rows = re.findall(r"X\((\w+), (\w+), (\d+), (\d+), (\d+), (\d+)\)", text)
    assert sorted(r[0] for r in rows) == sorted(tune.CLASS_TOKENS.values())
    layouts = dict((configgen.config_name(t), a) for t, a in entries)
    for r in rows:
        assert layouts[r[1]], r           # every class winner is built for every layout
        assert 0 <= int(r[2]) < len(binding.SCHED_MODES)
    assert layouts[configgen.config_name(fb)]


def test_every_class_dispatches_to_an_all_layout_configuration():
    # the dispatcher's choice also serves sgemm_ex and sgemm_strided_batched
    # with transposed operands, so it must be built for every layout
    for cls, shapes in tune.CLASS_SHAPES.items():
        for M, N, K, _, _ in shapes:
            cid, _ = binding.sgemm_choose_config(M, N, K)
            assert binding.sgemm_config_layouts(cid) == 1, (cls, binding.sgemm_config_info(cid)[0])
    assert binding.sgemm_config_layouts(binding.sgemm_config_count()) == binding.SGEMM_ERR_INVALID_VALUE


def test_default_policy_wins_within_noise():
    D, S = tune.DEFAULT_POLICY, (tune.SPK, 8, 4, 2)
    t = {("a", D): [1.003, 2.0], ("a", S): [1.0, 2.0], ("b", D): [1.5, 3.0]}
    assert tune.pick_with_default(t) == ("a", D)            # 0.15 % behind: noise
    t[("a", S)] = [0.9, 1.8]
    assert tune.pick_with_default(t) == ("a", S)            # 10 % ahead: a real win
    rec = {"stage2_ms": {"tiny": {f"a {list(D)}": [1.003], f"a {list(S)}": [1.0]}}}
    assert tune.winners_from_record(rec) == {"tiny": ("a", D)}
