"""Pins for the gating top-k oracle (oracle/gating.py), against facts that do not come from it:
closed forms of the three normalisations, a hand-worked grouped example (sigmoid scores chosen
as logits of round probabilities, so every score is known), numpy's stable argsort for the
ungrouped case, the defining inequalities of grouped top-k on random inputs, the scaling identity,
hash routing, and planted mistakes that must each fail one of them.

Source: "CANN 自定义算子详解：npu_moe_gating_top_k" (m.qwbw.cn/news/316089), sections 归一化公式,
分组排序公式, 专家选择公式, 路由权重缩放公式, 约束说明.
"""
import importlib.util
import math
import os

import numpy as np
import pytest

from oracle import gating

HERE = os.path.dirname(os.path.abspath(__file__))


def test_normalisation_closed_forms(g=gating):
    assert g.normalize(np.array([[0.0]]), 1)[0, 0] == pytest.approx(0.5)
    assert g.normalize(np.array([[math.log(3.0)]]), 1)[0, 0] == pytest.approx(0.75)
    assert g.normalize(np.array([[0.0]]), 2)[0, 0] == pytest.approx(math.log(2.0))
    assert g.normalize(np.array([[math.log(3.0)]]), 2)[0, 0] == pytest.approx(math.log(4.0))
    assert g.normalize(np.array([[800.0]]), 2)[0, 0] == pytest.approx(800.0)     # no overflow
    assert np.allclose(g.normalize(np.zeros((1, 5)), 0), 0.2)
    assert np.allclose(g.normalize(np.array([[0.0, math.log(2.0)]]), 0), [1 / 3, 2 / 3])
    assert np.allclose(g.normalize(np.array([[1000.0, 1000.0]]), 0), [0.5, 0.5])


P = np.array([0.1, 0.9, 0.8, 0.2, 0.7, 0.6, 0.3, 0.95])   # the sigmoid scores of the hand example
X = np.log(P / (1 - P))[None, :]


def check_hand_examples(g=gating):
    # 4 groups of 2; group maxima 0.9, 0.8, 0.7, 0.95 -> keep groups 3 and 0 -> experts 7, 1, 6
    r = g.gating_topk(X, 3, k_group=2, group_count=4, norm_type=1, group_select_mode=0)
    assert r["expert_idx"][0].tolist() == [7, 1, 6]
    assert np.allclose(r["y_out"][0], np.array([0.95, 0.9, 0.3]) / 2.15, atol=1e-6)
    # top-2 sums 1.0, 1.0, 1.3, 1.25 -> keep groups 2 and 3 -> experts 7, 4, 5; scaled by 2.5
    r = g.gating_topk(X, 3, k_group=2, group_count=4, norm_type=1, group_select_mode=1,
                      routed_scaling_factor=2.5)
    assert r["expert_idx"][0].tolist() == [7, 4, 5]
    assert np.allclose(r["y_out"][0], np.array([0.95, 0.7, 0.6]) / 2.25 * 2.5, atol=1e-6)
    # a bias of +0.5 on expert 4 lifts group 2's maximum from 0.7 to 1.2: it now leads
    bias = np.zeros(8, np.float32)
    bias[4] = 0.5
    r = g.gating_topk(X, 2, k_group=1, group_count=4, norm_type=1, bias=bias)
    assert r["expert_idx"][0].tolist() == [4, 5]                 # group 2 now leads: 1.2, 0.6
    assert np.allclose(r["y_out"][0], np.array([1.2, 0.6]) / 1.8, atol=1e-6)
    # rows flagged in additional_token_mask take additional_bias instead of bias
    extra = np.zeros(8, np.float32)
    extra[0] = 2.0
    r = g.gating_topk(np.repeat(X, 2, axis=0), 1, k_group=1, group_count=1, norm_type=1, bias=bias,
                      additional_bias=extra, additional_token_mask=np.array([False, True]))
    assert r["expert_idx"][:, 0].tolist() == [4, 0]
    # hash routing: the table row, in its own order, whatever the scores
    tid2eid = np.array([[5, 2, 7], [1, 0, 3]], np.int32)
    r = g.gating_topk(np.repeat(X, 3, axis=0), 3, input_ids=np.array([1, 0, 1]), tid2eid=tid2eid,
                      norm_type=1)
    assert r["expert_idx"].tolist() == [[1, 0, 3], [5, 2, 7], [1, 0, 3]]
    assert np.allclose(r["y_out"][1], np.array([0.6, 0.8, 0.95]) / 2.35, atol=1e-6)


def test_hand_examples():
    check_hand_examples()


def check_ungrouped_matches_stable_argsort(g=gating):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((40, 64)).astype(np.float16)
    for nt in (0, 1, 2):
        r = g.gating_topk(x, 6, norm_type=nt)
        s = r["norm_out"]
        ref = np.argsort(-s, axis=1, kind="stable")[:, :6]
        assert np.array_equal(r["expert_idx"], ref.astype(np.int32)), nt


def test_ungrouped_matches_stable_argsort():
    check_ungrouped_matches_stable_argsort()


def check_grouped_inequalities(g=gating):
    rng = np.random.default_rng(4)
    T, e, G, kg, k = 30, 64, 8, 3, 7
    x = rng.standard_normal((T, e)).astype(np.float32)
    bias = (rng.standard_normal(e) * 0.1).astype(np.float32)
    for mode in (0, 1):
        r = g.gating_topk(x, k, bias=bias, k_group=kg, group_count=G, group_select_mode=mode,
                          norm_type=1, routed_scaling_factor=1.7, eps=1e-9)
        s = r["norm_out"].astype(np.float64)
        grp = s.reshape(T, G, e // G)
        gscore = grp.max(-1) if mode == 0 else np.sort(grp, -1)[..., -2:].sum(-1)
        for t in range(T):
            idx = r["expert_idx"][t]
            assert len(set(idx.tolist())) == k
            kept = sorted(set((idx // (e // G)).tolist()))
            assert len(kept) <= kg
            # every kept group scores at least as high as every dropped one
            order = np.argsort(-gscore[t], kind="stable")
            top = set(order[:kg].tolist())
            assert set(kept) <= top
            assert gscore[t][list(top)].min() >= gscore[t][[q for q in range(G) if q not in top]].max()
            # every chosen expert beats every unchosen expert of the kept groups, in order
            cand = [j for q in top for j in range(q * (e // G), (q + 1) * (e // G))]
            rest = [j for j in cand if j not in set(idx.tolist())]
            assert s[t, idx].min() >= s[t, rest].max()
            assert np.all(np.diff(s[t, idx]) <= 0)
            # scaling identity
            ysum = s[t, idx].sum()
            assert r["y_out"][t].sum() == pytest.approx(1.7 * ysum / (ysum + 1e-9), rel=1e-12)


def test_grouped_inequalities():
    check_grouped_inequalities()


def test_constraints():
    x = np.zeros((2, 16), np.float32)
    for kw in [dict(k=0), dict(k=65), dict(k=17), dict(renorm=1), dict(group_count=3),
               dict(group_count=4, k_group=5), dict(group_count=4, k_group=1, k=5),
               dict(norm_type=3), dict(group_select_mode=2), dict(group_count=16, group_select_mode=1)]:
        args = dict(k=2)
        args.update(kw)
        with pytest.raises(gating.GatingArgError):
            gating.gating_topk(x, **args)
    with pytest.raises(gating.GatingArgError):
        gating.gating_topk(x, 2, input_ids=np.zeros(2, np.int64))


MUTANTS = {
    "group_min_not_max": ("gscores.append(vals[0] if group_select_mode == 0",
                          "gscores.append(vals[-1] if group_select_mode == 0"),
    "bias_ignored": ("            score[t] = (score[t] + np.asarray(bias, np.float32)).astype(np.float32)",
                     "            pass"),
    "no_eps_scale": ("y_out[t] = y / (y.sum() + eps) * routed_scaling_factor", "y_out[t] = y / y.sum()"),
    "sigmoid_sign": ("return 1.0 / (1.0 + np.exp(-x))", "return 1.0 / (1.0 + np.exp(x))"),
    "ascending_experts": ("chosen = sorted(cand, key=lambda j: (-float(row[j]), j))[:k]",
                          "chosen = sorted(cand, key=lambda j: (float(row[j]), j))[:k]"),
    "top2_as_top1": ("else float(np.float32(vals[0]) + np.float32(vals[1])))",
                     "else float(np.float32(vals[0]) + np.float32(vals[0])))"),
    "extra_bias_ignored": ("        if use_extra:", "        if False:"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    src = open(gating.__file__, encoding="utf-8").read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    path = tmp_path / f"gating_{name}.py"
    path.write_text(src.replace(old, new), encoding="utf-8")
    spec = importlib.util.spec_from_file_location(f"gating_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = False
    for pin in (test_normalisation_closed_forms, check_hand_examples,
                check_ungrouped_matches_stable_argsort, check_grouped_inequalities):
        try:
            pin(mod)
        except AssertionError:
            caught = True
            break
    assert caught, f"planted mistake {name} passed every pin"
