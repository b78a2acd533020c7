"""The pins catch plausible mistakes: each test plants one mistake in the oracle (on
the CPU, through monkeypatch) and checks that a pin test then fails."""
import numpy as np
import pytest

from oracle import accept, attention, draft, tree
from tests import test_oracle_accept as ta
from tests import test_oracle_attention as tat
from tests import test_oracle_draft as td
from tests import test_oracle_tree as tt


def test_causal_mask_instead_of_ancestor_mask_is_caught(monkeypatch):
    monkeypatch.setattr(tree, "tree_mask", lambda p: np.tril(np.ones((len(p), len(p)), bool)))
    with pytest.raises(AssertionError):
        tt.test_six_node_mask_matches_printed_example()


def test_depth_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(tree, "depths", lambda p: [0] + [1] * (len(p) - 1))
    with pytest.raises(AssertionError):
        tt.test_tree_221_diagram()


def test_rope_sign_error_is_caught(monkeypatch):
    orig = attention.apply_rope

    def wrong(x, pos, theta):
        return orig(x, -np.asarray(pos), theta)
    monkeypatch.setattr(attention, "apply_rope", wrong)
    with pytest.raises(AssertionError):
        tat.test_rope_closed_forms()


def test_rope_frequency_exponent_error_is_caught(monkeypatch):
    monkeypatch.setattr(attention, "rope_inv_freq",
                        lambda d, th: np.power(float(th), -np.arange(d // 2) / d))
    with pytest.raises(AssertionError):
        tat.test_rope_closed_forms()


def test_position_without_depth_is_caught(monkeypatch):
    monkeypatch.setattr(attention, "position_ids",
                        lambda parents, p: np.full(len(parents), p, dtype=np.int64))
    with pytest.raises(AssertionError):
        tat.test_each_node_equals_causal_pass_over_its_chain([-1, 0, 0, 1, 1, 2])


def test_unmasked_tree_part_is_caught(monkeypatch):
    monkeypatch.setattr(attention, "tree_mask", lambda p: np.ones((len(p), len(p)), bool))
    with pytest.raises(AssertionError):
        tat.test_non_ancestors_do_not_matter()


def test_score_product_instead_of_sum_is_caught(monkeypatch):
    orig = draft.expand_level

    def wrong(logits, k, parent_scores=None, parent_store=None, product=False):
        lv = orig(logits, k, parent_scores, parent_store, product)
        if parent_scores is not None:
            r = np.asarray(logits).shape[0]
            for s in range(r):
                for c in range(k):
                    lv.cu[s * k + c] = np.float32(parent_scores[s] * lv.logp[s * k + c])
            lv.selected = draft.topk_by_score(lv.cu, k)
        return lv
    monkeypatch.setattr(draft, "expand_level", wrong)
    with pytest.raises(AssertionError):
        td.test_store_score_is_path_sum_of_logp(0)


def test_tie_to_higher_index_is_caught(monkeypatch):
    def wrong(row, k):
        x = np.asarray(row, dtype=np.float64)
        return np.lexsort((-np.arange(x.size), -x))[:k].astype(np.int32)
    monkeypatch.setattr(draft, "row_topk", wrong)
    with pytest.raises(AssertionError):
        td.test_exact_ties_take_lower_indices()


def test_walk_ignoring_tokens_is_caught(monkeypatch):
    def wrong(tokens, parents, target):
        path, node = [0], 0
        kids = tree.children_of(parents)
        while kids[node]:
            node = kids[node][0]
            path.append(node)
        return path, int(target[node])
    monkeypatch.setattr(accept, "greedy_walk", wrong)
    with pytest.raises(AssertionError):
        ta.test_walk_on_the_221_tree()


def test_in_place_compaction_order_error_is_caught(monkeypatch):
    def wrong(cache, p_len, path):
        out = np.array(cache, copy=True)
        for i in reversed(range(len(path))):      # decreasing order reads clobbered rows
            out[..., p_len + i, :] = out[..., p_len + path[i], :]
        return out
    monkeypatch.setattr(accept, "compact", wrong)
    with pytest.raises(AssertionError):
        ta.test_compaction_moves_rows_and_keeps_the_rest()


def _lm_head_variant(later_tie_wins=False, drop_chunk_offset=False, smallest=False):
    """lm_head_argmax with one planted mistake (written out here, not shared)."""
    def f(hidden, weight, chunk=8192):
        h = np.asarray(hidden, np.float64)
        rows, v = h.shape[0], weight.shape[0]
        best = np.full(rows, np.inf if smallest else -np.inf)
        idx = np.zeros(rows, np.int64)
        for v0 in range(0, v, chunk):
            lg = h @ np.asarray(weight[v0:v0 + chunk], np.float64).T
            j = lg.argmin(axis=1) if smallest else lg.argmax(axis=1)
            m = lg[np.arange(rows), j]
            if smallest:
                better = m < best
            else:
                better = m >= best if later_tie_wins else m > best
            best[better] = m[better]
            idx[better] = (0 if drop_chunk_offset else v0) + j[better]
        return idx, best
    return f


@pytest.mark.parametrize("mistake", ["later_tie_wins", "drop_chunk_offset", "smallest"])
def test_lm_head_mistakes_are_caught(monkeypatch, mistake):
    from oracle import lm_head
    from tests import test_oracle_lm_head as tl
    monkeypatch.setattr(lm_head, "lm_head_argmax", _lm_head_variant(**{mistake: True}))
    pins = (tl.test_planted_rows_win_by_a_margin, tl.test_ties_go_to_the_lower_index_across_chunks,
            tl.test_negative_logits_and_a_single_entry)
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1


def _mutant(module, name, old, new):
    """module.name with one planted change (a textual substitution of its source)."""
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(getattr(module, name)))
    assert old in src, old
    ns = dict(vars(module))
    exec(compile(src.replace(old, new, 1), f"<mutant {name}>", "exec"), ns)
    return ns[name]


SAMPLING_MISTAKES = [
    # (function, planted change, the pin that must fail)
    ("rejection_walk", "p = resid / s", "p = resid",
     "test_first_emitted_token_follows_the_target"),
    ("rejection_walk", "resid[x] = 0.0", "pass",
     "test_first_emitted_token_follows_the_target"),
    # the draft side kept fixed: right only for siblings drawn with replacement
    ("rejection_walk", "qc[x] = 0.0", "pass",
     "test_first_token_distribution_is_exact_for_draws_without_replacement"),
    ("rejection_walk", "qc[x] = 0.0", "pass", "test_first_emitted_token_follows_the_target"),
    # the residual formed with the q of the next draw instead of the one x was tested with
    ("rejection_walk", """resid = np.maximum(0.0, p - qc)
                # the next sibling was drawn from q without the tokens drawn before it
                qc[x] = 0.0
                sq = qc.sum()
                if sq > 0.0:
                    qc = qc / sq""", """qc[x] = 0.0
                sq = qc.sum()
                if sq > 0.0:
                    qc = qc / sq
                resid = np.maximum(0.0, p - qc)""",
     "test_first_token_distribution_is_exact_for_draws_without_replacement"),
    ("rejection_walk", "if u_node[c] < min(1.0, ratio):", "if u_node[c] >= min(1.0, ratio):",
     "test_zero_temperature_is_the_greedy_walk"),
    ("filter_probs", "if not first and before >= top_p * total:",
     "if not first and before + e[t] > top_p * total:",
     "test_top_p_keeps_the_token_that_crosses"),
    ("filter_probs", "total = e[keep].sum()", "total = e.sum()",
     "test_top_p_applies_to_the_renormalised_top_k"),
    ("filter_probs", "keep &= e >= min(min_p, 1.0) * e[keep].max()",
     "keep &= e >= min(min_p, 1.0) * e.sum()",
     "test_min_p_is_relative_to_the_largest"),
    ("filter_probs", "order = np.lexsort((np.arange(v), -lg))",
     "order = np.lexsort((-np.arange(v), -lg))", "test_top_k_keeps_the_lower_id_on_a_tie"),
    ("sample_inverse_cdf", 'side="right"', 'side="left"', "test_inverse_cdf_skips_zero_mass"),
]


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("fn,old,new,pin", SAMPLING_MISTAKES)
def test_sampling_mistakes_are_caught(monkeypatch, fn, old, new, pin):
    import inspect

    from oracle import sampling
    from tests import test_oracle_sampling as ts
    monkeypatch.setattr(sampling, fn, _mutant(sampling, fn, old, new))
    test = getattr(ts, pin)
    marks = getattr(test, "pytestmark", [])
    cases = []
    for m in marks:
        if m.name == "parametrize":
            names = [a.strip() for a in m.args[0].split(",")]
            for vals in m.args[1]:
                cases.append(dict(zip(names, vals if len(names) > 1 else (vals,))))
    cases = cases or [{}]
    failed = 0
    for case in cases:
        try:
            test(**case)
        except AssertionError:
            failed += 1
    assert failed >= 1, f"{fn}: {new!r} passed every case of {pin}"
    assert inspect.isfunction(test)


VARIANT_MISTAKES = [
    ("expand_level", "cu[flat] = F32(parent_scores[s]) * F32(math.exp(float(logp[flat])))",
     "cu[flat] = F32(parent_scores[s]) + F32(math.exp(float(logp[flat])))",
     "test_product_scores_are_the_exponentials_of_the_log_sums"),
    ("map_draft_to_target", "for i in range(1, num_nodes):", "for i in range(0, num_nodes):",
     "test_draft_to_target_map"),
    ("fixed_tree", "for t in row_topk(lg[f], width):",
     "for t in np.argsort(-lg[f])[:width][::-1]:", "test_fixed_tree_by_hand_and_by_property"),
]


@pytest.mark.parametrize("fn,old,new,pin", VARIANT_MISTAKES)
def test_expansion_variant_mistakes_are_caught(monkeypatch, fn, old, new, pin):
    from oracle import draft
    from tests import test_oracle_draft as td
    monkeypatch.setattr(draft, fn, _mutant(draft, fn, old, new))
    with pytest.raises(AssertionError):
        getattr(td, pin)()


def test_grown_mask_without_the_parent_rows_is_caught(monkeypatch):
    from oracle import tree as Tr
    from tests import test_oracle_tree as tt2
    monkeypatch.setattr(Tr, "grow_level_mask", _mutant(
        Tr, "grow_level_mask", "bottom = np.concatenate([parent_rows, np.eye(k, dtype=bool)], axis=1)",
        "bottom = np.concatenate([np.zeros_like(parent_rows), np.eye(k, dtype=bool)], axis=1)"))
    with pytest.raises(AssertionError):
        tt2.test_grown_level_masks_equal_the_ancestor_mask()
