"""The pins hold the oracle: plausible slips planted in it must turn a pin red (CPU only).

Each case rewrites one line of one oracle function (the source text is edited and compiled in
the oracle module's own namespace, so the oracle's other functions call the slipped version),
then runs the pins that guard that step; at least one of them must fail.  The original text
must occur exactly once, so a case cannot pass by no longer matching the oracle.
"""
import inspect
import sys

import pytest

import oracle
import oracle.bf16 as bf16_mod
import oracle.wave_buffer as wb
import oracle.wave_index as wi_mod
import test_oracle_pins as pins
import test_oracle_wave_buffer as wb_pins


def _slipped(module, name, old, new):
    """`module.name` with `old` replaced by `new` in its source, defined in the module's namespace."""
    src = inspect.getsource(getattr(module, name))
    assert src.count(old) == 1, (name, old)
    ns = dict(vars(module))
    exec(compile(src.replace(old, new), f"<slipped {name}>", "exec"), ns)
    return ns[name]


def _plant(monkeypatch, module, name, fn):
    """Put fn in place of module.name, in the module and where the package re-exports it."""
    monkeypatch.setattr(module, name, fn)
    if getattr(oracle, name, None) is not None:
        monkeypatch.setattr(oracle, name, fn)


def _plant_method(monkeypatch, cls, name, old, new):
    """cls.name with `old` replaced by `new` in its source (dedented), defined in its module's namespace."""
    src = inspect.getsource(getattr(cls, name))
    lines = src.splitlines(keepends=True)
    indent = len(lines[0]) - len(lines[0].lstrip())
    src = "".join(l[indent:] if l.strip() else l for l in lines)
    assert src.count(old) == 1, (name, old)
    ns = dict(vars(sys.modules[cls.__module__]))
    exec(compile(src.replace(old, new), f"<slipped {cls.__name__}.{name}>", "exec"), ns)
    monkeypatch.setattr(cls, name, ns[name])


def _some_pin_fails(checks):
    for check in checks:
        try:
            check()
        except Exception:      # an assertion, or arithmetic that a slip broke outright
            return True
    return False


# (function, original text, slipped text, the pins that guard it)
CASES = {
    "update sums raw keys": (
        wi_mod, "update", "np.add.at(u, a, _unit_rows(k_idx))", "np.add.at(u, a, k_idx)",
        [pins.test_update_sums_unit_vectors_hand_value, pins.test_kmeans_second_round_centroid_hand_value]),
    "update resets empty clusters": (
        wi_mod, "update", "c = c_prev.copy()", "c = np.zeros_like(c_prev)",
        [pins.test_update_empty_cluster_keeps_previous_centroid]),
    "update skips the final normalisation": (
        wi_mod, "update", "c[ne] = bf16_round(_unit_rows(u[ne]))", "c[ne] = bf16_round(u[ne])",
        [pins.test_update_sums_unit_vectors_hand_value, pins.test_kmeans_second_round_centroid_hand_value]),
    "init takes raw keys as seeds": (
        wi_mod, "init_centroids", "return bf16_round(_unit_rows(seeds))", "return bf16_round(seeds)",
        [pins.test_zero_keys_have_no_direction, pins.test_kmeans_second_round_centroid_hand_value]),
    "assignment ties to the highest id": (
        wi_mod, "assign", "return np.argmax(scores, axis=1)",
        "return scores.shape[1] - 1 - np.argmax(scores[:, ::-1], axis=1)",
        [pins.test_ties_go_to_lowest_id, pins.test_kmeans_second_round_centroid_hand_value]),
    "assignment by the farthest centroid": (
        wi_mod, "assign", "return np.argmax(scores, axis=1)", "return np.argmin(scores, axis=1)",
        [pins.test_brute_force_tiny, pins.test_planted_clusters_recovered]),
    "top-k ties to the highest id": (
        wi_mod, "select_topk", "order = np.lexsort((ids, -scores[ids]))", "order = np.lexsort((-ids, -scores[ids]))",
        [pins.test_ties_go_to_lowest_id]),
    "top-k keeps the lowest scores": (
        wi_mod, "select_topk", "order = np.lexsort((ids, -scores[ids]))", "order = np.lexsort((ids, scores[ids]))",
        [pins.test_brute_force_tiny]),
    "estimate drops the counts n_j": (
        wi_mod, "decode_unit", "D = np.exp(l - M).sum() + (nE * np.exp(e - M)).sum()",
        "D = np.exp(l - M).sum() + np.exp(e - M).sum()",
        [pins.test_two_token_cluster_estimate_closed_form, pins.test_estimate_is_jensen_lower_bound_per_cluster]),
    "estimate numerator scaled by the counts": (
        wi_mod, "decode_unit", "N = np.exp(l - M) @ vx + np.exp(e - M) @ vs[E]",
        "N = np.exp(l - M) @ vx + (nE * np.exp(e - M)) @ vs[E]",
        [pins.test_two_token_cluster_estimate_closed_form, lambda: pins.test_singleton_clusters_make_estimation_exact(3)]),
    "logits scaled by 1/d": (
        wi_mod, "decode_unit", "scale = 1.0 / math.sqrt(d)", "scale = 1.0 / d",
        [lambda: pins.test_all_clusters_selected_is_full_attention(4)]),
    "retrieved clusters also estimated": (
        wi_mod, "decode_unit", "E[R] = False", "E[R] = E[R]",
        [lambda: pins.test_all_clusters_selected_is_full_attention(4),
         pins.test_two_token_cluster_estimate_closed_form]),
    "index centroid is the unit-norm mean": (
        wi_mod, "build_unit_index", "mu[ne] = bf16_round(ksum[ne] / counts[ne, None])",
        "mu[ne] = bf16_round(_unit_rows(ksum[ne]))",
        [lambda: pins.test_singleton_clusters_make_estimation_exact(3), pins.test_two_token_cluster_estimate_closed_form]),
    "members listed in reverse position order": (
        wi_mod, "build_unit_index", 'perm = idx[np.argsort(assignment[idx], kind="stable")]',
        "perm = idx[np.lexsort((-idx, assignment[idx]))]",
        [pins.test_index_conservation, pins.test_segments_are_clustered_independently]),
    "value sums of the keys": (
        wi_mod, "build_unit_index", "np.add.at(vsum, assignment[idx], V[idx])",
        "np.add.at(vsum, assignment[idx], K[idx])",
        [pins.test_index_conservation, lambda: pins.test_singleton_clusters_make_estimation_exact(3)]),
    "local window one token short": (
        wi_mod, "steady_positions", "hi = np.arange(max(n - p.local_window, p.n_sink), n)",
        "hi = np.arange(max(n - p.local_window + 1, p.n_sink), n)",
        [pins.test_steady_zone_partition, lambda: pins.test_all_clusters_selected_is_full_attention(4)]),
    "budget rounded down": (
        wi_mod, "budget_k", "return int(math.ceil(p.budget_frac * n_clusters))",
        "return int(math.floor(p.budget_frac * n_clusters))",
        [pins.test_budget_matches_configured_counts]),
    "bf16 rounding truncates": (
        bf16_mod, "bf16_round", "np.rint(np.ldexp(m, 8))", "np.trunc(np.ldexp(m, 8))",
        [pins.test_bf16_round_matches_torch_cast, pins.test_bf16_round_hand_values]),
    "bf16 rounding keeps one bit too many": (
        bf16_mod, "bf16_round", "return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)",
        "return np.ldexp(np.rint(np.ldexp(m, 9)), e - 9)",
        [pins.test_bf16_round_matches_torch_cast, pins.test_bf16_round_hand_values]),
    "sinks not in the steady zone": (
        wi_mod, "steady_positions", "lo = np.arange(min(p.n_sink, n))", "lo = np.arange(0)",
        [pins.test_steady_zone_partition, lambda: pins.test_all_clusters_selected_is_full_attention(4)]),
    "growth one segment early": (
        wi_mod, "grown_segments", "return n_appended // p.seg_len",
        "return (n_appended + p.local_window) // p.seg_len",
        [pins.test_budget_counts_grown_clusters, pins.test_all_clusters_after_growth_is_full_attention,
         pins.test_grown_segment_equals_build_of_that_segment_alone,
         lambda: pins.test_window_keeps_between_w_and_w_plus_s_rows(300, 0)]),
    "growth one append late": (
        wi_mod, "grown_segments", "return n_appended // p.seg_len", "return max(n_appended - 1, 0) // p.seg_len",
        [lambda: pins.test_window_keeps_between_w_and_w_plus_s_rows(8, 512),
         lambda: pins.test_window_keeps_between_w_and_w_plus_s_rows(300, 512)]),
    "grown segment taken from the window's end": (
        wi_mod, "grow_unit_index", "pos = w0 + g * S + np.arange(S)", "pos = K_all.shape[0] - S + np.arange(S)",
        [pins.test_grown_segment_equals_build_of_that_segment_alone, pins.test_all_clusters_after_growth_is_full_attention]),
    "group retrieval by the first head's scores": (
        wi_mod, "decode_unit", "select_topk(mu @ q_heads.sum(axis=0), nonempty, k)",
        "select_topk(mu @ q_heads[0], nonempty, k)",
        [pins.test_group_topk_variant_pins]),
    "dense comparator without the appended rows": (
        wi_mod, "full_attention", "if k_app is not None and k_app.shape[1] > 0:", "if False:",
        [pins.test_full_attention_equals_wave_index_with_every_cluster_retrieved, pins.test_full_attention_closed_forms]),
    "merge rescales with the wrong sign": (
        wi_mod, "lse_merge", "Z = sum(z * math.exp(m - M) for m, z, _ in parts if m > -np.inf)",
        "Z = sum(z * math.exp(M - m) for m, z, _ in parts if m > -np.inf)",
        [pins.test_lse_merge_associative]),
}


@pytest.mark.parametrize("case", list(CASES))
def test_pins_catch_planted_slip(case, monkeypatch):
    module, name, old, new, checks = CASES[case]
    for check in checks:          # the pins pass on the oracle as written
        check()
    _plant(monkeypatch, module, name, _slipped(module, name, old, new))
    assert _some_pin_fails(checks), f"no pin caught: {case}"


LRU_CASES = {
    "hit not made most recently used": (
        "self.lru.move_to_end(p)\n", "pass\n"),
    "evicts the most recently used page": (
        "victim, last = next(iter(self.lru.items()))", "victim, last = next(reversed(self.lru.items()))"),
    "no protection within the round": (
        "if last == t:", "if False:"),
    "highest free slot": (
        "s = min(self.free)", "s = max(self.free)"),
}


@pytest.mark.parametrize("case", list(LRU_CASES))
def test_wave_buffer_pins_catch_planted_slip(case, monkeypatch):
    old, new = LRU_CASES[case]
    checks = [wb_pins.test_hand_worked_lru_trace, wb_pins.test_round_order_and_same_round_protection,
              wb_pins.test_free_slot_is_the_lowest, lambda: wb_pins.test_matches_brute_force_lru(0)]
    for check in checks:
        check()
    _plant_method(monkeypatch, wb.LruPagePolicy, "round", old, new)
    assert _some_pin_fails(checks), f"no pin caught: {case}"
