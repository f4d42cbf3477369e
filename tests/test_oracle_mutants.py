"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a private copy of the oracle (its C source or
its Python steps) on the CPU: a dropped term, a transposed operand, a wrong
index or sign, a missing normalisation, an off-by-one range. The copy is built
and imported on its own, every pin of test_oracle_pins runs against it, and at
least one pin must fail. The real oracle is never modified.
"""
import importlib.util
import inspect
import os

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
ORACLE_DIR = os.path.join(ROOT, "oracle")
GOLDEN = os.path.join(HERE, "golden")

C, PY = "tb_oracle.c", "__init__.py"

# (name, file, text in the oracle, planted replacement)
MUTANTS = [
    # bf16 rounding
    ("bf16_ties_away_from_zero", C, "double m = nearbyint(ldexp(a, -q));", "double m = round(ldexp(a, -q));"),
    ("bf16_truncates", C, "double m = nearbyint(ldexp(a, -q));", "double m = floor(ldexp(a, -q));"),
    ("bf16_nine_significant_bits", C, "int q = e - 8; ", "int q = e - 9; "),
    ("bf16_subnormal_spacing", C, "if (q < -133) q = -133;", "if (q < -134) q = -134;"),
    # projection
    ("project_drops_last_term", C,
     "for (int d = 0; d < D; ++d)\n                        acc += tbo_bf16_to_double(Kh[t * D + d])",
     "for (int d = 0; d < D - 1; ++d)\n                        acc += tbo_bf16_to_double(Kh[t * D + d])"),
    ("project_transposed_Wk", C, "W[(int64_t)d * dp + j]", "W[(int64_t)j * D + d]"),
    ("project_rounds_a_biased_sum", C, "Ph[t * dp + j] = tbo_bf16_from_double(acc);",
     "Ph[t * dp + j] = tbo_bf16_from_double(acc * (1.0 + 0x1p-9));"),
    # scores
    ("score_mean_not_divided", C, "? best : sum / G;", "? best : sum;"),
    ("score_heads_interleaved", C, "(int64_t)h * G + g) * dp", "(int64_t)g * Hkv + h) * dp"),
    ("score_max_is_min", C, "if (dot > best) best = dot;", "if (dot < best || best == -INFINITY) best = dot;"),
    ("score_wrong_sign", C, "dot += p;", "dot -= p;"),
    ("score_drops_last_term", C, "for (int i = 0; i < dp; ++i) {", "for (int i = 0; i < dp - 1; ++i) {"),
    # top-k
    ("topk_ties_to_higher_index", C, "return (a->i < b->i) ? -1 : (a->i > b->i);",
     "return (a->i > b->i) ? -1 : (a->i < b->i);"),
    ("topk_keeps_smallest", C, "if (a->s > b->s) return -1;\n    if (a->s < b->s) return 1;",
     "if (a->s < b->s) return -1;\n    if (a->s > b->s) return 1;"),
    ("topk_positive_zero_above_negative", C, "if (a->s > b->s) return -1;\n    if (a->s < b->s) return 1;",
     "if (a->s > b->s || (a->s == b->s && signbit(b->s) && !signbit(a->s))) return -1;\n"
     "    if (a->s < b->s || (a->s == b->s && signbit(a->s) && !signbit(b->s))) return 1;"),
    ("topk_output_in_rank_order", C, "qsort(out, (size_t)k, sizeof *out, tbo_int_cmp);", ""),
    ("topk_one_short", C, "for (int64_t j = 0; j < k; ++j) out[j] = p[j].i;",
     "for (int64_t j = 0; j < k; ++j) out[j] = p[j + (j == k - 1 && k < n)].i;"),
    # neighbour fetching and the tail
    ("expand_window_one_short", C, "for (int64_t t = i - r; t <= i + r; ++t)",
     "for (int64_t t = i - r + (r > 0); t <= i + r; ++t)"),
    ("expand_drops_first_tail_token", C, "for (int64_t t = n_pred; t < n_t; ++t)",
     "for (int64_t t = n_pred + 1; t < n_t; ++t)"),
    ("expand_not_clipped_to_prediction", C, "if (t >= 0 && t < n_pred) mask[t] = 1;",
     "if (t >= 0 && t < n_pred - 1) mask[t] = 1;"),
    # attention
    ("attn_no_scale", C, "z[j] = scale * dot;", "z[j] = dot;"),
    ("attn_denominator_skips_first_row", C, "for (int64_t j = 0; j < c; ++j) denom += exp(z[j] - zmax);",
     "for (int64_t j = 1; j < c; ++j) denom += exp(z[j] - zmax);"),
    ("attn_gqa_mapping", C, "int h = hq / G;", "int h = hq % Hkv;"),
    ("attn_unnormalised", C, "double w = exp(z[j] - zmax) / denom;", "double w = exp(z[j] - zmax);"),
    ("attn_numerator_without_max", C, "double w = exp(z[j] - zmax) / denom;", "double w = exp(z[j]) / denom;"),
    ("attn_value_row_of_key", C, "o[d] += w * tbo_bf16_to_double(Vh[t * D + d]);",
     "o[d] += w * tbo_bf16_to_double(Kh[t * D + d]);"),
    # the decode step's schedule (Python)
    ("interval_scores_before_append", PY, "s, _ = score(q_imp, np.ascontiguousarray(Kp[:, :, :n_t, :]), agg)",
     "s, _ = score(q_imp, np.ascontiguousarray(Kp[:, :, :n, :]), agg)"),
    ("interval_reuse_forgets_tail", PY, "    sel, counts = expand(state.idx, r, state.n_pred, n_t)\n",
     "    sel, counts = expand(state.idx, r, state.n_pred, state.n_pred)\n"),
    ("decode_ignores_budget_rule", PY, "state.idx = topk(s, centres(k, r, budget_neighbours))",
     "state.idx = topk(s, k)"),
    ("decode_predicts_every_step", PY,
     "if t % T == 0:\n        s, _ = score(q_imp, np.ascontiguousarray(Kp[:, :, :n_t, :]), agg)",
     "if True:\n        s, _ = score(q_imp, np.ascontiguousarray(Kp[:, :, :n_t, :]), agg)"),
    ("centres_ignore_width", PY, "return max(1, k // (2 * r + 1)) if budget_neighbours else k",
     "return max(1, k // (r + 1)) if budget_neighbours else k"),
    # buffered step (Python)
    ("buffered_window_misses_newest", PY, "list(range(pre)) + sorted(body) + list(range(tail0, n_t))",
     "list(range(pre)) + sorted(body) + list(range(tail0, n_t - 1))"),
    ("buffered_projects_into_window", PY, "while n_t - W - P >= W:", "while n_t - P >= W:"),
    ("buffered_neighbours_cross_sink", PY, "if S <= j < P)", "if 0 <= j < P)"),
    ("buffered_sink_one_short", PY, "pre = min(S, n_t)", "pre = min(S - 1, n_t)"),
    ("buffered_centres_not_offset_by_sink", PY, "range(S + i - r, S + i + r + 1)", "range(i - r, i + r + 1)"),
    ("buffered_scores_include_sink", PY, "Kp[:, :, S:P, :]", "Kp[:, :, 0:P, :]"),
    ("buffered_reuse_drops_new_token", PY, "state.sel_rows = [row + [n] for row in state.sel_rows]",
     "state.sel_rows = [list(row) for row in state.sel_rows]"),
    # ragged batch (Python)
    ("ragged_uses_first_length", PY, "o, sl, c = decode_step(states[b], t, int(nb),",
     "o, sl, c = decode_step(states[b], t, int(ns[0]),"),
    # predictor (Python)
    ("silu_wrong_sign", PY, "return v / (1.0 + np.exp(-v))", "return v / (1.0 + np.exp(v))"),
    ("predictor_no_activation", PY, "h = silu(xf @ w1.T)", "h = xf @ w1.T"),
]


def _oracle_copy(tmp_path, file, old, new):
    d = tmp_path / "oracle_copy"
    d.mkdir()
    for f in (PY, C):
        with open(os.path.join(ORACLE_DIR, f)) as fh:
            src = fh.read()
        if f == file:
            assert src.count(old) == 1, f"mutation target not unique in {f}: {old!r}"
            src = src.replace(old, new)
        (d / f).write_text(src)
    name = f"oracle_copy_{tmp_path.name}"
    spec = importlib.util.spec_from_file_location(name, str(d / PY), submodule_search_locations=[str(d)])
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    return mod


def _pins(tmp_path):
    """A private instance of test_oracle_pins and every (pin, arguments) call it defines."""
    spec = importlib.util.spec_from_file_location(f"pins_{tmp_path.name}", os.path.join(HERE, "test_oracle_pins.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    calls = []
    for name, fn in vars(mod).items():
        if not name.startswith("test_") or not inspect.isfunction(fn):
            continue
        combos = [{}]
        for m in getattr(fn, "pytestmark", []):
            if m.name != "parametrize":
                continue
            names = [s.strip() for s in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
            grown = []
            for c in combos:
                for v in m.args[1]:
                    v = getattr(v, "values", v)
                    v = tuple(v) if len(names) > 1 else (v[0] if isinstance(v, tuple) and len(v) == 1 else v,)
                    grown.append({**c, **dict(zip(names, v))})
            combos = grown
        for c in combos:
            kw = dict(c)
            if "golden_dir" in inspect.signature(fn).parameters:
                kw["golden_dir"] = GOLDEN
            calls.append((name, fn, kw))
    return mod, calls


def test_real_oracle_passes_every_pin_through_the_harness(tmp_path):
    pins, calls = _pins(tmp_path)
    import oracle
    pins.oracle = oracle
    assert len(calls) >= 30
    for _, fn, kw in calls:
        fn(**kw)


@pytest.mark.parametrize("name,file,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_a_pin_catches_the_planted_mistake(tmp_path, name, file, old, new):
    mutant = _oracle_copy(tmp_path, file, old, new)
    pins, calls = _pins(tmp_path)
    pins.oracle = mutant
    for pin, fn, kw in calls:
        try:
            fn(**kw)
        except Exception:   # the pin failed (or the oracle's own checks refused): caught
            return
    pytest.fail(f"no pin fails with the planted mistake {name}")
