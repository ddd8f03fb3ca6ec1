"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake into a copy of the oracle's C++ source: a
flipped sign, a dropped term, a wrong index or head mapping, a transposed operand, a
lost accumulation.  It builds that copy as a library of its own and runs the pins of
test_oracle.py against it.  Every planted mistake must make at least one pin fail, and
the unchanged copy must pass them all.

Two kinds of pin compare the oracle with itself:
- the stored golden fixture;
- the row-sampled entry points against the full ones.
The fixture never counts.  The row-sampled comparison counts only for mistakes planted
in the row-sampled functions.  So every kill of a mistake in the full forward or
backward comes from a pin outside the oracle: finite differences, closed forms,
rotation and softmax invariants, or PyTorch's fp64 attention.
"""
import importlib.util
import os
from concurrent.futures import ThreadPoolExecutor

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
ORACLE_DIR = os.path.join(ROOT, "oracle")

# Pins that hold the oracle to something outside itself.
INDEPENDENT_PINS = (
    "test_rope_table_hand_values",
    "test_rope_theta_is_a_parameter",
    "test_rope_pairs_are_adjacent_and_rotate_counterclockwise",
    "test_rope_preserves_norms_and_depends_only_on_offset",
    "test_hand_case_two_positions_two_dims",
    "test_row_zero_attends_only_to_itself",
    "test_zero_queries_give_causal_running_mean",
    "test_probability_rows_sum_to_one_and_mask_is_exact_zero",
    "test_gqa_equals_mha_with_repeated_kv",
    "test_delta_is_rowsum_of_dO_times_O",
    "test_backward_matches_central_finite_differences",
    "test_matches_torch_sdpa_fp64_with_autograd",
    "test_row_sampled_oracle_zero_queries_closed_form",
    "test_prologue_rows_have_unit_rms_and_ignore_the_row_scale",
    "test_prologue_matches_torch_rms_norm_matmul_and_rope",
)
ROW_CONSISTENCY_PIN = "test_row_sampled_oracle_matches_full_oracle"

# (name, part, edits): part "full" for the full forward/backward and the rotation,
# "rows" for the row-sampled entry points; each edit is (text, replacement, k) and
# replaces the k-th occurrence (0-based) of the text in the source.
S_DECL = "const double s = 1.0 / std::sqrt((double)D);"
MUTANTS = [
    # rotary embedding
    ("rope_rotates_clockwise", "full", [("out[2 * i] = x0 * c - x1 * s;", "out[2 * i] = x0 * c + x1 * s;", 0)]),
    ("rope_frequency_exponent_halved", "full",
     [("std::pow(theta, -2.0 * (double)i / (double)D)", "std::pow(theta, -1.0 * (double)i / (double)D)", 0)]),
    ("rope_half_split_pairs", "full",
     [("double x0 = x[2 * i], x1 = x[2 * i + 1];", "double x0 = x[i], x1 = x[i + D / 2];", 0)]),
    ("rope_positions_start_at_one", "full", [("return (double)t * std::pow", "return (double)(t + 1) * std::pow", 0)]),
    ("rope_theta_ignored", "full", [("std::pow(theta, ", "std::pow(10000.0, ", 0)]),
    ("gradients_rotated_forward_not_back", "full",
     [("out[2 * i] = g0 * c + g1 * s;", "out[2 * i] = g0 * c - g1 * s;", 0),
      ("out[2 * i + 1] = -g0 * s + g1 * c;", "out[2 * i + 1] = g0 * s + g1 * c;", 0)]),
    # forward
    ("logit_scale_one_over_d", "full", [(S_DECL, "const double s = 1.0 / (double)D;", 0)]),
    ("strict_causal_mask", "full",
     [("for (int j = 0; j <= i; ++j) {", "for (int j = 0; j < i; ++j) {", 0),
      ("for (int j = 0; j <= i; ++j) sum += std::exp(S[j] - m);", "for (int j = 0; j < i; ++j) sum += std::exp(S[j] - m);", 0),
      ("for (int j = 0; j <= i; ++j) P[(size_t)i * T + j]", "for (int j = 0; j < i; ++j) P[(size_t)i * T + j]", 0)]),
    ("no_causal_mask", "full",
     [("for (int j = 0; j <= i; ++j) {", "for (int j = 0; j < T; ++j) {", 0),
      ("for (int j = 0; j <= i; ++j) sum += std::exp(S[j] - m);", "for (int j = 0; j < T; ++j) sum += std::exp(S[j] - m);", 0),
      ("for (int j = 0; j <= i; ++j) P[(size_t)i * T + j]", "for (int j = 0; j < T; ++j) P[(size_t)i * T + j]", 0)]),
    ("lse_drops_row_max", "full", [("lse[i] = m + std::log(sum);", "lse[i] = std::log(sum);", 0)]),
    ("gqa_heads_interleaved_forward", "full", [("const int g = h / G;", "const int g = h % Hkv;", 0)]),
    ("pv_reads_query_row_of_v", "full",
     [("acc += P[(size_t)i * T + j] * v[idx4(b, j, g, d, T, Hkv, D)];",
       "acc += P[(size_t)i * T + j] * v[idx4(b, i, g, d, T, Hkv, D)];", 0)]),
    # backward
    ("backward_logit_scale_one_over_d", "full", [(S_DECL, "const double s = 1.0 / (double)D;", 1)]),
    ("gqa_heads_interleaved_backward", "full",
     [("for (int h = g * G; h < (g + 1) * G; ++h) {", "for (int h = g; h < Hq; h += Hkv) {", 0)]),
    ("dp_reads_query_row_of_v", "full",
     [("acc += dO[idx4(b, i, h, d, T, Hq, D)] * v[idx4(b, j, g, d, T, Hkv, D)];",
       "acc += dO[idx4(b, i, h, d, T, Hq, D)] * v[idx4(b, i, g, d, T, Hkv, D)];", 0)]),
    ("ds_drops_delta", "full", [("* (dP[(size_t)i * T + j] - delta);", "* dP[(size_t)i * T + j];", 0)]),
    ("ds_sign_flipped", "full", [("* (dP[(size_t)i * T + j] - delta);", "* (delta - dP[(size_t)i * T + j]);", 0)]),
    ("dq_drops_scale", "full", [("dqr[(size_t)i * D + d] = s * acc;", "dqr[(size_t)i * D + d] = acc;", 0)]),
    ("dq_drops_diagonal", "full",
     [("for (int j = 0; j <= i; ++j) acc += dS[(size_t)i * T + j] * kr[(size_t)j * D + d];",
       "for (int j = 0; j < i; ++j) acc += dS[(size_t)i * T + j] * kr[(size_t)j * D + d];", 0)]),
    ("dk_drops_scale", "full", [("dkr[(size_t)j * D + d] += s * acck;", "dkr[(size_t)j * D + d] += acck;", 0)]),
    ("dk_keeps_last_head_only", "full", [("dkr[(size_t)j * D + d] += s * acck;", "dkr[(size_t)j * D + d] = s * acck;", 0)]),
    ("dv_keeps_last_head_only", "full", [("dvg[(size_t)j * D + d] += accv;", "dvg[(size_t)j * D + d] = accv;", 0)]),
    ("dv_transposed_probabilities", "full",
     [("accv += P[(size_t)i * T + j] * dO[idx4(b, i, h, d, T, Hq, D)];",
       "accv += P[(size_t)j * T + i] * dO[idx4(b, i, h, d, T, Hq, D)];", 0)]),
    ("dv_reads_first_head_of_group", "full",
     [("accv += P[(size_t)i * T + j] * dO[idx4(b, i, h, d, T, Hq, D)];",
       "accv += P[(size_t)i * T + j] * dO[idx4(b, i, g * G, d, T, Hq, D)];", 0)]),
    ("dk_drops_diagonal", "full", [("for (int i = j; i < T; ++i) {", "for (int i = j + 1; i < T; ++i) {", 0)]),
    # row-sampled entry points
    # RMSNorm -> QKV projection -> RoPE prologue
    ("rms_sum_not_mean", "full", [("std::sqrt(ss / (double)dim + eps)", "std::sqrt(ss + eps)", 0)]),
    ("rms_eps_outside_sqrt", "full", [("std::sqrt(ss / (double)dim + eps)", "std::sqrt(ss / (double)dim) + eps", 0)]),
    ("rms_gain_ignored", "full", [("xh[c] = xm[c] / r * gamma[c];", "xh[c] = xm[c] / r;", 0)]),
    ("projection_transposed", "full", [("acc += w[(int64_t)n * dim + c] * xh[c];", "acc += w[(int64_t)c * N + n] * xh[c];", 0)]),
    ("kv_split_swapped", "full", [("(h < Hq + Hkv ? k + (m * Hkv + (h - Hq)) * D : v + (m * Hkv + (h - Hq - Hkv)) * D)",
                                   "(h < Hq + Hkv ? v + (m * Hkv + (h - Hq)) * D : k + (m * Hkv + (h - Hq - Hkv)) * D)", 0)]),
    ("prologue_rotates_v", "full", [("const bool rot = rotate && h < Hq + Hkv;", "const bool rot = rotate != 0;", 0)]),
    ("prologue_position_across_batch", "full", [("const int t = (int)(m % T);", "const int t = (int)m;", 0)]),
    ("rows_dq_drops_delta", "rows", [("const double ds = P[j] * (dP[j] - dl);", "const double ds = P[j] * dP[j];", 0)]),
    ("rows_gqa_heads_interleaved", "rows", [("const int g = h / (Hq / Hkv);", "const int g = h % Hkv;", 0)]),
    ("rows_lse_drops_row_max", "rows", [("const double l = m + std::log(sum);", "const double l = std::log(sum);", 0)]),
    ("rows_logit_scale_one_over_d", "rows", [(S_DECL, "const double s = 1.0 / (double)D;", 2)]),
    ("krows_drops_diagonal", "rows", [("for (int i = j; i < T; ++i) {", "for (int i = j + 1; i < T; ++i) {", 1)]),
    ("krows_dk_drops_scale", "rows",
     [("acck[(size_t)r * D + d] += s * ds * qi[d];", "acck[(size_t)r * D + d] += ds * qi[d];", 0)]),
    ("krows_first_head_only", "rows",
     [("for (int h = g * G; h < (g + 1) * G; ++h) {", "for (int h = g * G; h < g * G + 1; ++h) {", 1)]),
    ("krows_lse_drops_row_max", "rows", [("const double l = m + std::log(sum);", "const double l = std::log(sum);", 1)]),
]


def plant(src: str, edits) -> str:
    """Apply the edits in order; a text that is no longer in the source is an error, so
    that a change to the oracle cannot quietly turn a mutant into the original."""
    for old, new, k in edits:
        pos = -1
        for _ in range(k + 1):
            pos = src.find(old, pos + 1)
            assert pos >= 0, f"mutation target {old!r} (occurrence {k}) not in the oracle source"
        src = src[:pos] + new + src[pos + len(old):]
    return src


def _load_module(name: str, path: str):
    spec = importlib.util.spec_from_file_location(name, path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="module")
def variants(tmp_path_factory):
    """Every mutant and the unchanged source, each compiled to its own library (in
    parallel), keyed by name."""
    import oracle
    with open(os.path.join(ORACLE_DIR, "neattn_ref.cpp")) as f:
        src = f.read()
    out_dir = tmp_path_factory.mktemp("oracle_mutants")
    sources = {"unchanged": src}
    for name, _, edits in MUTANTS:
        sources[name] = plant(src, edits)
        assert sources[name] != src, name

    def compile_one(item):
        name, text = item
        cpp = out_dir / f"{name}.cpp"
        cpp.write_text(text)
        return name, oracle.compile_source(str(cpp), str(out_dir / f"lib_{name}.so"))

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        return dict(ex.map(compile_one, sources.items()))


def _oracle_on(lib_path: str, name: str):
    """A fresh instance of the oracle's Python binding that loads `lib_path`."""
    mod = _load_module(f"oracle_variant_{name}", os.path.join(ORACLE_DIR, "__init__.py"))
    mod.build = lambda force=False: lib_path
    return mod


def _pin_calls(pins_mod, names):
    """(label, function, kwargs) for every case of the named pins, parametrised ones
    expanded from their own parametrize marks."""
    calls = []
    for name in names:
        fn = getattr(pins_mod, name)
        cases = [{}]
        for mark in getattr(fn, "pytestmark", []):
            if mark.name == "parametrize":
                arg, values = mark.args[0], mark.args[1]
                cases = [{arg: v} for v in values]
        calls += [(f"{name}{list(c.values()) or ''}", fn, c) for c in cases]
    return calls


def _failing(mod, calls):
    failed = []
    for label, fn, kwargs in calls:
        try:
            fn(mod, **kwargs)
        except Exception:          # a failed assertion, a NaN, a rejected shape
            failed.append(label)
    return failed


@pytest.fixture(scope="module")
def pins():
    return _load_module("oracle_pins_for_mutants", os.path.join(HERE, "test_oracle.py"))


def test_unchanged_copy_passes_every_pin(variants, pins):
    mod = _oracle_on(variants["unchanged"], "unchanged")
    calls = _pin_calls(pins, INDEPENDENT_PINS + (ROW_CONSISTENCY_PIN,))
    assert _failing(mod, calls) == []


@pytest.mark.parametrize("name,part", [(m[0], m[1]) for m in MUTANTS], ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(variants, pins, name, part):
    names = INDEPENDENT_PINS + ((ROW_CONSISTENCY_PIN,) if part == "rows" else ())
    mod = _oracle_on(variants[name], name)
    failed = _failing(mod, _pin_calls(pins, names))
    assert failed, f"planted mistake {name!r} passes every pin"
