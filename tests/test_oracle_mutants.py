"""The oracle's pins catch plausible mistakes in the oracle.

Each case plants one slip in a copy of the oracle's C source (a dropped term,
a wrong sign, an off-by-one, a transposed index, a wrong head map, a wrong log
base, a wrong FP8 exponent bias), builds the copy with gcc, points the oracle
module at it, and runs the pins of test_oracle_pins.py against it: at least
one pin must fail.  Every mutant keeps its memory accesses inside the arrays
it is given (indices stay in range or meet the oracle's own range checks), so
a surviving mutant is a gap in the pins, not a crash.  The committed oracle is
never modified.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "decode_attn_oracle.c")

# (name, exact text in the oracle, planted replacement)
MUTANTS = [
    # the three-pass softmax
    ("exp_sum_without_max", "l += exp(s[j - lo] - m);", "l += exp(s[j - lo]);"),
    ("weight_sign_flipped", "const double p = exp(s[j - lo] - m) / l;",
     "const double p = exp(m - s[j - lo]) / l;"),
    ("weights_not_normalised", "const double p = exp(s[j - lo] - m) / l;",
     "const double p = exp(s[j - lo] - m);"),
    ("lse_log2", "*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    ("lse_without_max", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("scale_dropped", "s[j - lo] = J->scale * acc;", "s[j - lo] = acc;"),
    ("dot_product_drops_last_d", "for (int d = 0; d < D; ++d) acc += qd[d]",
     "for (int d = 0; d < D - 1; ++d) acc += qd[d]"),
    ("empty_row_lse_zero", "if (hi <= lo) { *lse_out = -INFINITY;",
     "if (hi <= lo) { *lse_out = 0.0;"),
    # which keys a row sees
    ("length_off_by_one", "int64_t hi = L;\n", "int64_t hi = L - 1;\n"),
    ("causal_off_by_one", "hi = L - J->q_len + 1 + t;", "hi = L - J->q_len + t;"),
    ("causal_tokens_reversed", "hi = L - J->q_len + 1 + t;", "hi = L - t;"),
    ("key_window_end_ignored", "if (hi > J->key_hi) hi = J->key_hi;", ""),
    ("key_window_start_ignored", "int64_t lo = J->key_lo > 0 ? J->key_lo : 0;",
     "int64_t lo = 0;"),
    ("row_token_index_wrong", "const int t = (int)((flat / Hq) % J->q_len);",
     "const int t = (int)(flat % J->q_len);"),
    # where the operands come from
    ("gqa_interleaved", "const int kvh = h / G;", "const int kvh = h % J->num_kv_heads;"),
    ("query_token_head_transposed", "(((int64_t)b * J->q_len + t) * Hq + h) * D",
     "(((int64_t)b * Hq + h) * J->q_len + t) * D"),
    ("block_table_ignored", "page = J->block_table[(int64_t)b * J->bt_stride + col];",
     "page = col;"),
    ("slot_off_by_one", "slot = j % J->page_size;", "slot = (j + 1) % J->page_size;"),
    ("values_read_from_key_cache", "kv_value(J, J->v, J->v_scale, vr + d)",
     "kv_value(J, J->k, J->v_scale, vr + d)"),
    # FP8 caches
    ("value_scale_dropped", "kv_value(J, J->v, J->v_scale, vr + d)",
     "kv_value(J, J->v, 1.0, vr + d)"),
    ("key_scale_dropped", "kv_value(J, J->k, J->k_scale, kr + d)",
     "kv_value(J, J->k, 1.0, kr + d)"),
    ("e4m3_normal_bias", "ldexp(8.0 + m, e - 10)", "ldexp(8.0 + m, e - 11)"),
    ("e4m3_subnormal_scale", "ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    ("e4m3_sign_dropped", "return sign ? -v : v;", "return v;"),
    # the merge of chunk results
    ("merge_weight_sum_without_max", "W += exp(pl[s] - M);", "W += exp(pl[s]);"),
    ("merge_weights_not_normalised", "const double w = exp(pl[s] - M) / W;",
     "const double w = exp(pl[s] - M);"),
    ("merge_lse_without_max", "lse[r] = M + log(W);", "lse[r] = log(W);"),
    ("merge_ignores_nvalid", "const int n = nvalid ? nvalid[r] : nsplit;",
     "const int n = nsplit;"),
]


def pin_calls():
    """(label, callable) for every pin, parametrised cases expanded, in the
    order the pin module defines them."""
    calls = []
    for name, fn in vars(pins).items():
        if not name.startswith("test_") or not callable(fn):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            calls.append((name, fn, {}))
            continue
        assert len(marks) == 1, name
        argnames = [a.strip() for a in marks[0].args[0].split(",")]
        for vals in marks[0].args[1]:
            vals = vals if len(argnames) > 1 else (vals,)
            calls.append((f"{name}{list(vals)}", fn, dict(zip(argnames, vals))))
    return calls


def build_mutant(old, new, path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique or missing: {old!r}"
    mutated = path + ".c"
    with open(mutated, "w") as f:
        f.write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o",
                           path, mutated, "-lm"])
    return path


def test_every_mutation_site_is_in_the_oracle():
    src = open(SRC).read()
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, name
        assert old != new, name


def first_failing_pin(lib, monkeypatch):
    """Label of the first pin that fails with the oracle library `lib`, or None."""
    monkeypatch.setattr(oracle, "build", lambda force=False: lib)
    monkeypatch.setattr(oracle, "_lib", None)
    for label, fn, kwargs in pin_calls():
        try:
            fn(**kwargs)
        except pytest.skip.Exception:
            continue
        except Exception:  # an assertion or an error raised by the oracle
            return label
    return None


def test_unmodified_copy_passes_every_pin(tmp_path, monkeypatch):
    # the control: the same copy-and-build route without a mutation
    lib = build_mutant("int oracle_decode_attn(", "int oracle_decode_attn(",
                       str(tmp_path / "liboracle_copy.so"))
    assert first_failing_pin(lib, monkeypatch) is None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path, monkeypatch):
    lib = build_mutant(old, new, str(tmp_path / f"liboracle_{name}.so"))
    caught_by = first_failing_pin(lib, monkeypatch)
    assert caught_by is not None, f"no pin fails with the planted mistake {name!r}"
