"""Plant one mistake at a time in a copy of the oracle (CPU only) and require
that the pins catch every one of them.  This checks the pins, not the oracle."""
import functools
import os
import subprocess

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "g3s_oracle.c")

# (name, text to replace, replacement, expected number of occurrences)
MUTANTS = [
    ("dropped_scale", "const double scale = 1.0 / sqrt((double)d);", "const double scale = 1.0;", 1),
    ("key_indexed_by_destination", "* load_elem(K, dtype, j * HD", "* load_elem(K, dtype, i * HD", 2),
    ("value_indexed_by_destination", "w * load_elem(V, dtype, j * HD", "w * load_elem(V, dtype, i * HD", 1),
    ("wrong_softmax_sign", "exp(dot * scale - m)", "exp(m - dot * scale)", 1),
    ("missing_normalisation", "o[(int64_t)h * d + f] /= wsum;", "(void)wsum;", 1),
    ("zero_degree_not_zero", "if (e1 <= e0) continue;", "if (e1 < e0) continue;", 1),
    ("variant_no_epsilon", "/= (ssum + eps);", "/= (ssum);", 1),
    ("variant_wrong_logit_clip", "exp(clampd(l, -5.0, 5.0))", "exp(clampd(l, -4.0, 4.0))", 1),
    ("variant_no_elementwise_clamp", "if (elementwise_clamp) t = clampd(t, -5.0, 5.0);", "", 1),
    ("variant_edge_feature_dropped", "const double u = t * load_elem(Eproj, dtype, e * HD + (int64_t)h * d + f);",
     "const double u = t;", 1),
    ("variant_edge_indexed_by_source", "load_elem(Eproj, dtype, e * HD", "load_elem(Eproj, dtype, j * HD", 1),
    ("variant_value_weight_unexp", "o[(int64_t)h * d + f] += s * load_elem", "o[(int64_t)h * d + f] += l * load_elem", 1),
    ("f16_exponent_bias", "expo - 25", "expo - 24", 1),
    ("bf16_shift", "(uint32_t)b << 16", "(uint32_t)b << 15", 1),
    ("aggregate_weight_of_wrong_head", "load_elem(W, dtype, e * H + h)", "load_elem(W, dtype, e * H)", 1),
    ("aggregate_feature_of_destination", "w * load_elem(X, dtype, j * HD", "w * load_elem(X, dtype, i * HD", 1),
    ("aggregate_no_epsilon", "/= (wsum + eps);", "/= (wsum);", 1),
    ("variant_scale_applied_twice", "load_elem(K, dtype, j * HD + (int64_t)h * d + f) * scale;",
     "load_elem(K, dtype, j * HD + (int64_t)h * d + f) * scale * scale;", 1),
]


def _pins_fail(lib):
    fwd = functools.partial(oracle.forward, lib=lib)
    caught = []
    agg = functools.partial(oracle.aggregate, lib=lib)
    for pin in pins.ALL_PINS + pins.AGG_PINS:
        try:
            pin(agg if pin in pins.AGG_PINS else fwd)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    return caught


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, count):
    text = open(SRC).read()
    assert text.count(old) == count, "mutation target drifted: %r" % old
    src = tmp_path / ("mut_%s.c" % name)
    src.write_text(text.replace(old, new))
    so = tmp_path / ("libmut_%s.so" % name)
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so),
                           str(src), "-lm"])
    lib = oracle.load_library(str(so))
    caught = _pins_fail(lib)
    assert caught, "no pin caught the planted mistake %s" % name
