"""Plant plausible mistakes in the oracle (on the CPU, in a temporary copy of
its source) and check that the pins catch every one of them.

A mutant is the oracle's C source with one exact text replacement; it is
compiled with the oracle's own flags into a temporary directory and run
through every pin of ``oracle_pins``.  The committed oracle is never touched.
"""
import os

import pytest

import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "es_oracle.c")

# (id, text in the float32 oracle, replacement, which occurrence (0-based))
MUTATIONS = [
    ("tanh_sign_of_decay_term", "float v = xv + ah;", "float v = xv - ah;", 0),
    ("tanh_dropped_decay_term", "float v = xv + ah;", "float v = xv;", 0),
    ("tanh_transposed_operand", "float ah = av * h[w];", "float ah = av * xv;", 0),
    ("tanh_missing_tanh", "h[w] = oracle_tanh(v);", "h[w] = v;", 0),
    ("maxplus_sign_of_cost", "float v = h[w] - cv;", "float v = h[w] + cv;", 0),
    ("maxplus_dropped_cost", "h[w] = oracle_maximum(v, xv);", "h[w] = oracle_maximum(h[w], xv);", 0),
    ("maxplus_min_instead_of_max", "if (a > b) return a;", "if (a < b) return a;", 0),
    ("maximum_zero_sign", "return signbit(a) ? b : a;", "return a;", 0),
    ("normcap_no_floor_at_one", "float d = oracle_maximum(1.0f, sqrtf(ss));", "float d = sqrtf(ss);", 0),
    ("normcap_norm_without_square", "float sq = y[w] * y[w];", "float sq = y[w] < 0 ? -y[w] : y[w];", 0),
    ("normcap_dropped_input", "y[w] = ah + xv;", "y[w] = ah;", 0),
    ("normcap_gate_on_input", "float ah = av * h[w];", "float ah = av * xv;", 1),
    ("reverse_ignored", "int64_t t = reverse ? T - 1 - s : s;", "int64_t t = s;", 0),
    ("output_in_trip_order", "float *ot = out + ((o * T + t) * J + j) * W;",
     "float *ot = out + ((o * T + s) * J + j) * W;", 0),
    ("initial_ignored", "h[w] = initial[(o * J + j) * W + w];", "h[w] = 0.0f;", 0),
    ("initial_lane_index", "h[w] = initial[(o * J + j) * W + w];", "h[w] = initial[(j * O + o) % (O * J) * W + w];", 0),
    ("second_sequence_time_shift", "const float *at = a + ((o * T + t) * J + j) * sw[1];",
     "const float *at = a + ((o * T + (t + 1) % T) * J + j) * sw[1];", 0),
    ("gate_ignores_broadcast", "float av = at[sw[1] == 1 ? 0 : w];", "float av = at[0];", 1),
    # backward pass
    ("bwd_tanh_derivative_sign", "float om = 1.0f - hh;", "float om = 1.0f + hh;", 0),
    ("bwd_tanh_dropped_decay_factor", "lam[w] = m * av;", "lam[w] = m;", 0),
    ("bwd_tanh_decay_grad_operand", "da[w] = m * p[w];", "da[w] = m * ht[w];", 0),
    ("bwd_maxplus_cost_sign", "da[w] = -lam[w];", "da[w] = lam[w];", 0),
    ("bwd_maxplus_tie_not_split", "float half = lam[w] * 0.5f;", "float half = lam[w];", 0),
    ("bwd_normcap_projection_sign", "float dlt = lam[w] - r;", "float dlt = lam[w] + r;", 0),
    ("bwd_normcap_missing_norm", "mu[w] = dlt / nrm;", "mu[w] = dlt;", 0),
    ("bwd_previous_state_is_own_output", "int64_t tp = reverse ? t + 1 : t - 1;", "int64_t tp = t;", 0),
    ("bwd_drops_carried_cotangent", "for (int64_t w = 0; w < W; w++) lam[w] = lam[w] + gt[w];",
     "for (int64_t w = 0; w < W; w++) lam[w] = gt[w];", 0),
    ("bwd_gate_sum_first_only", "for (int64_t w = 0; w < W; w++) acc = acc + da[w];", "acc = da[0];", 0),
]


def _mutate(src, old, new, occ):
    idx = -1
    for _ in range(occ + 1):
        idx = src.index(old, idx + 1)
    return src[:idx] + new + src[idx + len(old):]


def test_mutation_targets_exist():
    src = open(SRC).read()
    for mid, old, new, occ in MUTATIONS:
        assert src.count(old) > occ, mid


@pytest.mark.parametrize("mid,old,new,occ", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutant(mid, old, new, occ, tmp_path, oracle_mod):
    src = open(SRC).read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    cfile = tmp_path / "mutant.c"
    cfile.write_text(mutated)
    lib = oracle_mod.compile_source(str(cfile), str(tmp_path / "libmutant.so"))
    mutant = oracle_mod.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant.scan)
        except (AssertionError, ValueError):   # noqa: PERF203
            caught.append(pin.__name__)
    for pin in oracle_pins.BWD_PINS:
        try:
            pin(mutant.scan, mutant.scan_backward)
        except (AssertionError, ValueError):   # noqa: PERF203
            caught.append(pin.__name__)
    assert caught, "no pin caught the planted mistake %s" % mid
