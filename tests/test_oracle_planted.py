"""Planted mistakes: each pin of the oracle must reject a plausible error in the code it pins.

For every entry below, a copy of ``oracle/dspark_oracle.cpp`` with one mistake planted (an exact
text substitution that must apply exactly once) is compiled into a temporary directory, the
oracle's front end is pointed at it (``oracle.using_library``), and the named pin, called as it
runs in the suite, must fail.  Together with the pins passing on the real oracle, this shows
the pins are sensitive to the mistakes they are meant to catch: a dropped term, a wrong sign or
index, a transposed operand, a swapped gate, an off-by-one label.  Everything here runs on the
CPU.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

import pytest

from oracle import oracle
from tests import test_oracle_labels as labels
from tests import test_oracle_loss as loss
from tests import test_oracle_sampler as sampler
from tests import test_oracle_schedule_rnn as sched
from tests import test_oracle_sts as sts
from tests import test_oracle_verify as verify

SRC = os.path.join(os.path.dirname(oracle.__file__), "dspark_oracle.cpp")

# name: (text in dspark_oracle.cpp, planted replacement, the pin that must fail)
PLANTED = {
    "conditioning on the anchor at every step": (
        "prev = forced ? forced[bk] : t1;", "prev = forced ? forced[bk] : x0[b];",
        lambda: sampler.test_block_distribution_brute_force(oracle, 1.0)),
    "W2 read with its indices transposed": (
        "bias += a[j] * load(W2, wdt, (size_t)v * r + j);",
        "bias += a[j] * load(W2, wdt, (size_t)j * V + v);",
        lambda: sampler.test_bias_equals_dense_transition_table(oracle)),
    "Gumbel noise subtracted": (
        "gsc[v] = y[v] + gumbel(seed, b, k, v);", "gsc[v] = y[v] - gumbel(seed, b, k, v);",
        lambda: sampler.test_block_distribution_brute_force(oracle, 1.0)),
    "temperature dropped": (
        "y[v] = z / T;", "y[v] = z;",
        lambda: sampler.test_cold_temperature_is_argmax(oracle)),
    "log-sum-exp without its shift": (
        "return m + std::log(s);", "return std::log(s);",
        lambda: sampler.test_lse_against_long_double(oracle)),
    "Philox key schedule off by one": (
        "k0 += 0x9E3779B9u;  // golden-ratio Weyl increment", "k0 += 0x9E3779B8u;",
        lambda: sampler.test_philox_matches_independent_implementation(oracle)),
    "Eq 7 weight halves swapped": (
        "for (int j = 0; j < r; ++j) logit += load(w, wdt, (size_t)d + j) * e[j];",
        "for (int j = 0; j < r; ++j) logit += load(w, wdt, (size_t)j) * e[j];",
        lambda: labels.test_confidence_halves_and_index(oracle)),
    "S_k not a running product": (
        "        surv *= c[out];\n", "        surv = c[out];\n",
        lambda: labels.test_confidence_zero_weight_half(oracle)),
    "Eq 8 without the one half": (
        "*cstar = std::min(1.0, std::max(0.0, 1.0 - 0.5 * acc));",
        "*cstar = std::min(1.0, std::max(0.0, 1.0 - acc));",
        lambda: labels.test_tv_one_hot_vs_uniform(oracle, 1000)),
    "verify: the residual taken as q": (
        "w[v] = std::max(0.0, std::exp(tau[v] - Lt) - std::exp(y[v] - Ld));",
        "w[v] = std::exp(tau[v] - Lt);",
        verify.test_output_token_is_distributed_as_target),
    "verify: the acceptance ratio inverted": (
        "const double log_ratio = (tau[x] - Lt) - (y[x] - Ld);",
        "const double log_ratio = (y[x] - Ld) - (tau[x] - Lt);",
        verify.test_output_token_is_distributed_as_target),
    "verify: the bonus drawn from the last draft position's target row": (
        "const size_t tj = ((size_t)b * (gamma + 1) + gamma) * V;",
        "const size_t tj = ((size_t)b * (gamma + 1) + gamma - 1) * V;",
        verify.test_joint_law_brute_force_gamma2),
    "loss: position weights shifted by one": (
        "const double wk = std::exp(-(double)j / (double)gamma);",
        "const double wk = std::exp(-(double)(j + 1) / (double)gamma);",
        lambda: loss.test_position_weights_match_the_printed_values(4, 1e-12)),
    "loss: TV gradient without its mean term": (
        "a_tv * p[v] * (s_v - sp)", "a_tv * p[v] * s_v",
        lambda: loss.test_gradients_match_finite_differences(1.3, (0.0, 1.0, 0.0))),
    "loss: the confidence label without the one half": (
        "const double cstar = std::min(1.0, std::max(0.0, 1.0 - 0.5 * l1));",
        "const double cstar = std::min(1.0, std::max(0.0, 1.0 - l1));",
        loss.test_confidence_label_one_hot_against_uniform),
    "STS: the prefix without the chosen temperatures": (
        "prefix[n] *= sigmoid((double)conf[(size_t)n * gamma + k - 1] / tau[k - 1]);",
        "prefix[n] *= sigmoid((double)conf[(size_t)n * gamma + k - 1]);",
        sts.test_recovers_known_temperatures),
    "STS: survival label off by one": (
        "const double y = acc[n] >= k ? 1.0 : 0.0;", "const double y = acc[n] > k ? 1.0 : 0.0;",
        sts.test_ece_closed_forms),
    "STS: absolute value per sample instead of per bin": (
        "sums[m] += S - y;", "sums[m] += std::fabs(S - y);",
        sts.test_ece_closed_forms),
    "scheduler: the bonus token left out of the expected tokens": (
        "const double tau = (double)B + (double)fixed_sum / 4294967296.0;",
        "const double tau = (double)fixed_sum / 4294967296.0;",
        lambda: sched.test_schedule_brute_force(oracle, 3, 2)),
    "RNN: gate and candidate rows swapped": (
        "const double gate = sigmoid(u[j]);\n          const double cand = std::tanh(u[r + j]);",
        "const double gate = sigmoid(u[r + j]);\n          const double cand = std::tanh(u[j]);",
        lambda: sched.test_rnn_closed_gate_uses_previous_state(oracle)),
}


def _build_mutant(tmp, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"{name}: the text to replace must occur exactly once"
    d = os.path.join(tmp, f"m{abs(hash(name)) % 10**8}")
    os.makedirs(d, exist_ok=True)
    src = os.path.join(d, "dspark_oracle.cpp")
    open(src, "w").write(text.replace(old, new))
    lib = os.path.join(d, "liboracle.so")
    subprocess.run(["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared",
                    "-ffp-contract=off", "-o", lib, src], check=True)
    return lib


@pytest.fixture(scope="module")
def mutants(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("no host C++ compiler")
    tmp = str(tmp_path_factory.mktemp("planted"))
    with cf.ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        futs = {n: ex.submit(_build_mutant, tmp, n, o, w) for n, (o, w, _) in PLANTED.items()}
        return {n: f.result() for n, f in futs.items()}


@pytest.mark.parametrize("name", sorted(PLANTED))
def test_pin_rejects_planted_mistake(mutants, name):
    pin = PLANTED[name][2]
    with oracle.using_library(mutants[name]):
        with pytest.raises(AssertionError):
            pin()
