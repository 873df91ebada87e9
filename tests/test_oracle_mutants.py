"""The oracle's pins catch plausible mistakes planted in the oracle.

Each case copies ``oracle/sc_oracle.c``, plants one mistake in the copy (a
dropped term, a wrong sign, a wrong index, normalisation or tie rule, a
swapped operand), compiles it with gcc into a temporary directory and runs
the pin file ``test_oracle_pins.py`` against it in a child process, with
``SC_ORACLE_LIB`` pointing the oracle loader at the copy.  Every mutant must
make at least one pin fail; an unmutated copy built the same way must pass
them all, which shows that the children really load the copies.  The LM
head's oracle, written in Python, gets its mutants in-process instead (a
mutated copy of the function swapped into the module for one test).  The
committed oracle is never modified, and nothing here runs the CUDA library.
"""

import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "sc_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# name -> (text of the oracle, its replacement); each text occurs once.
MUTANTS = {
    # bf16 encoding
    "bf16 rounding: ties away from zero": ("double r = nearbyint(scaled);", "double r = round(scaled);"),
    "bf16 rounding: truncation": ("double r = nearbyint(scaled);", "double r = trunc(scaled);"),
    "bf16 decoding: wrong shift": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    # group advantages
    "advantages: biased std": ("sqrt(ss / (group_size - 1))", "sqrt(ss / group_size)"),
    "advantages: all-equal rule dropped": ("if (all_equal) {", "if (0) {"),
    "advantages: mean-only mode still divides": ("out[i] = normalize_std ? d / (std + eps) : d;",
                                                 "out[i] = d / (std + eps);"),
    # the softmax
    "log-sum-exp without its maximum": ("    double lse = m + log(l);\n    for (int v = 0; v < V; ++v) logp[v]",
                                        "    double lse = log(l);\n    for (int v = 0; v < V; ++v) logp[v]"),
    "temperature left out of log p": ("logp[v] = sco_bf16_to_double(z[v]) * invT - lse;",
                                      "logp[v] = sco_bf16_to_double(z[v]) - lse;"),
    # the recorded head
    "duplicate ids: the last occurrence wins": ("if (in_h[id] >= 0) {", "if (0) {"),
    "Q_H from the trainer instead of the recorded q": ("Q_H += exp((double)lp[in_h[v]]);", "Q_H += exp(logp[v]);"),
    "tail ratio inverted": ("double rho = fmax(tail_mu, 1e-6) / fmax(tail_pi, 1e-6);",
                            "double rho = fmax(tail_pi, 1e-6) / fmax(tail_mu, 1e-6);"),
    "tail ratio without its clamps": ("double rho = fmax(tail_mu, 1e-6) / fmax(tail_pi, 1e-6);",
                                      "double rho = tail_mu / tail_pi;"),
    "s: wrong sign of rho P_H": ("double s = 1.0 - Q_H + rho * P_H;", "double s = 1.0 - Q_H - rho * P_H;"),
    "s: Q_H term dropped": ("double s = 1.0 - Q_H + rho * P_H;", "double s = 1.0 + rho * P_H;"),
    # the gradient and the loss
    "centering term dropped from the gradient": ("if (p->centering && in_h[v] >= 0) mu_hat +=",
                                                 "if (0 && in_h[v] >= 0) mu_hat +="),
    "centering term: wrong sign of rho p": ("mu_hat += exp((double)lp[in_h[v]]) - rho * pv;",
                                           "mu_hat += exp((double)lp[in_h[v]]) + rho * pv;"),
    "gradient without 1/T": ("double coef = p->grad_scale * invT * (-A_eff);",
                             "double coef = p->grad_scale * (-A_eff);"),
    "gradient: wrong sign of the advantage": ("double coef = p->grad_scale * invT * (-A_eff);",
                                              "double coef = p->grad_scale * invT * A_eff;"),
    "gradient: indicator on the wrong token": ("(v == a ? 1.0 : 0.0)", "(v == a + 1 ? 1.0 : 0.0)"),
    "loss: wrong sign of the centered sum": ("double loss = -A_eff * (logp[a] - centered);",
                                             "double loss = -A_eff * (logp[a] + centered);"),
    "entropy: wrong sign": ("if (pv > 0.0) ent -= pv * logp[v];", "if (pv > 0.0) ent += pv * logp[v];"),
    "k3: wrong sign of d": ("exp(d) - 1.0 - d : 0.0;", "exp(d) - 1.0 + d : 0.0;"),
    # importance weights and the clipped baseline
    "tis: no truncation": ("wt = w < p->tis_max ? w : p->tis_max;", "wt = w;"),
    "mis: weight kept outside the interval": ("            wt = 0.0;\n            flags |= SCO_FLAG_IS_REJECT;",
                                              "            wt = w;\n            flags |= SCO_FLAG_IS_REJECT;"),
    "clipped GRPO: upper and lower widths swapped in the gradient": (
        "double wc = w < 1.0 - p->clip_low ? 1.0 - p->clip_low : (w > 1.0 + p->clip_high ? 1.0 + p->clip_high : w);\n"
        "        if (wc == w",
        "double wc = w < 1.0 - p->clip_high ? 1.0 - p->clip_high : (w > 1.0 + p->clip_low ? 1.0 + p->clip_low : w);\n"
        "        if (wc == w"),
    "clipped GRPO: the clipped side keeps its gradient": ("            wt = 0.0;\n            flags |= SCO_FLAG_CLIPPED;",
                                                          "            wt = w;\n            flags |= SCO_FLAG_CLIPPED;"),
    "per-rollout mean: one token too many": ("adv[r] / (double)counts[r]", "adv[r] / (double)(counts[r] + 1)"),
    # batch rules
    "padding and bad responses flagged the other way round":
        ("o->flags = resp < 0 ? SCO_FLAG_MASKED : SCO_FLAG_BAD_RESPONSE;",
         "o->flags = resp < 0 ? SCO_FLAG_BAD_RESPONSE : SCO_FLAG_MASKED;"),
    # sampler-side top-K capture
    "top-K: equal values ordered by higher id": ("return (a->id > b->id) - (a->id < b->id);",
                                                "return (a->id < b->id) - (a->id > b->id);"),
    "top-K: nucleus not renormalised": ("lognuc = log(cum);", "lognuc = 0.0;"),
    "top-K: count ignores the nucleus": ("int cnt = (int)(n_keep < K ? n_keep : K);",
                                         "int cnt = (int)(V < K ? V : K);"),
    "top-K: temperature left out of the probabilities":
        ("lp_out[t * K + k] = k < cnt ? (float)((double)e[k].z * inv_t - lse - lognuc) : 0.0f;",
         "lp_out[t * K + k] = k < cnt ? (float)((double)e[k].z - lse - lognuc) : 0.0f;"),
}

CONTROL = "control: no mutation"


def _build_and_run(key, name, workdir):
    src = open(SRC).read()
    if name != CONTROL:
        old, new = MUTANTS[name]
        assert src.count(old) == 1, f"{name}: the text to mutate occurs {src.count(old)} times"
        src = src.replace(old, new)
    d = os.path.join(workdir, f"m{key}")
    os.makedirs(d, exist_ok=True)
    c, so = os.path.join(d, "sc_oracle.c"), os.path.join(d, "libsc_oracle.so")
    with open(c, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC", "-shared", "-o", so, c,
                    "-lm", "-lpthread"], check=True)
    env = dict(os.environ, SC_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=900)
    return r.returncode, (r.stdout + r.stderr)[-3000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    work = str(tmp_path_factory.mktemp("oracle_mutants"))
    names = [CONTROL] + list(MUTANTS)
    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        futs = {n: ex.submit(_build_and_run, i, n, work) for i, n in enumerate(names)}
        return {n: f.result() for n, f in futs.items()}


def test_unmutated_copy_passes_every_pin(outcomes):
    rc, out = outcomes[CONTROL]
    assert rc == 0, f"the unmutated copy failed the pins (exit {rc}):\n{out}"


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_reject_planted_mistake(outcomes, name):
    rc, out = outcomes[name]
    # exit 1: the pins ran and at least one failed (a crash would be < 0)
    assert rc == 1, f"mutant '{name}' was not caught by the pins (exit {rc}):\n{out}"


# The LM head's oracle is Python (oracle.lmhead_rows): its mutants are planted
# in a copy of that function's source, swapped into the oracle module for one
# test, and its two pins (finite differences, the identity head) run directly.
LMHEAD_MUTANTS = {
    "dH from the bf16-rounded gradient": ("return g @ W, gw.T @ H,",
                                          "return bf16_to_double(bf16_round_array(g)) @ W, gw.T @ H,"),
    "dW from the bf16-rounded gradient": ("return g @ W, gw.T @ H,",
                                          "return g @ W, bf16_to_double(bf16_round_array(gw)).T @ H,"),
    "grad_scale applied twice to dH": ("return g @ W, gw.T @ H,", "return params.grad_scale * (g @ W), gw.T @ H,"),
    "logits truncated to bf16": ("z_bits = bf16_round_array(H @ W.T)",
                                 "z_bits = ((H @ W.T).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)"),
    "dW transposed": ("return g @ W, gw.T @ H,", "return g @ W, (gw.T @ H).T,"),
}


@pytest.mark.parametrize("name", list(LMHEAD_MUTANTS))
def test_lmhead_pins_reject_planted_mistake(name, monkeypatch):
    import inspect

    import oracle
    import test_oracle_pins as pins

    old, new = LMHEAD_MUTANTS[name]
    src = inspect.getsource(oracle.lmhead_rows)
    assert src.count(old) == 1, name
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    monkeypatch.setattr(oracle, "lmhead_rows", ns["lmhead_rows"])
    caught = 0
    for pin in (lambda: pins.test_lmhead_gradients_match_central_differences(1.0, 41),
                lambda: pins.test_lmhead_gradients_match_central_differences(1 / 0.7, 42),
                pins.test_lmhead_with_identity_head_reduces_to_the_row_oracle,
                pins.test_lmhead_logits_are_the_rounded_fp64_products):
        try:
            pin()
        except Exception:  # an assertion, or a shape mismatch the mutant causes
            caught += 1
    assert caught >= 1, f"LM-head mutant '{name}' passed every pin"


def test_lmhead_unmutated_copy_passes_its_pins(monkeypatch):
    import inspect

    import oracle
    import test_oracle_pins as pins

    ns = dict(vars(oracle))
    exec(compile(inspect.getsource(oracle.lmhead_rows), "<copy>", "exec"), ns)
    monkeypatch.setattr(oracle, "lmhead_rows", ns["lmhead_rows"])
    pins.test_lmhead_gradients_match_central_differences(1.0, 41)
    pins.test_lmhead_with_identity_head_reduces_to_the_row_oracle()
    pins.test_lmhead_logits_are_the_rounded_fp64_products()
