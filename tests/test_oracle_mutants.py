"""The oracle's pins catch planted mistakes.

Each mutant is a copy of the oracle's C source with one plausible mistake
planted in it — a dropped term, a flipped tie rule, a wrong beam constant, an
off-by-one window, a non-strict comparison — at a rule the page "GPU WFST
Beam-Search Decoder" fixes (§3 Decoding Semantics, §5.3 upper-bound
paragraph, §5.5 epsilon closure and lattice persistence, §7 backtrack and
lattice prune).  The mutant is compiled on the CPU into a temporary library
and the pin suite (tests/test_oracle_pins.py) runs against it in a child
process; every mutant must make a pin fail.  A mutant that survives names a
rule the pins do not hold down.

Nothing here touches the CUDA decoder, and the mutants exist only in a
temporary directory.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "wfst_oracle.c")
HDR = os.path.join(ROOT, "oracle", "wfst_oracle.h")
PINS = [os.path.join(ROOT, "tests", "test_oracle_pins.py"),
        os.path.join(ROOT, "tests", "test_oracle_interval_prune.py")]

# name -> [(text in the oracle, planted replacement), ...]; each text occurs once
MUTANTS = {
    # §1 / §5.3: end = (score + weight) + log_prob
    "emit: arc weight dropped": [("const float partial = sc + g->w[a];", "const float partial = sc;")],
    "emit: log-prob dropped": [("const float end = partial + lpv;", "const float end = partial;")],
    "emit: other association": [("const float end = partial + lpv;",
                                 "const float end = sc + (g->w[a] + lpv);")],
    "emit: max is the first candidate": [("if (d->ncand == 1 || end > max_end) max_end = end;",
                                          "if (d->ncand == 1) max_end = end;")],
    # §3: admission end > exact_max - b, strict
    "admit: non-strict": [("if (!(c.end > cutoff)) continue;", "if (!(c.end >= cutoff)) continue;")],
    "admit: no pruning": [("if (!(c.end > cutoff)) continue;", "if (0) continue;")],
    # recombination tie: lowest arc id
    "recombine: highest arc id on ties": [("(c.end == tk->score && c.arc < tk->arc)",
                                           "(c.end == tk->score && c.arc > tk->arc)")],
    "recombine: first candidate kept": [("if (c.end > tk->score || (c.end == tk->score && c.arc < tk->arc)) {",
                                         "if (0) {")],
    # §3: dynamic beam
    "beam: relax 0.9/0.1": [("float x = 0.8f * b;", "float x = 0.9f * b;"),
                            ("float y = 0.2f * sb;", "float y = 0.1f * sb;")],
    "beam: widen 1.5": [("b = m * 1.25f;", "b = m * 1.5f;")],
    "beam: tighten 0.75": [("b = m * 0.8f;", "b = m * 0.75f;")],
    "beam: widen from the current beam only": [("float m = b > sb ? b : sb;", "float m = b;")],
    "beam: tighten from the current beam only": [("float m = b < sb ? b : sb;", "float m = b;")],
    "beam: relax interval open at min_active": [("(min_a <= n && n <= d->p.max_active)",
                                                 "(min_a < n && n <= d->p.max_active)")],
    "beam: relax interval open at max_active": [("(min_a <= n && n <= d->p.max_active)",
                                                 "(min_a <= n && n < d->p.max_active)")],
    "beam: empty frontier tightens": [("if (n == 0 || (min_a", "if ((min_a")],
    "beam: last-frames window 4": [("d->t >= d->t_eff - 5", "d->t >= d->t_eff - 4")],
    "beam: last-frames window 6": [("d->t >= d->t_eff - 5", "d->t >= d->t_eff - 6")],
    "beam: last-frames max_active / 4": [("int32_t half = d->p.max_active / 2;",
                                          "int32_t half = d->p.max_active / 4;")],
    "beam: last-frames rule off": [("if (d->t_eff >= 0 && d->t >= d->t_eff - 5) {", "if (0) {")],
    # §5.5: epsilon closure
    "eps: arc weight dropped": [("float e = su + g->w[a];", "float e = su;")],
    "eps: no cutoff": [("if (!(e > cutoff)) continue;", "if (0) continue;")],
    "eps: non-strict cutoff": [("if (!(e > cutoff)) continue;", "if (!(e >= cutoff)) continue;")],
    "eps: highest arc id on ties": [("(e == k->score && a < k->arc)", "(e == k->score && a > k->arc)")],
    "eps: start frontier without closure": [("if (g->has_eps) {\n    float cutoff0",
                                             "if (0) {\n    float cutoff0")],
    "eps: start cutoff without the beam": [("float cutoff0 = 0.0f - p->search_beam;",
                                            "float cutoff0 = 0.0f;")],
    # §3: final step
    "final: final weight dropped": [("const float fe = d->tok[i].score + f;",
                                     "const float fe = d->tok[i].score;")],
    "final: highest state on ties": [("(fe == best_fe && s < d->tok[best].state)",
                                      "(fe == best_fe && s > d->tok[best].state)")],
    "final: allow_partial ignored": [("} else if (d->p.allow_partial && ", "} else if (0 && ")],
    "final: best token ties by highest arc": [("(k->score == d->tok[best].score && k->arc < d->tok[best].arc))",
                                               "(k->score == d->tok[best].score && k->arc > d->tok[best].arc))")],
    # §7: words are the non-zero output labels, in forward order
    "words: epsilon output labels kept": [("if (d->g->ol[d->tok[k].arc] != 0) nw++;", "nw++;"),
                                          ("if (o != 0) {", "if (1) {")],
    "words: reverse order": [("      --pos;\n      if (pos < cap) words[pos] = o;",
                              "      if (nw - 1 - (--pos) < cap) words[nw - 1 - pos] = o;")],
    # §3 / §7: lattice backward prune
    "lattice: non-strict keep made strict": [("d->keep[r] = (uint8_t)(tot >= thr);",
                                              "d->keep[r] = (uint8_t)(tot > thr);")],
    "lattice: backward uses the forward value": [("const float v = r->arcscore + bd;",
                                                  "const float v = r->end + bd;")],
    "lattice: frames in forward order": [("return x->frame > y->frame ? -1 : 1; /* later frames first */",
                                          "return x->frame < y->frame ? -1 : 1;")],
    "lattice: record score without the log-prob": [("c->arcscore = g->w[a] + lpv;", "c->arcscore = g->w[a];")],
    "lattice: output_beam ignored": [("const float thr = d->best_score - d->p.output_beam;",
                                      "const float thr = -INFINITY;")],
    "lattice: epsilon records before emitting ones": [("return x->cls < y->cls ? -1 : 1;         /* non-epsilon first */",
                                                       "return x->cls > y->cls ? -1 : 1;")],
    "lattice: epsilon records in topological order": [("return x->rank > y->rank ? -1 : 1;     /* reverse topological */",
                                                       "return x->rank < y->rank ? -1 : 1;")],
    "lattice: final record without its weight": [("(int32_t)(g->A + s), -1, -1, OR_REC_FINAL, fe, f)",
                                                  "(int32_t)(g->A + s), -1, -1, OR_REC_FINAL, fe, 0.0f)")],
    "lattice: epsilon record score is the end": [("OR_REC_EPS, e, g->w[a])", "OR_REC_EPS, e, e)")],
    # §5.5: the closure visits states in epsilon-topological order
    "eps: states visited by id": [("h->key = g->eps_rank;", "h->key = NULL;")],
    # §7: arcs of the best path in forward order
    "path: arcs in reverse order": [("    --pos;\n    if (pos < cap) arcs[pos] = d->tok[k].arc;",
                                     "    --pos;\n    if (len - 1 - pos < cap) arcs[len - 1 - pos] = d->tok[k].arc;")],
    # §3: the online (streaming) beam has no last-frames clause
    "stream: last-frames rule fires online": [("if (d->t_eff >= 0 && d->t >= d->t_eff - 5) {",
                                               "if (d->t >= d->t_eff - 5) {")],
    # work counters (closed forms)
    "counters: admitted counts every candidate": [("d->st[OR_ST_SUM_A] += admitted;",
                                                   "d->st[OR_ST_SUM_A] += d->ncand;")],
    "counters: frontier after the step": [("d->st[OR_ST_SUM_N] += n;", "d->st[OR_ST_SUM_N] += m;")],
    # §7: interval lattice prune (the conservative reading)
    "interval: frontier tokens start at 0, not -score": [("beta[i - tok0] = -d->tok[i].score;",
                                                           "beta[i - tok0] = 0.0f;")],
    "interval: window of N frames": [("const int32_t r0 = t - 2 * N < -1 ? -1 : t - 2 * N;",
                                      "const int32_t r0 = t - N < -1 ? -1 : t - N;")],
    "interval: no safety margin": [("const float room = d->p.output_beam + 1.0f;",
                                    "const float room = d->p.output_beam + 0.0f;")],
}

_CHILD = r"""
import sys
sys.path.insert(0, {root!r})
import oracle
oracle._LIB_PATH = {lib!r}
oracle.build = lambda force=False: {lib!r}
import pytest
sys.exit(pytest.main([*{pins!r}, "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                      "-k", "not workloads_0_and_3"]))
"""


def _plant(src, subs):
    for old, new in subs:
        assert src.count(old) == 1, f"mutation site not unique: {old!r}"
        src = src.replace(old, new)
    return src


def _run(name, subs, tmp):
    d = os.path.join(tmp, str(abs(hash(name))))
    os.makedirs(d)
    with open(SRC) as f:
        src = _plant(f.read(), subs)
    c = os.path.join(d, "wfst_oracle.c")
    with open(c, "w") as f:
        f.write(src)
    with open(HDR) as f, open(os.path.join(d, "wfst_oracle.h"), "w") as g:
        g.write(f.read())
    lib = os.path.join(d, "liboracle.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                    "-o", lib, c, "-lm"], check=True, capture_output=True)
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT, lib=lib, pins=PINS)], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-2000:]


def test_mutation_sites_exist():
    with open(SRC) as f:
        src = f.read()
    for name, subs in MUTANTS.items():
        _plant(src, subs)


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
            results = list(ex.map(lambda kv: _run(kv[0], kv[1], tmp), MUTANTS.items()))
    survivors = [name for name, rc, _ in results if rc == 0]
    broken = [(name, rc, out) for name, rc, out in results if rc not in (0, 1) and rc >= 0]
    assert not broken, f"pin suite did not run on a mutant: {broken[:1]}"
    assert not survivors, f"planted mistakes no pin catches: {survivors}"
