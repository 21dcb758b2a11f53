"""Plant plausible mistakes in a copy of the oracle and check the pins catch
each one.  The mutants are built from a temporary copy of oracle.c on the
CPU; the committed oracle is never modified."""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
import pins
import pins_gumbel
import pins_penalty
import pins_spec

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")

# (name, original text, replacement)
MUTATIONS = [
    ("top-p uses > instead of >=", "if (cum >= top_p)", "if (cum > top_p)"),
    ("ties keep the latest ids", "return (p->id < q->id) ? -1 : (p->id > q->id);",
     "return (p->id > q->id) ? -1 : (p->id < q->id);"),
    ("top-p before top-k (mass over all of L)", "for (int r = 0; r < K; ++r) mass_k +=",
     "for (int r = 0; r < nl; ++r) mass_k +="),
    ("temperature dropped", "w[i] = legal[i] ? exp(z[i] - m) : 0.0;",
     "w[i] = legal[i] ? exp(x[i] - m) : 0.0;"),
    ("draw in rank order instead of id order", "qsort(sp, (size_t)nstar, sizeof(int), id_cmp);",
     ";"),
    ("greedy tie keeps the last id", "if (legal[i] && (best < 0 || xs[i] > xs[best])) best = i;",
     "if (legal[i] && (best < 0 || xs[i] >= xs[best])) best = i;"),
    ("final renormalisation dropped", "if (prob) prob[id] = ((w[id] / total) / mass_k) / mass_p;",
     "if (prob) prob[id] = ((w[id] / total) / mass_k);"),
    ("mask bit order reversed", "return (int)((mask_row[i >> 5] >> (i & 31)) & 1u);",
     "return (int)((mask_row[i >> 5] >> (31 - (i & 31))) & 1u);"),
    ("fp16 exponent bias off by one", "v = ldexp((double)(1024 + mant), expo - 25);",
     "v = ldexp((double)(1024 + mant), expo - 24);"),
    ("Philox multipliers swapped", "uint64_t p0 = (uint64_t)ORC_PHILOX_M0 * (uint64_t)c[0];",
     "uint64_t p0 = (uint64_t)ORC_PHILOX_M1 * (uint64_t)c[0];"),
    ("Philox key schedule constant wrong", "k[1] += ORC_PHILOX_W1;", "k[1] += ORC_PHILOX_W0;"),
    ("u uses 23 bits", "return (double)(out[0] >> 8) * (1.0 / 16777216.0);",
     "return (double)(out[0] >> 9) * (1.0 / 16777216.0);"),
    ("-inf counted as legal", "legal[i] = (unsigned char)(mask_allows(mask_row, i) && !(isinf(xs[i]) && xs[i] < 0));",
     "legal[i] = (unsigned char)(mask_allows(mask_row, i));"),
    ("K clamped to top_k - 1", "int K = top_k < nl ? top_k : nl;",
     "int K = top_k < nl ? (top_k > 1 ? top_k - 1 : 1) : nl;"),
    # speculative verification (lecture notes, section 5.2)
    ("verify: accept when u*q > p", "if (u_acc[i] * b < a) continue;",
     "if (u_acc[i] * b > a) continue;"),
    ("verify: accept when u*q <= p", "if (u_acc[i] * b < a) continue;",
     "if (u_acc[i] * b <= a) continue;"),
    ("verify: residual without max(0, .)", "return r > 0.0 ? r : 0.0;", "return fabs(r);"),
    ("verify: residual q - p", "const double r = qr ? (double)pr[x] - (double)qr[x] : (double)pr[x];",
     "const double r = qr ? (double)qr[x] - (double)pr[x] : (double)pr[x];"),
    ("verify: no stop at the first rejection", "    j = i;\n    break;", "    j = i;"),
    ("verify: bonus drawn from position 0", "*pr = p + (size_t)j * ld;",
     "*pr = p + (size_t)(j < G ? j : 0) * ld;"),
    ("verify: draw uses position 0's uniform", "const double t = u_res[j] * St;",
     "const double t = u_res[0] * St;"),
    ("verify: draw takes cum >= u*S", "if (tok < 0 && c > t) tok = x;",
     "if (tok < 0 && c >= t) tok = x;"),
    ("verify: residual draw reuses word 0", "ur[i] = (double)(out[1] >> 8) * (1.0 / 16777216.0);",
     "ur[i] = (double)(out[0] >> 8) * (1.0 / 16777216.0);"),
    ("verify: token range check off by one", "if (d[i] < 0 || d[i] >= V) return -1;",
     "if (d[i] < 0 || d[i] > V) return -1;"),
    ("verify: drawn row not checked", "if (!prob_ok((*pr)[x]) || (*qr && !prob_ok((*qr)[x]))) return 0;",
     ";"),
    ("verify fx: weights in units of 2^-20", "S += (uint64_t)floor(ldexp((double)r, 42));",
     "S += (uint64_t)floor(ldexp((double)r, 20));"),
    # repetition penalty (CTRL rule) and the float encoders
    ("penalty: every logit divided", "float y = (x > 0.0f) ? x / th : x * th;",
     "float y = x / th;"),
    ("penalty: signs swapped", "float y = (x > 0.0f) ? x / th : x * th;",
     "float y = (x > 0.0f) ? x * th : x / th;"),
    ("penalty: once per occurrence", "if (t < 0 || t >= V || seen[t]) continue;",
     "if (t < 0 || t >= V) continue;"),
    ("penalty: invalid penalty accepted", "if (!(th > 0.0f) || isinf(th)) {", "if (isinf(th)) {"),
    ("penalty: bf16 truncates", "uint32_t r = b + 0x7fffu + ((b >> 16) & 1u);",
     "uint32_t r = b;"),
    ("penalty: f16 ties away from zero", "double q = rint(ldexp(a, 10 - e));",
     "double q = floor(ldexp(a, 10 - e) + 0.5);"),
    # Gumbel-max sampler
    ("gumbel: noise sign flipped", "v = (double)(x / t) - log(-log(u));",
     "v = (double)(x / t) + log(-log(u));"),
    ("gumbel: temperature ignored", "v = (double)(x / t) - log(-log(u));",
     "v = (double)x - log(-log(u));"),
    ("gumbel: kept mask ignored", "if (!mask_allows(mrow, i)) continue;", ";"),
    ("gumbel: greedy keeps the last maximum", "if (v > bv) {", "if (v >= bv) {"),
    ("gumbel: one word per block", "return ((double)(out[i & 3] >> 8) + 0.5) * (1.0 / 16777216.0);",
     "return ((double)(out[0] >> 8) + 0.5) * (1.0 / 16777216.0);"),
]


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="oracle_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(workdir, name, old, new):
    src = open(os.path.join(SRC, "oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    tag = str(abs(hash(name)))
    d = os.path.join(workdir, tag)
    os.makedirs(d, exist_ok=True)
    shutil.copy(os.path.join(SRC, "oracle.h"), d)
    with open(os.path.join(d, "oracle.c"), "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(d, "libmut.so")
    res = subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                          os.path.join(d, "oracle.c"), "-o", so, "-lm"],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    L = oracle.load(so)
    caught = []
    checks = pins.ALL_CHECKS + pins_spec.SPEC_CHECKS
    if name.startswith("verify"):
        checks = pins_spec.SPEC_CHECKS + pins.ALL_CHECKS
    if name.startswith("penalty"):
        checks = pins_penalty.PENALTY_CHECKS
    if name.startswith("gumbel"):
        checks = pins_gumbel.GUMBEL_CHECKS
    for chk in checks:
        try:
            out = chk(L=L)
        except AssertionError:
            caught.append(chk.__name__)
            break
        if out is False:   # check skipped (e.g. no libcurand)
            continue
    assert caught, f"no pin caught the planted mistake: {name}"
