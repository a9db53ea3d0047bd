"""The oracle's pins catch plausible mistakes: each mutant below is oracle.c with one planted
error (a dropped term, a wrong sign, a time index off by one, an operand swapped for another),
compiled on its own, and the pins of tests/test_oracle_pins.py and tests/test_delta_rule.py must
fail against every one of them.  The unmutated source, compiled the same way, must pass them.  Mistakes are planted in
the oracle on the CPU only; nothing here touches the CUDA library.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, text in oracle.c, replacement, which occurrence (0-based))
MUTANTS = [
    # diagonal scan
    ("scan fwd: stores the state before the update",
     "state = a[idx] * state + b[idx];\n            h[idx] = state;",
     "h[idx] = state;\n            state = a[idx] * state + b[idx];", 0),
    ("scan fwd: ignores h0", "double state = h0 ? h0[bi * D + d] : 0.0;", "double state = 0.0;", 0),
    ("scan bwd: adjoint decayed by a_t instead of a_{t+1}",
     "hbar = g[idx] + a_next * hbar;", "hbar = g[idx] + a[idx] * hbar;", 0),
    ("scan bwd: da from h_t instead of h_{t-1}", "da[idx] = hbar * hs[t - 1];", "da[idx] = hbar * hs[t];", 0),
    ("scan bwd: drops the gradient on h_T",
     "hbar = g[idx] + (dhT ? dhT[bi * D + d] : 0.0);", "hbar = g[idx];", 0),
    ("scan bwd: dh0 without a_1", "dh0[bi * D + d] = (T > 0) ? a_next * hbar : 0.0;",
     "dh0[bi * D + d] = (T > 0) ? hbar : 0.0;", 0),
    # selective scan
    ("selective fwd: input without delta", "double b_tn = delta[idx] * Bt[n] * x[idx];",
     "double b_tn = Bt[n] * x[idx];", 0),
    ("selective fwd: reads with B instead of C", "acc += Ct[n] * hs[n];", "acc += Bt[n] * hs[n];", 0),
    ("selective bwd: sign of the input term of ddelta",
     "gdelta += dadecay * a_tn * A[d * N + n] + hbar[n] * Bt[n] * x[idx];",
     "gdelta += dadecay * a_tn * A[d * N + n] - hbar[n] * Bt[n] * x[idx];", 0),
    ("selective bwd: dA without delta", "pa[n] += dadecay * a_tn * delta[idx];", "pa[n] += dadecay * a_tn;", 0),
    ("selective bwd: dC from h_{t-1}", "pC[n] += dy[idx] * hs[t * N + n];",
     "pC[n] += dy[idx] * hs[(t - 1) * N + n];", 0),
    ("selective bwd: dB without x", "pB[n] += hbar[n] * delta[idx] * x[idx];", "pB[n] += hbar[n] * delta[idx];", 0),
    ("selective bwd: recompute without delta in the input", "double b_tn = delta[idx] * Bt[n] * x[idx];",
     "double b_tn = Bt[n] * x[idx];", 1),
    # linear attention
    ("la fwd: decays the token's own write",
     "S[i * dv + j] = at * S[i * dv + j] + kt[i] * vt[j];", "S[i * dv + j] = at * (S[i * dv + j] + kt[i] * vt[j]);", 0),
    ("la fwd: reads with the key instead of the query",
     "for (i64 i = 0; i < dk; ++i) s += S[i * dv + j] * qt[i];",
     "for (i64 i = 0; i < dk; ++i) s += S[i * dv + j] * kt[i];", 0),
    ("la bwd: adjoint decayed by a_t instead of a_{t+1}",
     "Sbar[i * dv + j] = a_next * Sbar[i * dv + j] + qu[t * dk + i] * du[t * dv + j];",
     "Sbar[i * dv + j] = exp(lu[t]) * Sbar[i * dv + j] + qu[t * dk + i] * du[t * dv + j];", 0),
    ("la bwd: dlog a without the factor a_t", "dlog_a[u * T + t] = at * s;", "dlog_a[u * T + t] = s;", 0),
    ("la bwd: dS0 without a_1", "dS0[u * ss + i] = (T > 0 ? a_next : 1.0) * Sbar[i];", "dS0[u * ss + i] = Sbar[i];", 0),
    ("la bwd: dv contracted with the query",
     "for (i64 i = 0; i < dk; ++i) s += Sbar[i * dv + j] * ku[t * dk + i];",
     "for (i64 i = 0; i < dk; ++i) s += Sbar[i * dv + j] * qu[t * dk + i];", 0),
    ("la closed form: sign of the key term", "run += qd - kd;", "run += qd + kd;", 0),
    ("la closed form: drops the final-state term", "double run = tail;", "double run = 0.0;", 0),
    # state passing between slices
    ("state compose: decays the slice's own contribution",
     "acc = alpha[(j * BH + bh) * A + e / per] * acc + dS[(j * BH + bh) * n + e];",
     "acc = alpha[(j * BH + bh) * A + e / per] * (acc + dS[(j * BH + bh) * n + e]);", 0),
    ("state compose: ignores the edge state", "double acc = edge ? edge[bh * n + e] : 0.0;", "double acc = 0.0;", 0),
    ("decay total: sums decays instead of their logs", "alpha[bh * A + a] = exp(s);", "alpha[bh * A + a] = s;", 0),
    # gated linear attention
    ("gla fwd: one decay for every key dimension", "double ai = exp(lt[i]);", "double ai = exp(lt[0]);", 0),
    ("gla bwd: adjoint decayed by the first dimension's decay",
     "Sbar[i * dv + j] = anext[i] * Sbar[i * dv + j] + qu[t * dk + i] * du[t * dv + j];",
     "Sbar[i * dv + j] = anext[0] * Sbar[i * dv + j] + qu[t * dk + i] * du[t * dv + j];", 0),
    ("gla bwd: dlog a without the factor a_t[i]", "dlog_a[(u * T + t) * dk + i] = ai * s;",
     "dlog_a[(u * T + t) * dk + i] = s;", 0),
    ("gla bwd: dS0 without a_1", "dS0[u * ss + i * dv + j] = anext[i] * Sbar[i * dv + j];",
     "dS0[u * ss + i * dv + j] = Sbar[i * dv + j];", 0),
    ("gla closed form: drops the key term", "run += q[x] * dq[x] - k[x] * dkk[x];", "run += q[x] * dq[x];", 0),
    # delta rule
    ("delta: corrects with the new value instead of the stored one",
     "cur[i * dv + j] = at * (prev[i * dv + j] - bt * kt[i] * u[j]) + bt * kt[i] * vt[j];",
     "cur[i * dv + j] = at * (prev[i * dv + j] - bt * kt[i] * vt[j]) + bt * kt[i] * vt[j];", 0),
    ("delta: decays the token's own write",
     "cur[i * dv + j] = at * (prev[i * dv + j] - bt * kt[i] * u[j]) + bt * kt[i] * vt[j];",
     "cur[i * dv + j] = at * (prev[i * dv + j] - bt * kt[i] * u[j] + bt * kt[i] * vt[j]);", 0),
    ("delta bwd: dk without the stored-value term", "dkk[(un * T + t) * dk + m] = bt * s1 - at * bt * s2;",
     "dkk[(un * T + t) * dk + m] = bt * s1;", 0),
    ("delta bwd: sign of the correction in dbeta", "db += kS[j] * (vt[j] - at * u[j]);",
     "db += kS[j] * (vt[j] + at * u[j]);", 0),
    ("delta bwd: adjoint without the rank-one part",
     "tmp[i * dv + j] = at * (Sbar[i * dv + j] - bt * kt[i] * kS[j]);", "tmp[i * dv + j] = at * Sbar[i * dv + j];", 0),
    ("delta bwd: dv without beta", "dvv[(un * T + t) * dv + j] = bt * sk;", "dvv[(un * T + t) * dv + j] = sk;", 0),
    ("delta bwd: dlog a without the rank-one part", "dlog_a[un * T + t] = at * (s - bt * c);",
     "dlog_a[un * T + t] = at * s;", 0),
    ("delta bwd: dq read from the state before the step", "const double *cur = states + (t + 1) * ss;",
     "const double *cur = states + t * ss;", 0),
]


def _plant(src, old, new, occurrence):
    at = -1
    for _ in range(occurrence + 1):
        at = src.find(old, at + 1)
        assert at >= 0, f"mutation site not found in oracle.c (occurrence {occurrence}): {old!r}"
    return src[:at] + new + src[at + len(old):]


def _compile(src_text, path):
    c = path + ".c"
    with open(c, "w") as f:
        f.write(src_text)
    r = subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-std=c11", "-fopenmp", "-o", path + ".so", c, "-lm"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return path + ".so"


def _run_pins(lib):
    env = dict(os.environ, OMP_NUM_THREADS="1")
    pins = [os.path.join(ROOT, "tests", f) for f in ("test_oracle_pins.py", "test_delta_rule.py")]
    r = subprocess.run([sys.executable, "-m", "pytest"] + pins + ["-q", "-p", "no:cacheprovider", "--oracle-lib", lib],
                       capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)
    failed = sorted({line.split("::")[1].split(" ")[0].split("[")[0] for line in r.stdout.splitlines()
                     if line.startswith("FAILED ")})
    return r.returncode, failed, r.stdout[-2000:]


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    d = tmp_path_factory.mktemp("mutants")
    src = open(SRC).read()
    jobs = [("unmutated", src)] + [(name, _plant(src, old, new, occ)) for name, old, new, occ in MUTANTS]
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        libs = list(ex.map(lambda ij: _compile(ij[1][1], str(d / f"m{ij[0]}")), enumerate(jobs)))
        runs = list(ex.map(_run_pins, libs))
    return {name: run for (name, _), run in zip(jobs, runs)}


def test_unmutated_oracle_passes_its_pins(results):
    rc, failed, out = results["unmutated"]
    assert rc == 0 and not failed, out


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_every_planted_mistake_fails_a_pin(results, name):
    rc, failed, out = results[name]
    assert rc == 1 and failed, f"mutant survived the pins: {name}\n{out}"
