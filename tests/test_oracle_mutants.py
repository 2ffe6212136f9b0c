"""The oracle's pins catch plausible mistakes: each case below plants one mistake in a
scratch copy of ``oracle/`` (a dropped term, a wrong sign, a transposed operand, a
swapped or shifted index, a wrapper passing the wrong argument), rebuilds it there and runs the CPU pin tests
(``tests/test_oracle_*.py``) against the copy; every case must make at least one pin
fail.  Nothing here touches the oracle in the tree or any GPU code.

Left out as equivalent: writing the eviction budget test as ``L < S + W`` instead of
``L <= S + W`` (at L = S + W both keep every token in order), the absorbed-value mean
scaled by 1 instead of the weight sum (the weights sum to one), and a wrapper dropping the
position offset it passes for both the query and the keys (rotary scores depend only on
position differences, so a shift common to both changes nothing).
"""
import os
import py_compile
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C = "oracle/lla_oracle.c"

# (file, text in the oracle, planted mistake, what the mistake is)
MUTANTS = [
    (C, "y[i0] = x[i0] * c - x[i1] * s;\n        y[i1] = x[i0] * s + x[i1] * c;\n    }\n}\n\n/* §3",
     "y[i0] = x[i0] * c + x[i1] * s;\n        y[i1] = -x[i0] * s + x[i1] * c;\n    }\n}\n\n/* §3",
     "RoPE rotates the wrong way"),
    (C, "-2.0 * (double)f / (double)dm->d", "-1.0 * (double)f / (double)dm->d", "RoPE frequency exponent"),
    (C, "{ *i0 = f; *i1 = f + dm->d / 2; }", "{ *i0 = 2 * f; *i1 = 2 * f + 1; }", "half-split pairs taken as interleaved"),
    (C, "{ *i0 = 2 * f; *i1 = 2 * f + 1; }", "{ *i0 = f; *i1 = f + dm->d / 2; }", "interleaved pairs taken as half-split"),
    (C, "acc += (xv[u] - m[u]) * W[u * r + k];", "acc += (xv[u] + m[u]) * W[u * r + k];", "encode adds the mean"),
    (C, "acc += (xv[u] - m[u]) * W[u * r + k];", "acc += (xv[u] - m[u]) * W[k * Td + u];", "encode W_down transposed"),
    (C, "const double* m = mu + (long)h * Td;", "const double* m = mu;", "encode mean of head 0 for every head"),
    (C, "const double* W = w_down + (long)h * Td * r;", "const double* W = w_down;", "encode W_down of head 0 for every head"),
    (C, "cache + (((long)seq_idx[n] * H + h) * L_max + pos[n]) * r;",
     "cache + (((long)h * B + seq_idx[n]) * L_max + pos[n]) * r;", "cache index with sequence and head swapped"),
    (C, "acc += (xv[u] - mu[u]) * w_down[u * r + k];", "acc += xv[u] * w_down[u * r + k];", "LLA-2D encode drops the mean"),
    (C, "xhat[e] = acc + mu_t[e];", "xhat[e] = acc;", "reconstruction drops the mean"),
    (C, "acc += c[k] * W[(long)e * r + k];", "acc += c[k] * W[(long)k * d + e];", "reconstruction W_up transposed"),
    (C, "Wk = w_up_k + (((long)t * H + h) * d) * rk;\n            Wv",
     "Wk = w_up_k + (((long)h * dm->T + t) * d) * rk;\n            Wv", "W_up,k indexed [head][loop]"),
    (C, "Wv = w_up_v + (((long)t * H + h) * d) * rv;\n            muk_t",
     "Wv = w_up_v + (((long)h * dm->T + t) * d) * rv;\n            muk_t", "W_up,v indexed [head][loop]"),
    (C, "muk_t = mu_k + (long)h * dm->T * d + (long)t * d;\n            muv_t = mu_v + (long)h * dm->T * d + (long)t * d;\n        } else",
     "muk_t = mu_k + (long)h * dm->T * d;\n            muv_t = mu_v + (long)h * dm->T * d + (long)t * d;\n        } else",
     "K mean of loop 0 at every loop"),
    (C, "muv_t = mu_v + (long)h * dm->T * d + (long)t * d;\n        } else",
     "muv_t = mu_v + (long)t * dm->H * d + (long)h * d;\n        } else", "V mean indexed [loop][head]"),
    (C, "Wk = w_up_k + ((long)t * H * d + (long)h * d) * rk;", "Wk = w_up_k + ((long)h * d) * rk;",
     "LLA-2D W_up,k of loop 0 at every loop"),
    (C, "muv_t = mu_v + ((long)t * H + h) * d;", "muv_t = mu_v + ((long)h) * d;", "LLA-2D V mean of loop 0"),
    (C, "(double)(q_pos[b] + pos_offset), qr);\n        const double scale = 1.0 / sqrt((double)d);\n        for (long j = 0; j < L; ++j) {\n            const double* ck",
     "(double)(q_pos[b]), qr);\n        const double scale = 1.0 / sqrt((double)d);\n        for (long j = 0; j < L; ++j) {\n            const double* ck",
     "query position ignores the offset"),
    (C, "rope_rotate(dm, kh, (double)(j + pos_offset), kr);", "rope_rotate(dm, kh, (double)(j + 1 + pos_offset), kr);",
     "key positions off by one"),
    (C, "rope_rotate(dm, kh, (double)(j + pos_offset), kr);", "for (int e = 0; e < d; ++e) kr[e] = kh[e];",
     "keys not rotated"),
    (C, "const double scale = 1.0 / sqrt((double)d);\n        for (long j = 0; j < L; ++j) {\n            const double* ck",
     "const double scale = 1.0 / (double)d;\n        for (long j = 0; j < L; ++j) {\n            const double* ck",
     "score scale 1/d"),
    (C, ": cache_k + ((long)b * L_max + j) * rk;", ": cache_k + ((long)b * L_max + L - 1 - j) * rk;",
     "LLA-2D keys read in reverse"),
    (C, "{ p[j] = exp(s[j] - m); z += p[j]; }", "{ p[j] = exp(s[j] - m); z += p[j]; }\n    z *= 1.0 + 1e-9;",
     "softmax normaliser off by 1e-9"),
    (C, "lse[bh] = m + log(z);\n        free(qr); free(kh); free(kr); free(vh); free(s); free(p); free(av);",
     "lse[bh] = log(z);\n        free(qr); free(kh); free(kr); free(vh); free(s); free(p); free(av);",
     "log-sum-exp drops the max"),
    (C, "o[e] += p[j] * vh[e];\n            }\n        } else {", "o[e] += p[L - 1 - j] * vh[e];\n            }\n        } else {",
     "value weights in reverse"),
    (C, "o[e] = acc + psum * muv_t[e];", "o[e] = acc;", "absorbed values drop the mean"),
    (C, "av[k] += p[j] * cv[k];", "av[k] += cv[k] / (double)L;", "absorbed values uniform weights"),
    (C, "(double)(win_pos[b] + w), kr);", "(double)(win_pos[b]), kr);", "window keys all at the first position"),
    (C, "rope_rotate(dm, kh, (double)j, kr);\n            } else {", "rope_rotate(dm, kh, (double)(j + 1), kr);\n            } else {",
     "hybrid latent positions off by one"),
    (C, "v = v_win + (bh * W + (j - nl)) * d;", "v = v_win + (bh * W + (nw - 1 - (j - nl))) * d;",
     "window values in reverse"),
    (C, "const double scale = 1.0 / sqrt((double)dq);", "const double scale = 1.0 / sqrt((double)d);",
     "decoupled scale without the rotary width"),
    (C, "pos * pow(dm->rope_base, -2.0 * f / d_rope);", "pos * pow(dm->rope_base, -2.0 * f / dm->d);",
     "rotary branch frequencies over d"),
    (C, "rope_rotate_branch(dm, d_rope, qv + d, ", "rope_rotate_branch(dm, d_rope, qv, ", "rotary query read from the content part"),
    (C, "for (int e = 0; e < d_rope; ++e) acc += qr[e] * kr[e];", "", "rotary score term dropped"),
    (C, "for (int e = 0; e < d; ++e) acc += qv[e] * kh[e];\n            for (int e = 0; e < d_rope",
     "for (int e = 0; e < d_rope", "content score term dropped"),
    (C, "rope_rotate(dm, k + (bh * L_max + j) * d, (double)(j + pos_offset), kr);",
     "rope_rotate(dm, k + (bh * L_max + j) * d, (double)(j), kr);", "uncompressed keys ignore the offset"),
    (C, "o[e] += p[j] * v[(bh * L_max + j) * d + e];", "o[e] += p[j] * v[(bh * L_max + j) * d + (d - 1 - e)];",
     "uncompressed value columns reversed"),
    (C, "else rounded = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "else rounded = fl + 1.0;", "bf16 ties away from zero"),
    (C, "double scaled = ldexp(fabs(x), 8 - e);", "double scaled = ldexp(fabs(x), 7 - e);", "bf16 with 7 significant bits"),
    (C, "if (e < -125) e = -125;", "", "bf16 subnormal spacing dropped"),
    (C, "if (y > 3.3895313892515355e38) y = INFINITY;", "", "bf16 overflow to infinity dropped"),
    (C, "double teacher = 2.0 * dm->T * dm->d;", "double teacher = 1.0 * dm->T * dm->d;", "ratio without K and V"),
    (C, "if (dm->variant == 1) teacher *= dm->H;", "", "LLA-2D ratio without the heads"),
    (C, "if (dm->variant == 0) per_layer *= dm->H;", "", "per-head latent count without the heads"),
    ("oracle/paged.py", "= pool[pg]\n", "= pool[pg][:, ::-1]\n", "page rows read in reverse"),
    ("oracle/paged.py", "pg = int(bt[b, lp])\n            out", "pg = int(bt[b, min(lp + 1, max_pages - 1)])\n            out",
     "gather reads the next table entry"),
    ("oracle/paged.py", "return int(bt[b, j // page_size]), j % page_size",
     "return int(bt[b, j % page_size]), j // page_size", "slot with page and row swapped"),
    ("oracle/paged.py", "rows = dense[b, :, lp * P:min((lp + 1) * P, L), :]",
     "rows = dense[b, :, lp * P + 1:min((lp + 1) * P + 1, L), :]", "scatter shifted by one row"),
    ("oracle/__init__.py", "slp, qposp,\n                             int(pos_offset), wkp, wvp, mkp, mvp,",
     "slp, qposp,\n                             int(pos_offset), wkp, wvp, mvp, mkp,", "decode wrapper swaps the K and V means"),
    ("oracle/__init__.py", "kwp, vwp, nwp, wposp", "vwp, kwp, nwp, wposp", "hybrid wrapper swaps window keys and values"),
    ("oracle/__init__.py", "B, L_max, 1 if round_to_bf16 else 0)", "B, L_max, 0)", "encode wrapper never rounds to bf16"),
    ("oracle/evict.py", "list(range(L - window, L))", "list(range(L - window - 1, L - 1))", "eviction window off by one"),
    ("oracle/evict.py", "= cache[b][:, keep]", "= cache[b][:, sorted(keep, reverse=True)]", "kept tokens in reverse"),
]


def _copy(dst):
    """The oracle sources and the CPU pin tests, without built files."""
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    os.makedirs(os.path.join(dst, "tests"))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    pins = sorted(f for f in os.listdir(os.path.join(ROOT, "tests"))
                  if f.startswith("test_oracle_") and f.endswith("_pins.py") or f == "test_oracle_pins.py")
    for f in pins + ["conftest.py"]:
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    return ["tests/" + f for f in pins]


def _run(args):
    i, base = args
    f, old, new, _ = MUTANTS[i]
    dst = os.path.join(base, "m%02d" % i)
    pins = _copy(dst)
    path = os.path.join(dst, f)
    with open(path) as fh:
        src = fh.read()
    assert src.count(old) == 1, (i, "text to mutate not found once")
    with open(path, "w") as fh:
        fh.write(src.replace(old, new))
    # the mutant must still build: a failure below is then a pin, not the compiler
    if f.endswith(".c"):
        cc = subprocess.run(["gcc", "-std=c11", "-fopenmp", "-fsyntax-only", path], capture_output=True, text=True)
        assert cc.returncode == 0, (i, cc.stderr[-400:])
    else:
        py_compile.compile(path, doraise=True)
    env = {k: v for k, v in os.environ.items() if k != "PYTHONPATH"}
    env["OMP_NUM_THREADS"] = "1"
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"] + pins,
                       cwd=dst, env=env, capture_output=True, text=True, timeout=600)
    return i, r.returncode, r.stdout[-400:]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    # the unmutated copy passes, so a failure below is the planted mistake's
    clean = tmp_path / "clean"
    pins = _copy(str(clean))
    env = {k: v for k, v in os.environ.items() if k != "PYTHONPATH"}
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"] + pins,
                       cwd=str(clean), env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(_run, [(i, str(tmp_path)) for i in range(len(MUTANTS))]))
    survivors = [(i, MUTANTS[i][3]) for i, rc, _ in results if rc != 1]
    assert not survivors, survivors


@pytest.mark.parametrize("i", range(len(MUTANTS)))
def test_mutation_text_present(i):
    """Each planted mistake names text the oracle holds exactly once (a stale case
    fails here rather than passing unmutated)."""
    f, old, new, _ = MUTANTS[i]
    with open(os.path.join(ROOT, f)) as fh:
        assert fh.read().count(old) == 1
    assert old != new
