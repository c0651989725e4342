"""Mutation check of the oracle's pins (CPU only).

The pins in test_oracle.py are meant to catch any plausible slip in the
oracle: a dropped term, a wrong sign, index or stride, a transposed operand,
a misread storage format. This file plants each such slip, one at a time, in
a private copy of the oracle package and runs the whole of test_oracle.py
against that copy in a process of its own. Every mutant must make at least
one pin fail (pytest exit status 1: a failed check, not a crash), and the
unchanged copy must pass every pin, which shows that the harness itself
works.

Left out on purpose are mutants that are equivalent in exact arithmetic, which
no pin can or should catch: taking the softmax shift from another score than
the maximum (the shift cancels between numerator and denominator), or a wrong
block maximum in the online recurrence (the same cancellation).

Each mutant is a literal substitution that must match the source exactly once,
so a change to the oracle's text fails this file loudly instead of leaving a
mutant that no longer changes anything.
"""
import os
import re
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")
PINS = os.path.join(ROOT, "tests", "test_oracle.py")
C = "decode_attn_oracle.c"
PY = "__init__.py"

# (name, file, text in the oracle, the slip planted in its place)
MUTANTS = [
    # the plain definition: scores, softmax, weighted sum
    ("K read with the wrong KV head", C,
     "int kv = h / (s->n_heads / s->n_kv_heads);\n    const double *qh",
     "int kv = h % s->n_kv_heads;\n    const double *qh"),
    ("V read with the wrong KV head", C,
     "int kv = h / (s->n_heads / s->n_kv_heads);\n    orc_scores(",
     "int kv = h % s->n_kv_heads;\n    orc_scores("),
    ("scale dropped", C, "sc[j] = s->scale * dot;", "sc[j] = dot;"),
    ("exp sign flipped", C, "sc[j] = exp(sc[j] - m);", "sc[j] = exp(m - sc[j]);"),
    ("no normalisation by Z", C, "out[e] = acc / Z;", "out[e] = acc;"),
    ("Z off by one", C, "double Z = 0.0;", "double Z = 1.0;"),
    ("last position left out of the weighted sum", C,
     "for (int j = 0; j < L; ++j)\n            acc += sc[j]",
     "for (int j = 0; j < L - 1; ++j)\n            acc += sc[j]"),
    ("K position and head strides transposed", C,
     "(int64_t)j * s->k_pos_stride +\n                      (int64_t)kv * s->k_head_stride",
     "(int64_t)j * s->k_head_stride +\n                      (int64_t)kv * s->k_pos_stride"),
    ("V position and head strides transposed", C,
     "(int64_t)j * s->v_pos_stride +\n                  (int64_t)kv * s->v_head_stride",
     "(int64_t)j * s->v_head_stride +\n                  (int64_t)kv * s->v_pos_stride"),
    ("V batch offset dropped", C,
     "int64_t idx = (int64_t)b * s->v_batch_stride + ", "int64_t idx = 0 * s->v_batch_stride + "),
    # storage readers
    ("f16 exponent bias off by one", C, "expo - 25", "expo - 24"),
    ("f16 subnormal scale off by one", C, "ldexp((double)mant, -24)", "ldexp((double)mant, -25)"),
    ("f16 implicit leading bit dropped", C, "(mant | 0x400)", "(mant)"),
    ("f16 sign dropped", C, "return sign ? -v : v;", "return v;"),
    ("bf16 read as f16", C, "case ORC_BF16: return orc_from_bf16(",
     "case ORC_BF16: return orc_from_f16("),
    # the merge of partial triples
    ("merge: l summed without exp(m_i - m)", C, "L += w * l[i];", "L += l[i];"),
    ("merge: O summed without exp(m_i - m)", C, "out[e] += w * O[(int64_t)i * dv + e];",
     "out[e] += O[(int64_t)i * dv + e];"),
    ("merge: reference taken as the smallest m", C, "if (m[i] > M) M = m[i];",
     "if (m[i] < M) M = m[i];"),
    ("LSE merge: O_i not divided by l_i", C, "wgt * (O[(int64_t)i * dv + e] / l[i])",
     "wgt * O[(int64_t)i * dv + e]"),
    ("LSE merge: log of the weight sum dropped", C, "double lse_star = lse_max + log(z);",
     "double lse_star = lse_max;"),
    ("merge: merged m not returned", C, "if (m_out) *m_out = M;", "if (m_out) *m_out = 0.0;"),
    ("merge: merged l not returned", C, "if (l_out) *l_out = L;", "if (l_out) *l_out = 1.0;"),
    ("LSE merge: merged LSE taken from the largest partial", C, "if (m_out) *m_out = lse_star;",
     "if (m_out) *m_out = lse_max;"),
    # the online recurrence inside a segment
    ("recurrence: O not rescaled by alpha", C,
     "for (int e = 0; e < s->v_dim; ++e) O[e] *= alpha;",
     "for (int e = 0; e < s->v_dim; ++e) O[e] *= 1.0;"),
    ("recurrence: l not rescaled by alpha", C, "l *= alpha;", "l *= 1.0;"),
    ("recurrence: alpha sign flipped", C, "exp(m - mn)", "exp(mn - m)"),
    ("recurrence: weights from the old maximum", C, "double p = exp(sc[j] - mn);",
     "double p = exp(sc[j] - m);"),
    ("empty segment not neutral in m", C, "*m_out = -1e30;", "*m_out = 0.0;"),
    ("split: chunk rounded down", C, "int chunk = (L + n_splits - 1) / n_splits;",
     "int chunk = L / n_splits;"),
    ("split: segment one position short", C, "z = a + chunk;", "z = a + chunk - 1;"),
    ("split: wrong KV head", C,
     "int kv = h / (s->n_heads / s->n_kv_heads);\n        int L = seq_lens[b];",
     "int kv = h % s->n_kv_heads;\n        int L = seq_lens[b];"),
    # the Python compositions
    ("several tokens: causal limit one position short", PY, "(lens - T + 1 + t)",
     "(lens - T + t)"),
    ("several tokens: causal limit one position long", PY, "(lens - T + 1 + t)",
     "(lens - T + 2 + t)"),
    ("projection: weight matrix transposed", PY, '"...hc,hec->...he"', '"...hc,hce->...he"'),
    ("projection: pairs take the first heads' matrices", PY, "W[[h for _, h in pairs]]",
     "W[[i for i, _ in enumerate(pairs)]]"),
]

_RUNNER = (
    "import sys\n"
    "sys.path.insert(0, sys.argv[1])\n"
    "import oracle\n"
    "assert oracle.__file__.startswith(sys.argv[1]), oracle.__file__\n"
    "sys.path.insert(1, sys.argv[2])\n"
    "import pytest\n"
    "sys.exit(pytest.main(['-x', '-q', '-rf', '-p', 'no:cacheprovider', '-m', 'not gpu',\n"
    "                      sys.argv[3]]))\n"
)


def _copy_oracle(dst: str, mutant=None) -> None:
    shutil.copytree(ORACLE, os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("_build", "__pycache__", "*.so"))
    if mutant is None:
        return
    _, fname, old, new = mutant
    path = os.path.join(dst, "oracle", fname)
    with open(path) as f:
        src = f.read()
    if src.count(old) != 1:
        raise AssertionError(f"mutant {mutant[0]!r}: its text occurs {src.count(old)} times "
                             f"in oracle/{fname}, not once")
    with open(path, "w") as f:
        f.write(src.replace(old, new))


def _run_pins(mutant):
    """Run test_oracle.py against a copy of the oracle (mutated unless None).
    Returns (pytest exit status, the first failing check or the output's tail)."""
    with tempfile.TemporaryDirectory(prefix="orc_mut_") as tmp:
        try:
            _copy_oracle(tmp, mutant)
        except AssertionError as e:
            return -1, str(e)
        env = dict(os.environ, OMP_NUM_THREADS="1", PYTHONDONTWRITEBYTECODE="1")
        r = subprocess.run([sys.executable, "-c", _RUNNER, tmp, ROOT, PINS], cwd=ROOT, env=env,
                           capture_output=True, text=True, timeout=600)
        out = r.stdout + r.stderr
        failed = re.findall(r"^FAILED (\S+)", out, flags=re.M)
        return r.returncode, (failed[0] if failed else out[-2000:])


@pytest.fixture(scope="module")
def results():
    jobs = [None] + MUTANTS
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        outcomes = list(ex.map(_run_pins, jobs))
    return {("control" if j is None else j[0]): o for j, o in zip(jobs, outcomes)}


def test_unchanged_copy_passes_every_pin(results):
    status, detail = results["control"]
    assert status == 0, f"the unmutated copy of the oracle fails its pins:\n{detail}"


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_is_caught_by_a_pin(results, name):
    status, detail = results[name]
    assert status == 1, (f"mutant {name!r} was not caught by a failing check "
                         f"(pytest exit status {status}):\n{detail}")
