"""The oracle's pins catch planted mistakes.

Each case copies oracle/, synth/ and the oracle's pin tests into a temporary
directory and plants one plausible mistake in the copy: a swapped operand, a
dropped rounding, a wrong index, a wrong tie rule or a dropped term. It then
runs the pins there. Every planted mistake must make them fail, and the
unmodified copy must pass. The files under oracle/ are never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, file, original text, planted text).  Not listed: mistakes that give
# the same results in exact arithmetic, such as an all-zero residual falling
# back to q instead of p (the residual max(0, p - q) of two distributions is
# all zero only when p = q).
MUTATIONS = [
    ("accept test p and q swapped", "oracle/verify.py",
     "u[j] * q_rows[j][x] < p_rows[j][x]", "u[j] * p_rows[j][x] < q_rows[j][x]"),
    ("residual sign", "oracle/verify.py", "diff = p - q", "diff = q - p"),
    ("bonus token from the last drafted row", "oracle/verify.py",
     "tok = inverse_cdf(np.asarray(p_rows[gamma]), u[gamma])",
     "tok = inverse_cdf(np.asarray(p_rows[gamma-1]), u[gamma])"),
    ("greedy stop one position late", "oracle/verify.py",
     "            n = j\n", "            n = j + 1\n"),
    ("greedy argmax ties to the highest index", "oracle/verify.py",
     "int(np.nonzero(t[j] == np.max(t[j]))[0][0])",
     "int(np.nonzero(t[j] == np.max(t[j]))[0][-1])"),
    ("inverse CDF takes >= for >", "oracle/head.py",
     "hits = np.nonzero(cum > target)[0]", "hits = np.nonzero(cum >= target)[0]"),
    ("LSE without the temperature", "oracle/head.py",
     "\"lse\": m / T + logW", "\"lse\": m + logW"),
    ("z not rounded to bf16", "oracle/head.py",
     "        z = round_to_bf16(z)\n", "        z = z\n"),
    ("W_up rows reversed", "oracle/head.py",
     "return np.asarray(z, np.float64) @ np.asarray(w_up, np.float64).T",
     "return np.asarray(z, np.float64) @ np.asarray(w_up, np.float64).T[::-1]"),
    ("trimmed head maps through reversed ids", "oracle/head.py",
     "out[\"tokens\"] = np.asarray(kept_ids, np.int64)[out[\"tokens\"]]",
     "out[\"tokens\"] = np.asarray(kept_ids, np.int64)[::-1][out[\"tokens\"]]"),
    ("low-rank verify reads W_up rows reversed", "oracle/verify.py",
     "draft = np.stack([up_projection(z[b], w_up) for b in range(B)])",
     "draft = np.stack([up_projection(z[b], np.asarray(w_up)[::-1]) for b in range(B)])"),
    ("bf16 keeps one bit too many", "oracle/bf16.py",
     "_BF16_SIG_BITS = 8", "_BF16_SIG_BITS = 9"),
    ("bf16 ties rounded away from even", "oracle/bf16.py",
     "y = np.rint(x / spacing) * spacing", "y = np.floor(x / spacing + 0.5) * spacing"),
    ("top-k ties to the highest id", "oracle/specvocab.py",
     "order = np.lexsort((ids, -s))", "order = np.lexsort((-ids, -s))"),
    ("router h' not rounded to bf16", "oracle/specvocab.py",
     "        hp = round_to_bf16(hp)\n", "        hp = hp\n"),
    ("expected tokens drop the last run", "oracle/theory.py",
     "return total + run", "return total"),
    ("inverse CDF falls back to the first positive weight", "oracle/head.py",
     "return int(positive[-1])", "return int(positive[0])"),
    ("logprob adds log W", "oracle/head.py",
     "\"logprob\": (float(l[token]) - m) / T - logW",
     "\"logprob\": (float(l[token]) - m) / T + logW"),
    ("draw ignores the temperature", "oracle/head.py",
     "w = np.exp((l - m) / T)", "w = np.exp(l - m)"),
    ("residual takes |p - q|", "oracle/verify.py",
     "resid = np.where(diff > 0, diff, diff * 0)", "resid = np.abs(diff)"),
    ("softmax multiplies by T", "oracle/verify.py",
     "w = np.exp((l - np.max(l)) / float(temperature))",
     "w = np.exp((l - np.max(l)) * float(temperature))"),
    ("greedy bonus from the last drafted row", "oracle/verify.py",
     "return [int(x) for x in draft_tokens[:n]] + [a[n]], n",
     "return [int(x) for x in draft_tokens[:n]] + [a[min(n, gamma - 1)]], n"),
    ("SpecVocab q not normalised", "oracle/specvocab.py",
     "q[i] = w / w.sum()", "q[i] = w"),
    ("SpecVocab exact logits from the next row of h", "oracle/specvocab.py",
     "zc[i] = np.asarray(u_full[cand[i]], np.float64) @ hidden[i]",
     "zc[i] = np.asarray(u_full[cand[i]], np.float64) @ hidden[(i + 1) % M]"),
    ("SpecVocab token not mapped to its vocabulary id", "oracle/specvocab.py",
     "tokens[i] = cand[i][red[\"token\"]]", "tokens[i] = red[\"token\"]"),
    ("Philox multipliers swapped", "oracle/philox.py",
     "PHILOX_M4x32 = (0xD2511F53, 0xCD9E8D57)", "PHILOX_M4x32 = (0xCD9E8D57, 0xD2511F53)"),
    ("Philox nine rounds", "oracle/philox.py", "ROUNDS = 10", "ROUNDS = 9"),
    ("Philox key bumped before the first round", "oracle/philox.py",
     "        if i > 0:  # the key schedule", "        if i >= 0:  # the key schedule"),
    ("Philox round keeps c1 in place of the low product", "oracle/philox.py",
     "(p1 >> bits) ^ c1 ^ k0, p1 & mask,", "(p1 >> bits) ^ c1 ^ k0, c1,"),
    ("vectorised Philox drops the second key word", "oracle/philox.py",
     "(p0 >> s32) ^ c3 ^ k1, p0 & m32)", "(p0 >> s32) ^ c3, p0 & m32)"),
    ("uniform from the last output word", "oracle/philox.py",
     "x0 = philox4x32_10(ctr, key)[..., 0]", "x0 = philox4x32_10(ctr, key)[..., 3]"),
    ("offset words swapped in the counter", "oracle/philox.py",
     "ctr = np.stack([row, slot, np.full_like(row, offset & _MASK32),\n"
     "                    np.full_like(row, offset >> 32)], axis=-1)",
     "ctr = np.stack([row, slot, np.full_like(row, offset >> 32),\n"
     "                    np.full_like(row, offset & _MASK32)], axis=-1)"),
    ("uniform keeps 23 bits", "oracle/philox.py",
     "return (x0 >> 8) * 2.0 ** -24", "return (x0 >> 9) * 2.0 ** -23"),
    ("closed form one power short", "oracle/theory.py",
     "return (1 - alpha ** (gamma + 1)) / (1 - alpha)", "return (1 - alpha ** gamma) / (1 - alpha)"),
]


def _copy(dst):
    ign = shutil.ignore_patterns("__pycache__", "*.pyc")
    for d in ("oracle", "synth"):
        shutil.copytree(os.path.join(ROOT, d), os.path.join(dst, d), ignore=ign)
    os.makedirs(os.path.join(dst, "tests"))
    for f in os.listdir(os.path.join(ROOT, "tests")):
        if f.startswith("test_oracle_") and f != os.path.basename(__file__) or f == "conftest.py":
            shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"),
                    ignore=ign)
    shutil.copy(os.path.join(ROOT, "pytest.ini"), os.path.join(dst, "pytest.ini"))


def _pins_pass(dst) -> bool:
    env = dict(os.environ)
    env.pop("PYTHONPATH", None)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests"], cwd=dst, env=env, capture_output=True, text=True, timeout=900)
    if r.returncode not in (0, 1):   # 1 = tests failed; anything else is a broken run
        raise RuntimeError(r.stdout[-2000:] + r.stderr[-2000:])
    return r.returncode == 0


def test_unmodified_copy_passes(tmp_path):
    _copy(str(tmp_path))
    assert _pins_pass(str(tmp_path))


@pytest.mark.parametrize("name,path,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, path, old, new):
    _copy(str(tmp_path))
    f = os.path.join(str(tmp_path), path)
    src = open(f, encoding="utf-8").read()
    assert src.count(old) == 1, f"anchor not found once in {path}: {old!r}"
    with open(f, "w", encoding="utf-8") as fh:
        fh.write(src.replace(old, new))
    assert not _pins_pass(str(tmp_path)), f"the pins did not catch: {name}"
