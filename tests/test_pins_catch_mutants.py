"""The oracle's pins catch plausible mistakes. Each case plants one mistake in
a copy of the oracle (a dropped term, a wrong sign, index or axis, a
transposed operand, an off-by-one mask, another reading of a mapping) and
runs the oracle pin tests against it in a subprocess: at least one pin must
fail. The control run, with nothing planted, must pass, so a failure cannot
come from the mechanism itself. CPU only; the mistakes live in the copy,
never in the oracle's file."""
import json
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_FILES = ["tests/test_oracle_softmax.py", "tests/test_oracle_attention.py",
             "tests/test_oracle_gqa.py", "tests/test_oracle_merge_decode.py"]

# (what the mistake is, text in oracle/attention.py, replacement)
MUTANTS = [
    ("scores without the scale",
     "s = scale * (qb @ k.T)", "s = qb @ k.T"),
    ("causal mask one key too far",
     "cols[None, :] <= rows[:, None]", "cols[None, :] <= rows[:, None] + 1"),
    ("causal mask transposed (keys after the query)",
     "cols[None, :] <= rows[:, None]", "cols[None, :] >= rows[:, None]"),
    ("lse without the max",
     "lse[c0:c0 + r.shape[0]] = (m + np.log(l))[:, 0]", "lse[c0:c0 + r.shape[0]] = np.log(l)[:, 0]"),
    ("forward output not normalised",
     "o[c0:c0 + r.shape[0]] = p @ v", "o[c0:c0 + r.shape[0]] = e @ v"),
    ("forward output from the keys",
     "o[c0:c0 + r.shape[0]] = p @ v", "o[c0:c0 + r.shape[0]] = p @ k"),
    ("safe softmax without the max shift",
     "    e = np.exp(x - m)\n", "    e = np.exp(x)\n"),
    ("online softmax rescale with the wrong sign",
     "alpha = math.exp(m - m_new) if m != -math.inf else 0.0",
     "alpha = math.exp(m_new - m) if m != -math.inf else 0.0"),
    ("online softmax numerator not rescaled",
     "u = alpha * u + np.tensordot(e, vb, axes=(0, 0))", "u = u + np.tensordot(e, vb, axes=(0, 0))"),
    ("backward: dS without the D term",
     "ds = p * (dp - Dr[:, None])\n        dq[r]", "ds = p * dp\n        dq[r]"),
    ("backward: D summed over the wrong axis",
     "Dr = np.sum(p * dp, axis=1)\n        ds", "Dr = np.sum(p * dp, axis=0)\n        ds"),
    ("backward: dV with P not transposed",
     "dv += p.T @ do[r]", "dv += p @ do[r]"),
    ("backward: dP from K instead of V",
     "dp = do[r] @ v.T\n        Dr", "dp = do[r] @ k.T\n        Dr"),
    ("backward: dQ without the scale",
     "dq[r] = scale * (ds @ k)", "dq[r] = ds @ k"),
    ("backward: dK from dO instead of Q",
     "dk += scale * (ds.T @ q[r])", "dk += scale * (ds.T @ do[r])"),
    ("grouped-query heads interleaved instead of consecutive",
     "return h // (H // Hkv)", "return h % Hkv"),
    ("grouped-query K/V gradient overwritten instead of summed",
     "dk[b, g] += dkh", "dk[b, g] = dkh"),
    ("merge: rescale of the carried state with the wrong sign",
     "a_old = np.where(live, np.exp(np.where(live, m - m_new, 0.0)), 0.0)",
     "a_old = np.where(live, np.exp(np.where(live, m_new - m, 0.0)), 0.0)"),
    ("merge: carried normaliser not rescaled",
     "l = l * a_old + a_new", "l = l + a_new"),
    ("paged cache: slot and block swapped",
     "blocks = np.asarray(block_table_row)[t // bs]\n    return cache[blocks, :, t % bs, :]",
     "blocks = np.asarray(block_table_row)[t % bs]\n    return cache[blocks, :, t // bs, :]"),
    ("decode: the new token's query masked causally",
     "K[g], V[g], scale, False)", "K[g], V[g], scale, True)"),
    ("causal pair count without the diagonal",
     "return N * (N + 1) // 2 if causal else N * N", "return N * (N - 1) // 2 if causal else N * N"),
    ("backward FLOPs counted as four products",
     '"bwd": 10 * d', '"bwd": 8 * d'),
]


def run_pins(mutant):
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([ROOT, os.path.join(ROOT, "tests")] +
                                        ([env["PYTHONPATH"]] if env.get("PYTHONPATH") else []))
    env.pop("ORACLE_MUTANT", None)
    if mutant is not None:
        env["ORACLE_MUTANT"] = json.dumps([mutant[1], mutant[2]])
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
           "-p", "oracle_mutant_plugin", "-m", "not gpu", *PIN_FILES]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:] + r.stderr[-2000:]


def test_mutation_sites_exist_once():
    with open(os.path.join(ROOT, "oracle", "attention.py"), encoding="utf-8") as f:
        src = f.read()
    for name, old, new in MUTANTS + NEUTRAL:
        assert src.count(old) == 1, name
        assert old != new, name


# Replacements that keep the meaning: the copied, re-executed oracle must
# still pass every pin, so the mechanism itself fails nothing.
NEUTRAL = [
    ("row chunk written another way", "ROW_CHUNK = 1024", "ROW_CHUNK = 1 << 10"),
    ("smaller row chunks (rows are independent)", "ROW_CHUNK = 1024", "ROW_CHUNK = 3"),
]


def test_control_run_passes():
    rc, out = run_pins(None)
    assert rc == 0, out


@pytest.mark.parametrize("case", NEUTRAL, ids=[c[0] for c in NEUTRAL])
def test_neutral_rewrite_passes(case):
    rc, out = run_pins(case)
    assert rc == 0, out


def test_every_planted_mistake_fails_a_pin():
    with ThreadPoolExecutor(max_workers=min(6, os.cpu_count() or 1)) as ex:
        results = list(ex.map(run_pins, MUTANTS))
    survivors = []
    for (name, _, _), (rc, out) in zip(MUTANTS, results):
        # exit code 1: tests ran and one failed. Anything else (an error in
        # the plugin or in collection) is not a caught mistake.
        if rc != 1:
            survivors.append((name, rc, out[-600:]))
    assert not survivors, survivors
