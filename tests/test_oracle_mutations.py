"""The oracle's pins catch plausible mistakes.

Each case plants one mistake (a dropped term, a flipped sign, a wrong index,
layout or bias) in a temporary copy of the oracle's C source, builds that copy
on the CPU, points the oracle module at it, and runs the pins of
``tests/test_oracle.py`` until one fails (an assertion, or the oracle refusing
its input); the case passes when one does.  The oracle's own source and
library are not touched.
"""
import inspect
import os
import shutil
import subprocess

import pytest

import oracle
from oracle import build as oracle_build
from tests import test_oracle as pins

# (mistake, text in the oracle's source, replacement, which occurrence, occurrences)
MUTATIONS = [
    ("score scale dropped", "s[j] = scale * acc;", "s[j] = acc;", 0, 1),
    ("lse without the row max", "*lse = m + log(l);", "*lse = log(l);", 0, 1),
    ("output not divided by the sum", "for (int d = 0; d < dv; ++d) out[d] /= l;", "", 0, 1),
    ("exponent sign flipped", "double p = exp(s[j] - m);", "double p = exp(m - s[j]);", 0, 1),
    ("decode: KV head by modulo", "int kvh = h / group;", "int kvh = h % Hk;", 0, 2),
    ("prefill: KV head by modulo", "int kvh = h / group;", "int kvh = h % Hk;", 1, 2),
    ("decode: page slot j % 64", "block_table[(int64_t)b * max_pages + j / ORACLE_PAGE]",
     "block_table[(int64_t)b * max_pages + j % ORACLE_PAGE]", 0, 2),
    ("decode: token-major rows in a page", "int64_t row = ((page * Hk + kvh) * ORACLE_PAGE + j % ORACLE_PAGE) * D;",
     "int64_t row = ((page * ORACLE_PAGE + j % ORACLE_PAGE) * Hk + kvh) * D;", 0, 1),
    ("causal limit one key short", "int64_t lim = off + i + 1;", "int64_t lim = off + i;", 0, 3),
    ("default qo_offset 0", "qo_offset ? qo_offset[b] : kv_len - q_len", "qo_offset ? qo_offset[b] : 0", 0, None),
    ("MLA rope term dropped", "kd[j * Dqk + Dk + d] = load_elem(k_rope, elem_kind, (cu_k[b] + j) * rope_dim + d);",
     "kd[j * Dqk + Dk + d] = 0.0;", 0, 1),
    ("e4m3 exponent bias 8", "mag = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "mag = ldexp(1.0 + (double)m / 8.0, e - 8);", 0, 1),
]


def pin_calls():
    """Every pin of tests/test_oracle.py as a no-argument call (parametrized
    pins once per parameter value)."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_") or fn.__module__ != pins.__name__:
            continue
        params = list(inspect.signature(fn).parameters)
        if not params:
            calls.append((name, fn, {}))
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        assert len(marks) == 1 and len(params) == 1, f"{name}: one parametrized argument expected"
        argname, values = marks[0].args[0], marks[0].args[1]
        for v in values:
            calls.append((f"{name}[{v}]", fn, {argname: v}))
    return calls


def build_mutant(tmp_path, old, new, which, count):
    src = open(oracle_build.SRC).read()
    if count is not None:
        assert src.count(old) == count, f"the oracle source changed: {old!r} occurs {src.count(old)} times"
    at = -1
    for _ in range(which + 1):
        at = src.index(old, at + 1)
    mutated = src[:at] + new + src[at + len(old):]
    path = tmp_path / "oracle_mutant.c"
    path.write_text(mutated)
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-fno-fast-math", str(path), "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    return str(lib)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("mistake,old,new,which,count", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_a_planted_mistake_fails_a_pin(tmp_path, monkeypatch, mistake, old, new, which, count):
    lib = build_mutant(tmp_path, old, new, which, count)
    monkeypatch.setattr(oracle, "_LIB", lib)
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "_build", lambda *a, **k: lib)
    caught = None
    for name, fn, kw in pin_calls():
        try:
            fn(**kw)
        except Exception:  # a failed assertion, or the oracle refusing its input
            caught = name
            break
    monkeypatch.setattr(oracle, "_lib", None)  # the next user reloads the real library
    assert caught is not None, f"no pin fails with the mistake: {mistake}"


def test_pins_pass_on_the_unmodified_source(tmp_path, monkeypatch):
    """The harness itself: the same rebuild of the unchanged source passes every pin."""
    src = open(oracle_build.SRC).read()
    lib = build_mutant(tmp_path, src[:40], src[:40], 0, None)
    monkeypatch.setattr(oracle, "_LIB", lib)
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "_build", lambda *a, **k: lib)
    for name, fn, kw in pin_calls():
        fn(**kw)
    monkeypatch.setattr(oracle, "_lib", None)
    assert os.path.exists(lib)
