"""The oracle's pins catch plausible mistakes.

Each case plants one mistake (a dropped term, a flipped sign, a wrong index,
layout or bias) in a temporary copy of the oracle's C source, builds that copy
on the CPU, points the oracle module at it, and runs the pins of
``tests/test_oracle.py`` until one fails (an assertion, or the oracle refusing
its input); the case passes when one does.  The oracle's own source and
library are not touched.
"""
import importlib.util
import inspect
import os
import shutil
import subprocess

import pytest

import oracle
from oracle import build as oracle_build
from oracle import scheduler as scheduler_src
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
    ("append: page row p / 64", "int64_t dst = ((page * Hk + h) * ORACLE_PAGE + p % ORACLE_PAGE) * D;",
     "int64_t dst = ((page * Hk + h) * ORACLE_PAGE + p / ORACLE_PAGE) * D;", 0, 1),
    ("append: e4m3 scale multiplied", "float kf = (float)oracle_bf16_to_double(k_new[src + d]) / k_scale[h];",
     "float kf = (float)oracle_bf16_to_double(k_new[src + d]) * k_scale[h];", 0, 1),
    ("fp8 MLA: q_scale dropped", "double qs = (double)q_scale[h], ks = (double)k_scale[g];",
     "double qs = 1.0, ks = (double)k_scale[g];", 0, 1),
    ("fp8 MLA: k_scale of head 0", "double qs = (double)q_scale[h], ks = (double)k_scale[g];",
     "double qs = (double)q_scale[h], ks = (double)k_scale[0];", 0, 1),
    ("e4m3 rope key: token scale dropped", "double rs = (double)k_rope_scales[t];", "double rs = 1.0;", 0, 1),
]

# the same for the scheduler's restatement (oracle/scheduler.py) and its pins
SCHEDULER_MUTATIONS = [
    ("chunk rounded down", "chunk = max(MIN_CHUNK, _cdiv(units, cap * ITEMS_PER_SHARE))",
     "chunk = max(MIN_CHUNK, units // (cap * ITEMS_PER_SHARE))"),
    ("last split one page long", "return (s * pages) // nsplit, ((s + 1) * pages) // nsplit",
     "return (s * pages) // nsplit, ((s + 1) * pages) // nsplit + (s + 1 == nsplit)"),
    ("item cost without the +1", "items.append((hi - lo + 1, len(items), b, s, kvh))",
     "items.append((hi - lo, len(items), b, s, kvh))"),
    ("ties by descending index", "key=lambda it: (-it[0], it[1])", "key=lambda it: (-it[0], -it[1])"),
    ("snake dealing without the turn", "per_cta[pos if rnd % 2 == 0 else grid - 1 - pos]", "per_cta[pos]"),
    ("forced splits not capped by the pages", "n.append(min(forced_splits, p, MAX_SPLITS))",
     "n.append(min(forced_splits, MAX_SPLITS))"),
    ("flat page list: page count rounded down", "counts.append((n + page_size - 1) // page_size)",
     "counts.append(n // page_size)"),
    ("flat page list: offset not advanced", "        start += c\n    return table", "    return table"),
    ("flat page list: ids right-aligned", "table[b][j] = int(kv_indices[start + j])",
     "table[b][width - c + j] = int(kv_indices[start + j])"),
]


def pin_calls(module=pins):
    """Every pin of a test module as a no-argument call (parametrized pins once
    per parameter set)."""
    calls = []
    for name, fn in inspect.getmembers(module, inspect.isfunction):
        if not name.startswith("test_") or fn.__module__ != module.__name__:
            continue
        params = list(inspect.signature(fn).parameters)
        if not params:
            calls.append((name, fn, {}))
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        assert len(marks) == 1, f"{name}: one parametrize mark expected"
        argnames = [x.strip() for x in marks[0].args[0].split(",")]
        assert sorted(argnames) == sorted(params), f"{name}: every argument comes from the mark"
        for v in marks[0].args[1]:
            kw = dict(zip(argnames, v if len(argnames) > 1 else (v,)))
            calls.append((f"{name}[{v}]", fn, kw))
    return calls


def first_failing_pin(module):
    for name, fn, kw in pin_calls(module):
        try:
            fn(**kw)
        except Exception:  # a failed assertion, or the oracle refusing its input
            return name
    return None


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
    caught = first_failing_pin(pins)
    monkeypatch.setattr(oracle, "_lib", None)  # the next user reloads the real library
    assert caught is not None, f"no pin fails with the mistake: {mistake}"


@pytest.mark.parametrize("mistake,old,new", SCHEDULER_MUTATIONS, ids=[m[0] for m in SCHEDULER_MUTATIONS])
def test_a_planted_scheduler_mistake_fails_a_pin(tmp_path, monkeypatch, mistake, old, new):
    from tests import test_scheduler_oracle as sched_pins
    src = open(scheduler_src.__file__).read()
    assert src.count(old) == 1, f"the scheduler source changed: {old!r}"
    path = tmp_path / "scheduler_mutant.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("scheduler_mutant", path)
    mutant = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mutant)
    monkeypatch.setattr(sched_pins, "S", mutant)
    assert first_failing_pin(sched_pins) is not None, f"no pin fails with the mistake: {mistake}"


def test_scheduler_pins_pass_on_an_unmodified_copy(tmp_path, monkeypatch):
    from tests import test_scheduler_oracle as sched_pins
    path = tmp_path / "scheduler_copy.py"
    path.write_text(open(scheduler_src.__file__).read())
    spec = importlib.util.spec_from_file_location("scheduler_copy", path)
    copy = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(copy)
    monkeypatch.setattr(sched_pins, "S", copy)
    for name, fn, kw in pin_calls(sched_pins):
        fn(**kw)


def test_pins_pass_on_the_unmodified_source(tmp_path, monkeypatch):
    """The harness itself: the same rebuild of the unchanged source passes every pin."""
    src = open(oracle_build.SRC).read()
    lib = build_mutant(tmp_path, src[:40], src[:40], 0, None)
    monkeypatch.setattr(oracle, "_LIB", lib)
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "_build", lambda *a, **k: lib)
    for name, fn, kw in pin_calls(pins):
        fn(**kw)
    monkeypatch.setattr(oracle, "_lib", None)
    assert os.path.exists(lib)
