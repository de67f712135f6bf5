"""The oracle's pins catch plausible slips: each case plants one mistake in a copy
of oracle/attention.c, builds it, runs every pin of test_oracle_attention.py
against that build (oracle.using_library) and requires at least one pin to fail.
The unchanged source, built the same way, must pass them all, so a failure
comes from the planted slip. Every slip keeps its memory accesses inside the
arrays it is given (a wrong index stays a valid one), so the mutant builds
cannot fault. CPU only (gcc). The same for the split and the planner: a copy of
oracle/split.py or oracle/planner.py with one slip is loaded as a module of its
own, its functions stand in for the oracle's while the pins of
test_oracle_split_planner.py run (all but the one that compares the library's
controller with the oracle's, which pins the library, not the oracle), and for
the batch builder (oracle/scheduler.py) with the pins of test_scheduler.py
that do not involve the library."""
import importlib.util
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_attention as pins
import test_oracle_split_planner as py_pins
import test_scheduler as sched_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attention.c")

# (name, [(text in attention.c, its replacement)]): each text occurs exactly once
SLIPS = [
    ("scale 1/d instead of 1/sqrt(d)",
     [("scale = 1.0 / sqrt((double)head_dim);", "scale = 1.0 / (double)head_dim;")]),
    ("history left out of the causal limit",
     [("long last_key = hist + i;", "long last_key = i;")]),
    ("the row's own key left out (off by one)",
     [("long nkeys = last_key + 1;", "long nkeys = last_key > 0 ? last_key : 1;")]),
    ("GQA map by modulo instead of by group",
     [("int kvh = h / group;", "int kvh = h % num_kv_heads;")]),
    ("keys read at the mirrored offset inside their page",
     [("const uint16_t *krow = k_cache + (((size_t)page * num_kv_heads + kvh) * page_size +\n"
       "                                              j % page_size) * head_dim;",
       "const uint16_t *krow = k_cache + (((size_t)page * num_kv_heads + kvh) * page_size +\n"
       "                                              (page_size - 1 - j % page_size)) * head_dim;")]),
    ("no maximum subtracted before exp",
     [("score[j] = exp(score[j] - mx);", "score[j] = exp(score[j]);")]),
    ("weights not normalised",
     [("double p = score[j] / denom;", "double p = score[j];")]),
    ("softmax denominator starts at one",
     [("double denom = 0.0;", "double denom = 1.0;")]),
    ("values gathered from the key cache",
     [("const uint16_t *vrow = v_cache +", "const uint16_t *vrow = k_cache +")]),
    ("query row of the kv head instead of the q head",
     [("const uint16_t *qrow = q + ((size_t)t * num_q_heads + h) * head_dim;",
       "const uint16_t *qrow = q + ((size_t)t * num_q_heads + kvh) * head_dim;")]),
    ("KV write: offset inside the page shifted by one",
     [("int64_t off = slot % page_size;", "int64_t off = (slot + 1) % page_size;")]),
    ("KV write: keys written into the value cache's slot order",
     [("v_cache[dst + x] = v[src + x];", "v_cache[dst + x] = k[src + x];")]),
]

PINS = [getattr(pins, n) for n in sorted(dir(pins)) if n.startswith("test_")]


def _build(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    lib = tmp_path / f"lib{name}.so"
    src.write_text(text)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", str(lib), str(src), "-lm"],
                   check=True)
    return str(lib)


def _failing_pins(lib):
    failed = []
    with oracle.using_library(lib):
        with np.errstate(all="ignore"):
            for pin in PINS:
                try:
                    pin()
                except (Exception, pytest.fail.Exception):
                    failed.append(pin.__name__)
    return failed


@pytest.fixture(scope="module")
def source():
    if shutil.which("gcc") is None:
        pytest.skip("gcc is not available")
    with open(SRC) as f:
        return f.read()


def test_unchanged_source_passes_every_pin(source, tmp_path):
    assert len(PINS) >= 10
    assert _failing_pins(_build(tmp_path, "control", source)) == []


@pytest.mark.parametrize("k", range(len(SLIPS)), ids=[s[0] for s in SLIPS])
def test_a_planted_slip_fails_some_pin(source, tmp_path, k):
    name, edits = SLIPS[k]
    text = source
    for old, new in edits:
        assert text.count(old) == 1, f"{name}: the text to change must occur once"
        text = text.replace(old, new)
    failed = _failing_pins(_build(tmp_path, f"mutant{k}", text))
    assert failed, f"no pin caught the slip '{name}'"


# ---------------------------------------------------------------- split and planner
PY_SLIPS = [
    ("split.py", "simple split takes the larger half first",
     [("b = len(query_lens) // 2", "b = (len(query_lens) + 1) // 2")]),
    ("split.py", "ties in distance go to the largest k",
     [("if best_diff is None or diff < best_diff:", "if best_diff is None or diff <= best_diff:")]),
    ("split.py", "balance measured against the larger half",
     [("balanced = abs(n1 - n2) / small <= balance_threshold",
       "balanced = abs(n1 - n2) / max(n1, n2) <= balance_threshold")]),
    ("split.py", "length threshold applied to the larger half",
     [("long_enough = small >= length_threshold", "long_enough = max(n1, n2) >= length_threshold")]),
    ("split.py", "aim at the total instead of its half",
     [("best = total // 2", "best = total")]),
    ("planner.py", "target latency keeps the constant term",
     [("return latency_quadratic(base_chunk_size, a, b, c) - latency_quadratic(0, a, b, c)",
       "return latency_quadratic(base_chunk_size, a, b, c)")]),
    ("planner.py", "linear coefficient of the chunk equation without the 2",
     [("lin = 2.0 * a * L + b", "lin = a * L + b")]),
    ("planner.py", "rounded up to the page multiple",
     [("units = math.floor(xs / page_size * (1.0 + 1e-9))", "units = math.ceil(xs / page_size)")]),
    ("planner.py", "smoothing drops the base term",
     [("xs = smooth_factor * x + (1.0 - smooth_factor) * base_chunk_size", "xs = smooth_factor * x")]),
    ("planner.py", "model-length cap ignores the prefix",
     [("aligned = min(aligned, max_model_len - L)", "aligned = min(aligned, max_model_len)")]),
    ("planner.py", "two-variable feature C*C instead of C*(C+H)",
     [("rows.append([float(np.sum(cs * (cs + hs))), float(np.sum(cs + hs)), float(len(cs))])\n    X = np.asarray(rows)",
       "rows.append([float(np.sum(cs * cs)), float(np.sum(cs + hs)), float(len(cs))])\n    X = np.asarray(rows)")]),
    ("planner.py", "calibrated root with 2aH",
     [("lin = a * H + b", "lin = 2.0 * a * H + b")]),
    ("planner.py", "online refit never forgets old batches",
     [("X = np.asarray(self.rows[-self.window:])", "X = np.asarray(self.rows)"),
      ("t = np.asarray(self.times[-self.window:])", "t = np.asarray(self.times)")]),
    ("scheduler.py", "a chunk not limited by what is left of its prompt",
     [("c = min(rem, budget)", "c = budget")]),
    ("scheduler.py", "progressive caps: always the last size",
     [("c = min(c, self.caps[min(r.chunks, len(self.caps) - 1)])", "c = min(c, self.caps[-1])")]),
    ("scheduler.py", "tile alignment of a prompt's last chunk too",
     [("if c < rem and self.tile > 0:", "if self.tile > 0 and c > self.tile:")]),
    ("scheduler.py", "decode rows take no budget",
     [("                    batch.append((r, 1, True))\n                    budget -= 1",
       "                    batch.append((r, 1, True))")]),
    ("scheduler.py", "slots one past their position",
     [("out[\"slot_mapping\"] += [r.pages[p // self.P] * self.P + p % self.P for p in range(s0, s0 + c)]",
       "out[\"slot_mapping\"] += [r.pages[p // self.P] * self.P + (p + 1) % self.P for p in range(s0, s0 + c)]")]),
    ("scheduler.py", "finished requests keep their pages",
     [("                self.free.extend(r.pages)\n", "")]),
    ("scheduler.py", "new pages taken from the back of the free list",
     [("r.pages.append(self.free.popleft())", "r.pages.append(self.free.pop())")]),
]

PY_PINS = [getattr(py_pins, n) for n in sorted(dir(py_pins))
           if n.startswith("test_") and n != "test_online_controller_matches_oracle"]
SCHED_PINS = [getattr(sched_pins, n) for n in sorted(dir(sched_pins))
              if n.startswith("test_") and "library" not in n]
PY_NAMES = {"scheduler.py": ["Scheduler"],
            "split.py": ["simple_split", "balanced_split"],
            "planner.py": ["latency_quadratic", "target_latency", "solve_chunk", "postprocess", "plan_chunks",
                           "fit_quadratic", "fit_two_var", "solve_chunk_two_var", "OnlineCalibrator"]}


def _py_failing_pins(module, text, tmp_path, tag):
    path = tmp_path / f"{tag}.py"
    path.write_text(text)
    spec = importlib.util.spec_from_file_location(f"oracle_slip_{tag}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    saved = {n: getattr(oracle, n) for n in PY_NAMES[module]}
    failed = []
    try:
        for n in PY_NAMES[module]:
            setattr(oracle, n, getattr(mod, n))
        with np.errstate(all="ignore"):
            for pin in (SCHED_PINS if module == "scheduler.py" else PY_PINS):
                try:
                    pin()
                except (Exception, pytest.fail.Exception):
                    failed.append(pin.__name__)
    finally:
        for n, f in saved.items():
            setattr(oracle, n, f)
    return failed


def _py_source(module):
    with open(os.path.join(os.path.dirname(oracle.__file__), module)) as f:
        return f.read()


@pytest.mark.parametrize("module", sorted(PY_NAMES))
def test_unchanged_python_oracle_passes_every_pin(module, tmp_path):
    assert len(PY_PINS) >= 10 and len(SCHED_PINS) >= 2
    assert _py_failing_pins(module, _py_source(module), tmp_path, "control_" + module[:-3]) == []


@pytest.mark.parametrize("k", range(len(PY_SLIPS)), ids=[s[1] for s in PY_SLIPS])
def test_a_planted_python_slip_fails_some_pin(tmp_path, k):
    module, name, edits = PY_SLIPS[k]
    text = _py_source(module)
    for old, new in edits:
        assert text.count(old) == 1, f"{name}: the text to change must occur once"
        text = text.replace(old, new)
    failed = _py_failing_pins(module, text, tmp_path, f"slip{k}")
    assert failed, f"no pin caught the slip '{name}'"
