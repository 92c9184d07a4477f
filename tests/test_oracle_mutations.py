"""Plant plausible mistakes in copies of the oracle (CPU only) and check that
the pins in test_oracle_pins.py catch every one of them.

Each mutation edits one expression of ``oracle/pa_oracle.c`` in a temporary
copy, compiles it, swaps it in for the real oracle and runs the pins.  The
real oracle is never modified.
"""
import inspect
import os

import pytest

import oracle
import test_oracle_pins as pins

MUTATIONS = {
    "scale dropped": ("scores[j] = dot * J->scale;", "scores[j] = dot;"),
    "query position off by one": ("const int64_t t = J->q_pos0[s] + (i - J->q_start[s]);",
                                  "const int64_t t = J->q_pos0[s] + (i - J->q_start[s]) - 1;"),
    "GQA map interleaved": ("const int hk = h / group;", "const int hk = h % J->Hkv;"),
    "softmax not normalised": ("const double w = scores[j] / denom;",
                               "const double w = scores[j];"),
    "keys used as values": ("const double *vj = J->v + ", "const double *vj = J->k + "),
    "max added instead of subtracted": ("scores[j] = exp(scores[j] - mx);",
                                        "scores[j] = exp(scores[j] + mx);"),
    "slot without block size": ("(int64_t)table[j / bs] * bs + j % bs",
                                "(int64_t)table[j / bs] + j % bs"),
    "K and V sources swapped": ("memcpy(k_cache + dst, k_new + src, row);",
                                "memcpy(k_cache + dst, v_new + src, row);"),
    "copy-on-write copies K only": (
        "memmove(v_cache + (size_t)dst * blk, v_cache + (size_t)src * blk, blk);", ""),
    "dot product over half the dims": ("for (int c = 0; c < d; ++c) dot += qi[c] * kj[c];",
                                       "for (int c = 0; c < d / 2; ++c) dot += qi[c] * kj[c];"),
    "GQA group taken as the KV head count": ("const int group = J->Hq / J->Hkv;",
                                             "const int group = J->Hkv;"),
    "store ignores the KV head": (
        "const size_t dst = (size_t)(((blk * Hkv + h) * bs + off)) * row;",
        "const size_t dst = (size_t)(((blk * Hkv) * bs + off)) * row;"),
    "copy direction reversed": (
        "memmove(k_cache + (size_t)dst * blk, k_cache + (size_t)src * blk, blk);",
        "memmove(k_cache + (size_t)src * blk, k_cache + (size_t)dst * blk, blk);"),
    "slot offset from the block index": ("(int64_t)table[j / bs] * bs + j % bs",
                                         "(int64_t)table[j / bs] * bs + j / bs"),
}


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argnames, values = params[0].args[0], params[0].args[1]
            for val in values:
                out.append((f"{name}{val}", fn, dict(zip(argnames.split(","), val))))
        else:
            out.append((name, fn, {}))
    return out


@pytest.mark.parametrize("label", list(MUTATIONS))
def test_pins_catch_planted_mistake(label, tmp_path, monkeypatch):
    old, new = MUTATIONS[label]
    with open(os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mutated = tmp_path / "pa_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    so = oracle.compile_source(str(mutated), str(tmp_path / "libmutant.so"))
    monkeypatch.setattr(oracle, "_lib", oracle.load(so))
    caught = []
    for name, fn, kwargs in _pin_functions():
        try:
            fn(**kwargs)
        except (AssertionError, ValueError, pytest.fail.Exception):
            caught.append(name)
    assert caught, f"no pin caught the planted mistake '{label}'"
