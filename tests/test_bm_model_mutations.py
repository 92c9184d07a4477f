"""Plant plausible mistakes in copies of the reference block-manager model
(oracle/bm_model.py) and check that the pins in test_bm_model.py catch every
one of them.

Each mutation edits one statement of the model's source in memory, loads the
edited text as a separate module and runs every pin against it.  The real
model is never modified.
"""
import importlib.util
import inspect
import os
import sys

import pytest

import test_bm_model as pins
from conftest import ROOT

MUTATIONS = {
    "fork does not count the new holder": ("            self.ref[b] += 1\n",
                                           "            pass\n"),
    "sole holder copies on write": ("elif self.ref[bl[-1]] > 1:", "elif self.ref[bl[-1]] >= 1:"),
    "copy source keeps its reference": ("            self._release(src)\n", ""),
    "slot without block size": ("return bl[-1] * self.bs + L % self.bs, src, dst",
                                "return bl[-1] + L % self.bs, src, dst"),
    "copy left out of the budget": ("            need += 1\n", "            pass\n"),
    "freed blocks queued last": ("            self.free.append(b)\n",
                                 "            self.free.insert(0, b)\n"),
    "shuffle draws from [0, i)": ("j = r % (i + 1)", "j = r % i"),
    "splitmix shift constant": ("z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64",
                                "z = ((z ^ (z >> 31)) * 0xBF58476D1CE4E5B9) & _M64"),
    "fork aliases the parent's table": ("self.blocks[child] = list(self.blocks[parent])",
                                        "self.blocks[child] = self.blocks[parent]"),
    "new block one token late": ("        if L % self.bs == 0:\n            bl.append(self._take())",
                                 "        if L % self.bs == 1:\n            bl.append(self._take())"),
}


def _load_mutant(src, name):
    spec = importlib.util.spec_from_loader(name, loader=None)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod
    try:
        exec(compile(src, f"<{name}>", "exec"), mod.__dict__)
    finally:
        sys.modules.pop(name, None)
    return mod


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if name.startswith("test_"):
            out.append((name, fn))
    return out


def test_unmutated_model_passes_every_pin():
    for _, fn in _pin_functions():
        fn()


@pytest.mark.parametrize("label", list(MUTATIONS))
def test_pins_catch_planted_mistake(label, monkeypatch):
    old, new = MUTATIONS[label]
    with open(os.path.join(ROOT, "oracle", "bm_model.py")) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mutant = _load_mutant(src.replace(old, new), "bm_model_mutant")
    for attr in ("BlockManagerModel", "OutOfBlocks", "initial_order", "splitmix64"):
        monkeypatch.setattr(pins, attr, getattr(mutant, attr))
    caught = []
    for name, fn in _pin_functions():
        try:
            fn()
        except (Exception, pytest.fail.Exception):  # an assertion, or the mutant breaking
            caught.append(name)
    assert caught, f"no pin caught the planted mistake '{label}'"
