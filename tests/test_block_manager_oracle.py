"""The reference block manager against its pins, and planted mistakes in it
each caught by at least one pin (CPU only)."""
import importlib.util
import os
import sys

import pytest

from oracle import block_manager as bm
from tests import block_manager_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=[p.__name__ for p in pins.ALL_PINS])
def test_pin(pin):
    pin(bm)


# (name, original text, replacement); only the first occurrence is replaced
MUTANTS = [
    ("fork_without_reference", "            self.ref[b] += 1\n", "            pass\n"),
    ("copy_when_unshared", "        elif self.ref[table[logical]] > 1:", "        elif self.ref[table[logical]] > 0:"),
    ("never_copy", "        elif self.ref[table[logical]] > 1:", "        elif self.ref[table[logical]] > 99:"),
    ("free_ignores_sharing", "            if self.ref[b] == 0:\n                self.free.append(b)",
     "            self.free.append(b)"),
    ("lifo_pool", "                blk = self.free.popleft()\n                self.ref[blk] = 1\n                table.append(blk)",
     "                blk = self.free.pop()\n                self.ref[blk] = 1\n                table.append(blk)"),
    ("slot_offset_from_block", "            slots.append(table[logical] * bs + offset)",
     "            slots.append(table[logical] * bs + logical % bs)"),
    ("copy_keeps_old_reference", "                self.ref[old] -= 1\n", "                pass\n"),
    ("need_ignores_copy", "            need += 1\n        first_new", "            need += 0\n        first_new"),
]


def _load_mutant(tmp_path, name, old, new):
    with open(bm.__file__) as f:
        src = f.read()
    assert old in src, name
    path = tmp_path / f"bm_{name}.py"
    path.write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location(f"bm_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    mod = _load_mutant(tmp_path, name, old, new)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mod)
        except Exception:  # any failure of a pin counts
            caught.append(pin.__name__)
    assert caught, f"mutant {name} survived every pin"
