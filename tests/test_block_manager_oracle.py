"""The reference block manager against its pins, and plausible mistakes
planted in copies of it caught by them (no GPU)."""
import importlib.util
import os

import pytest

import block_manager_pins as P
from oracle import block_manager as M

SRC = M.__file__


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(M)


MUTANTS = [
    ("cow_keeps_reference", "                    self.ref[last] -= 1\n", ""),
    ("cow_without_remap", "                    table[pos // bs] = new\n", ""),
    ("fork_without_reference", "            self.ref[b] += 1\n", "            pass\n"),
    ("no_new_block_when_full", "            if pos % bs == 0:", "            if pos % bs == 0 and not table:"),
    ("highest_free_block", "        b = min(free)", "        b = max(free)"),
    ("free_keeps_reference", "            self.ref[b] -= 1\n        del self.lengths[seq]",
     "            pass\n        del self.lengths[seq]"),
    ("slot_offset_logical", "    return table[position // block_size] * block_size + position % block_size",
     "    return table[position // block_size] * block_size + position // block_size"),
    ("append_not_atomic", "        if self.blocks_needed(seq, n) > self.num_free():\n            raise OutOfBlocks()\n", ""),
    ("batch_no_rollback", "            self.ref, self.tables, self.lengths = saved\n", ""),
    ("batch_rollback_keeps_tables",
     "            self.ref, self.tables, self.lengths = saved\n",
     "            self.ref, self.lengths = saved[0], saved[2]\n"),
    ("batch_repeat_allowed",
     "        if len(set(seqs)) != len(seqs) or any(s not in self.tables for s in seqs):",
     "        if any(s not in self.tables for s in seqs):"),
    ("batch_table_check_late",
     "            if (self.lengths[s] + n + bs - 1) // bs > self.max_blocks_per_seq:\n                raise TableFull()\n",
     ""),
    ("batch_reversed_order",
     "            for s, n in zip(seqs, counts):\n                sl, pr = self.append_tokens(s, n)",
     "            for s, n in reversed(list(zip(seqs, counts))):\n                sl, pr = self.append_tokens(s, n)"),
    ("build_batch_pads_zero",
     "[pad_block] * (max_blocks - len(self.tables[s]))",
     "[0] * (max_blocks - len(self.tables[s]))"),
    ("build_batch_length_in_blocks",
     "            lens.append(self.lengths[s])",
     "            lens.append(len(self.tables[s]) * self.block_size)"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, name
    path = tmp_path / f"bm_{name}.py"
    path.write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location(f"bm_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(mod)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
