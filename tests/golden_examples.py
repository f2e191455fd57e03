"""Reader for tests/golden/pack_worked_examples.txt (hand-worked examples)."""
from __future__ import annotations

import os
from dataclasses import dataclass, field

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "pack_worked_examples.txt")


def _halves(tokens):
    return np.array([np.float16(float(t)) for t in tokens], dtype=np.float16)


@dataclass
class Example:
    name: str
    N: int = 0
    M: int = 0
    W: list = field(default_factory=list)
    mask: list = field(default_factory=list)
    values: list = field(default_factory=list)
    masks: list = field(default_factory=list)
    bad: int = 0
    cases: list = field(default_factory=list)  # (x fp16 [K], y list, s list)

    @property
    def W_arr(self):
        return np.stack(self.W)

    @property
    def mask_arr(self):
        return np.array(self.mask, dtype=np.uint8)

    @property
    def values_arr(self):
        return np.stack(self.values)

    @property
    def masks_arr(self):
        return np.array(self.masks, dtype=np.uint32)


def load_examples(path: str = GOLDEN):
    examples, cur, pending_x, pending_y = [], None, None, None
    with open(path) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            if key == "example":
                cur = Example(rest[0])
            elif key == "end":
                examples.append(cur)
                cur = None
            elif key in ("N", "M", "bad"):
                setattr(cur, key, int(rest[0]))
            elif key == "W":
                cur.W.append(_halves(rest))
            elif key == "mask":
                cur.mask.append([int(t) for t in rest])
            elif key == "values":
                cur.values.append(_halves(rest))
            elif key == "masks":
                cur.masks.append([int(t, 16) for t in rest])
            elif key == "x":
                pending_x = _halves(rest)
            elif key == "y":
                pending_y = [float(t) for t in rest]
            elif key == "s":
                cur.cases.append((pending_x, pending_y, [float(t) for t in rest]))
                pending_x = pending_y = None
            else:
                raise ValueError("unknown golden key %r" % key)
    return examples
