"""Reader for the hand-derived fixtures in tests/golden/."""
import glob
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _hex(vals, dtype):
    return np.array([int(v, 16) for v in vals], dtype=dtype)


def load(path):
    plan, ranks, cur = {}, [], None
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "rank":
                cur = {"rank": int(vals[0])}
                ranks.append(cur)
            elif cur is None:
                if key in ("n", "ranks", "block", "cold"):
                    plan[key] = int(vals[0])
                elif key == "w":
                    plan[key] = _hex(vals, np.uint16)
                else:
                    plan[key] = _hex(vals, np.uint8)
            else:
                if key == "desc":
                    cur[key] = tuple(int(v) for v in vals)
                elif key == "flags":
                    cur[key] = np.array([int(v) for v in vals], dtype=np.uint8)
                else:
                    cur[key] = _hex(vals, np.uint8)
    plan["rank_data"] = ranks
    return plan


def all_fixtures():
    return sorted(glob.glob(os.path.join(GOLDEN_DIR, "*.txt")))
