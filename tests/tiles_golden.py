"""Reader for tests/golden/tiles_small.txt (hand-worked tile schedules)."""
from pathlib import Path

import numpy as np

GOLDEN = Path(__file__).resolve().parent / "golden" / "tiles_small.txt"


def load_cases():
    cases, cur = [], None
    for raw in GOLDEN.read_text().splitlines():
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0], "fwd": [], "bwd": []}
        elif key == "end":
            for d in ("fwd", "bwd"):
                cur[d] = np.asarray(cur[d], dtype=np.int32).reshape(-1, 4)
            cases.append(cur)
            cur = None
        elif key in ("fwd", "bwd"):
            cur[key].append([int(x) for x in vals])
        elif key in ("q_lengths", "kv_lengths", "fwd_cta_ptr", "bwd_cta_ptr"):
            cur[key] = np.asarray([int(x) for x in vals], dtype=np.int32)
        else:
            cur[key] = int(vals[0])
    return cases
