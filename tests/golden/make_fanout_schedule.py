"""Writes the oracle-derived rows of fanout_schedule.json (prints them; the
first row of that file is worked by hand).  Calls only the oracle."""
import json
import os
import sys

sys.path.insert(0, os.path.join(os.path.dirname(__file__), "..", ".."))
import oracle  # noqa: E402

for K, B, a, r in [(4, 20, 0.6, 0.5), (6, 40, 0.7, 1.0), (8, 128, 0.9, 2.0)]:
    F = [int(x) for x in oracle.fanout_schedule(K, B, a, r)]
    print(json.dumps({"K": K, "budget": B, "a": a, "r": r, "F": F}))
