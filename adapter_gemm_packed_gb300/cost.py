"""The measured step-time table behind mlora_cost_estimate (T(H, 1) of the planner's cost model).

``cost_table_gb300.json`` holds steps of this library measured on one GB300 by
``python bench.py --calibrate``: for each layer shape and pack size, the forward + backward +
AdamW time of a pack of 1024-token jobs.  :func:`estimate` asks the C ABI for a plan's step time
from it; the interpolation itself is the library's (see mlora_cost_estimate in include/mlora.h).
"""
from __future__ import annotations

import json
import os

from . import _mlora as M

TABLE_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "cost_table_gb300.json")


def load_table(path: str = TABLE_PATH) -> list[tuple]:
    """[(d_in, d_out, n_tokens, lora_work, step_ms), ...] from the measured table."""
    with open(path) as f:
        rec = json.load(f)
    return [(p["d_in"], p["d_out"], p["n_tokens"], p["lora_work"], p["step_ms"]) for p in rec["points"]]


def estimate(plan, table=None) -> tuple[float, int]:
    """(step ms, basis) of a plan from the measured table (basis as in mlora_cost_estimate)."""
    return M.mlora_cost_estimate(plan, load_table() if table is None else table)
