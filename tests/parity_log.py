"""Collects the parity numbers the GPU tests measure; written as JSON to
$WAN_PARITY_REPORT at exit when that variable is set."""

import atexit
import json
import os

_ROWS = []


def record(case: str, max_abs: float, psnr_db=None, **extra):
    _ROWS.append({"case": case, "max_abs": max_abs, "psnr_db": psnr_db, **extra})


@atexit.register
def _dump():
    path = os.environ.get("WAN_PARITY_REPORT")
    if path and _ROWS:
        old = []
        if os.path.exists(path):
            with open(path) as f:
                old = json.load(f)
        with open(path, "w") as f:
            json.dump(old + _ROWS, f, indent=1)
