"""Readers for the text fixtures in this folder (each cites its source page)."""
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))


def _read(name):
    out = {"rows": []}
    with open(os.path.join(_HERE, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key in ("row", "mask_row"):
                out["rows"].append([int(x) for x in vals])
            elif key == "block_mask_row":
                out.setdefault("block_rows", []).append([int(x) for x in vals])
            elif len(vals) == 1:
                out[key] = int(vals[0])
            else:
                out[key] = [int(x) for x in vals]
    return out


def bsr_3x3_example():
    d = _read("bsr_3x3_example.txt")
    d["mask"] = np.array(d.pop("rows"), dtype=bool)
    return d


def causal_bottom_right():
    d = _read("causal_bottom_right.txt")
    d["mask"] = np.array(d.pop("rows"), dtype=bool)
    return d


def varbsr_example():
    d = _read("varbsr_example.txt")
    d["mask"] = np.array(d.pop("rows"), dtype=bool)
    d["block_mask_map"] = np.array(d.pop("block_rows"), dtype=bool)[None]
    d["block_row_sz"] = np.array(d["block_row_sz"], dtype=np.int32)[None]
    d["block_col_sz"] = np.array(d["block_col_sz"], dtype=np.int32)[None]
    return d
