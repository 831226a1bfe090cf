"""Readers for the text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                key, _, val = line.partition(":")
                yield key.strip(), val.split()


def hand_cases():
    cases, cur = [], None
    for key, val in _lines("conv_hand_cases.txt"):
        if key == "case":
            cur = {"name": val[0]}
            cases.append(cur)
        elif key == "shape":
            cur["shape"] = [int(v) for v in val]
        else:
            cur[key] = np.array([float(v) for v in val], dtype=np.float64)
    return cases


def tuning_log():
    log = {"trials": [], "splits": [], "knobs": []}
    for key, val in _lines("tvm_tuning_log_resnet_last.txt"):
        if key == "trial":
            log["trials"].append((int(val[0]), float(val[1]), float(val[2])))
        elif key == "retimed":
            log["retimed"] = float(val[0])
        elif key == "split":
            log["splits"].append((val[0], int(val[1]), int(val[2]), int(val[3])))
        elif key == "knob":
            log["knobs"].append((val[0], int(val[1])))
        elif key == "space_total":
            log["space_total"] = int(val[0])
    return log
