"""Readers for the text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def hand_steps():
    """Cases of golden/hand_steps.txt as dicts: name, shape (nx, ny, nz), lam,
    steps, b (nz, ny, nx) float64, expect = list of (field, a, x, y, z, v)."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "hand_steps.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            key = tok[0]
            if key == "case":
                cur = {"name": tok[1], "b_entries": [], "expect": []}
            elif key == "shape":
                cur["shape"] = tuple(int(t) for t in tok[1:4])
            elif key == "lam":
                cur["lam"] = float(tok[1])
            elif key == "steps":
                cur["steps"] = int(tok[1])
            elif key == "b":
                cur["b_entries"].append((int(tok[1]), int(tok[2]), int(tok[3]), float(tok[4])))
            elif key == "expect":
                cur["expect"].append((tok[1], int(tok[2]), int(tok[3]), int(tok[4]), int(tok[5]),
                                      float(tok[6])))
            elif key == "end":
                nx, ny, nz = cur["shape"]
                b = np.zeros((nz, ny, nx))
                for x, y, z, v in cur["b_entries"]:
                    b[z, y, x] = v
                cur["b"] = b
                cases.append(cur)
                cur = None
            else:
                raise ValueError("bad line in hand_steps.txt: %r" % line)
    return cases


def expected_fields(case):
    """Dense expected p, r (3, nz, ny, nx) and z (nz, ny, nx) of a hand case."""
    nx, ny, nz = case["shape"]
    out = {"p": np.zeros((3, nz, ny, nx)), "r": np.zeros((3, nz, ny, nx)),
           "z": np.zeros((1, nz, ny, nx))}
    for field, a, x, y, z, v in case["expect"]:
        out[field][a, z, y, x] = v
    out["z"] = out["z"][0]
    return out


def traffic_model():
    """(steps, ncu_rows, padded) from golden/traffic_model.txt."""
    steps, ncu, padded = [], [], []
    with open(os.path.join(GOLDEN, "traffic_model.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "step":
                steps.append((tok[1], int(tok[2]), int(tok[3]), float(tok[4]), float(tok[5])))
            elif tok[0] == "ncu":
                ncu.append((tok[1], float(tok[2]), float(tok[3]), float(tok[4]), float(tok[5])))
            elif tok[0] == "padded_volume":
                padded.append((int(tok[1]), float(tok[2])))
    return steps, ncu, padded
