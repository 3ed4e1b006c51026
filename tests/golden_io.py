"""Readers for the hand-derived fixtures under tests/golden/."""
import os
import re

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_verify_cases(name="verify_cases.txt"):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                m = re.match(r"case (\S+) B=(\d+) V=(\d+)", line)
                cur = {"name": m.group(1), "B": int(m.group(2)), "V": int(m.group(3)), "rows": []}
                cases.append(cur)
            elif line.startswith("row "):
                vals = line.split(":", 1)[1].split()
                cur["rows"].append([float(v) for v in vals])
            elif line.startswith("drafted:"):
                cur["drafted"] = [int(v) for v in line.split(":", 1)[1].split()]
            elif line.startswith("expect:"):
                kv = dict(p.split("=") for p in line.split(":", 1)[1].split())
                cur["tau"] = int(kv["tau"])
                cur["committed"] = [int(v) for v in kv["committed"].split(",")]
                cur["last"] = int(kv["last"])
    for c in cases:
        c["logits"] = np.array(c["rows"], dtype=np.float32)
        assert c["logits"].shape == (c["B"], c["V"]), c["name"]
        assert len(c["drafted"]) == c["B"] - 1, c["name"]
    return cases


def load_sampling_cases(name="sampling_cases.txt"):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                m = re.match(r"case (\S+) B=(\d+) V=(\d+) T=([0-9.]+)", line)
                cur = {"name": m.group(1), "B": int(m.group(2)), "V": int(m.group(3)), "T": float(m.group(4)),
                       "rows": []}
                cases.append(cur)
            elif line.startswith("row "):
                cur["rows"].append([float(v) for v in line.split(":", 1)[1].split()])
            elif line.startswith("drafted:"):
                cur["drafted"] = [int(v) for v in line.split(":", 1)[1].split()]
            elif line.startswith("uniforms:"):
                cur["uniforms"] = [float(v) for v in line.split(":", 1)[1].split()]
            elif line.startswith("expect:"):
                kv = dict(p.split("=") for p in line.split(":", 1)[1].split())
                cur["tau"] = int(kv["tau"])
                cur["committed"] = [int(v) for v in kv["committed"].split(",")]
                cur["last"] = int(kv["last"])
    for c in cases:
        c["logits"] = np.array(c["rows"], dtype=np.float32)
        assert c["logits"].shape == (c["B"], c["V"]), c["name"]
        assert len(c["drafted"]) == c["B"] - 1 and len(c["uniforms"]) == c["B"], c["name"]
    return cases
