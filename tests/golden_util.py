"""Helpers that turn the hand-derived cases in tests/golden/closed_form_cases.json into tensors."""
import json
import math
import os

import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_form_cases.json")

_SAFE = {"exp": math.exp, "sqrt": math.sqrt, "log": math.log, "__builtins__": {}}


def load():
    with open(GOLDEN) as f:
        return json.load(f)


def ev(expr: str) -> float:
    """Evaluate a closed-form expression from the fixture (exp, sqrt, log and arithmetic only)."""
    return float(eval(expr, _SAFE))


def _key(s):
    return tuple(int(x) for x in s.split(","))


def sparse_tensor(shape, spec):
    """bf16 tensor of ``shape``; spec maps 'i,j,k' (all but the last dim) -> [[dim, value], ...]."""
    t = torch.zeros(shape, dtype=torch.float32)
    for key, entries in spec.items():
        ix = _key(key)
        for dim, val in entries:
            t[ix + (int(dim),)] = float(val)
    return t.to(torch.bfloat16)


def focal_case_tensors(case):
    B, Hq, Hkv, Mq, T, d = (case[n] for n in ("B", "Hq", "Hkv", "Mq", "T", "d"))
    q = sparse_tensor((B, Hq, Mq, d), case["q"])
    k = sparse_tensor((B, Hkv, T, d), case["k"])
    v = sparse_tensor((B, Hkv, T, d), case["v"])
    length = torch.tensor(case["len"], dtype=torch.int32)
    return q, k, v, length
