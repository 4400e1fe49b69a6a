"""Loads the hand-worked delay-and-sum examples of tests/golden/ and builds
their inputs.  The expected values there are closed forms derived by hand from
the definition of the sum (their derivation is in the fixture), not outputs of
the oracle or of the CUDA path."""
from __future__ import annotations

import json
import os

import numpy as np

FIXTURE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "das_worked_examples.json")

# the record formulas the fixture states, as code
_RECORDS = {
    "s[b,q,m,k] = (b + 1) * (1 + k + 10 m + 100 q)":
        lambda b, q, m, k: (b + 1) * (1 + k + 10 * m + 100 * q),
    "s[b,q,m,k] = (b + 1) * ((1 + k + 10 m) + i 2 k)":
        lambda b, q, m, k: (b + 1) * ((1 + k + 10 * m) + 2j * k),
}


def examples():
    with open(FIXTURE) as f:
        return json.load(f)["examples"]


def inputs(ex):
    """rf (B x Q x M x K), tau_tx and w_tx (Q x N) float32, rx (M x 3)."""
    B, Q, M, K = ex["B"], ex["Q"], ex["M"], ex["K"]
    b, q, m, k = np.meshgrid(np.arange(B), np.arange(Q), np.arange(M), np.arange(K), indexing="ij")
    rf = _RECORDS[ex["rf"]](b, q, m, k)
    rf = rf.astype(np.complex64 if ex["dtype"] == "c64" else np.float32)
    tau = np.asarray(ex["tau_tx"], dtype=np.float32)
    w = np.asarray(ex["w_tx"], dtype=np.float32)
    rx = np.asarray(ex["rx"], dtype=np.float32)
    return rf, tau, w, rx


def expected(ex):
    """y[b, n] = (b + 1) * y_unit[n] (B x N, complex128)."""
    unit = np.array([re + 1j * im for re, im in ex["y_unit"]])
    return (np.arange(ex["B"]) + 1)[:, None] * unit[None, :]
