"""The oracle still reproduces the stored fixture (same answer on every host)."""
import json
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def load_fixture():
    with open(os.path.join(HERE, "golden", "oracle_small.json")) as f:
        doc = json.load(f)
    s = doc["shape"]
    shp = (s["B"], s["N"], s["H"], s["D"])

    def arr(key):
        return np.array([int(x, 16) for x in doc[key].split()], dtype=np.uint16).reshape(shp)
    O = np.array([float.fromhex(x) for x in doc["O"]]).reshape(shp)
    L = np.array([float.fromhex(x) for x in doc["LSE"]]).reshape(s["B"], s["H"], s["N"])
    return s, arr("q"), arr("k"), arr("v"), O, L


def test_oracle_reproduces_fixture():
    s, q, k, v, O, L = load_fixture()
    O2, L2 = oracle.attn(q, k, v, key_valid_len=s["key_valid_len"], scale=s["scale"])
    np.testing.assert_allclose(O2, O, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L2, L, rtol=0, atol=1e-13)
