"""Write exact rational fixtures for the token oracle.

Run from the repository root:  python tests/golden/make_golden.py

It calls only ``oracle.brute`` (the exact unrolled-product form of the
recurrence, evaluated in ``fractions.Fraction``); no value comes from the CUDA
library. Inputs are small integers / dyadic rationals, base-2 gates with
integer logs, so every stored number is exact. Stored as "p/q" strings.
"""
import json
import os
import sys
from fractions import Fraction

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
from oracle import brute  # noqa: E402

F = Fraction


def case_scalar():
    # one head, T=4, K=3, V=2, scalar base-2 gate
    q = [[F(1), F(0), F(1, 2)], [F(0), F(1), F(-1)], [F(1, 4), F(1), F(0)], [F(1), F(1), F(1)]]
    k = [[F(1, 2), F(1, 2), F(0)], [F(0), F(1), F(0)], [F(1, 2), F(0), F(-1, 2)], [F(1, 4), F(1, 2), F(1, 4)]]
    v = [[F(1), F(-2)], [F(3), F(1)], [F(-1), F(1, 2)], [F(2), F(0)]]
    g = [0, -1, -2, -1]
    beta = [F(1, 2), F(1), F(3, 4), F(1, 4)]
    h0 = [[F(1), F(0)], [F(0), F(1)], [F(1, 2), F(-1, 2)]]
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, per_key=False, scale=F(1, 2))


def case_per_key():
    c = case_scalar()
    c["g"] = [[0, -1, -2], [-1, 0, 0], [-2, -1, -1], [0, 0, -3]]
    c["per_key"] = True
    return c


def enc(x):
    if isinstance(x, list):
        return [enc(y) for y in x]
    x = Fraction(x)
    return f"{x.numerator}/{x.denominator}"


def main():
    out = {}
    for name, c in (("scalar_gate_exp2", case_scalar()), ("per_key_gate_exp2", case_per_key())):
        o, S = brute.states(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], c["scale"],
                            c["per_key"])
        M = brute.transfer(c["k"], c["g"], c["beta"], c["per_key"])
        out[name] = {key: enc(val) if key not in ("per_key",) else val for key, val in c.items()}
        out[name].update(o=enc(o), ht=enc(S), M=enc(M))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "exact_tiny.json")
    with open(path, "w") as fh:
        json.dump({"source": "oracle.brute exact unrolled products (make_golden.py)",
                   "cases": out}, fh, separators=(",", ":"))
    print("wrote", path)


if __name__ == "__main__":
    main()
