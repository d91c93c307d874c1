"""Writes tests/golden/tiny_case.txt from the fp64 oracle alone.

The case is small enough to read by eye: one sequence, one head, T = 8,
dk = dv = 2, hand-picked inputs.  Re-run only when the oracle's arithmetic is
deliberately changed; the commit that does so names the passage that
justifies it.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def case():
    T, dk, dv = 8, 2, 2
    ang = np.linspace(0.0, 1.4, T)
    k = np.stack([np.cos(ang), np.sin(ang)], -1)
    q = np.stack([np.cos(ang + 0.3), np.sin(ang + 0.3)], -1)
    v = np.stack([np.linspace(-1, 1, T), np.linspace(2, 0, T)], -1)
    theta = np.stack([np.linspace(-3, 3, T), np.linspace(2, -2, T)], -1)
    beta = np.linspace(0.2, 0.9, T)
    S0 = np.array([[0.5, -0.25], [0.125, 1.0]])
    shp = lambda a, d: a.reshape(1, T, 1, d)
    return (shp(q, dk), shp(k, dk), shp(v, dv), shp(theta, dk), beta.reshape(1, T, 1),
            S0.reshape(1, 1, dk, dv))


def main():
    q, k, v, th, be, S0 = case()
    o, S = oracle.fwd(q, k, v, th, be, -5.0, S0, nthreads=1)
    with open(os.path.join(HERE, "tiny_case.txt"), "w") as f:
        f.write("# written by tests/golden/make_golden.py from the fp64 oracle (g_min = -5)\n")
        f.write("# o[t, j] for t = 0..7, j = 0..1\n")
        for t in range(o.shape[1]):
            f.write("o %d %.17e %.17e\n" % (t, o[0, t, 0, 0], o[0, t, 0, 1]))
        f.write("# final state S[i, j]\n")
        for i in range(2):
            f.write("S %d %.17e %.17e\n" % (i, S[0, 0, i, 0], S[0, 0, i, 1]))


if __name__ == "__main__":
    main()
