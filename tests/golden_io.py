"""Readers of the text fixtures under tests/golden/ (no arithmetic of the method)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str):
    """Non-comment lines of a golden fixture, split on whitespace."""
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def load_hash_worked():
    """hash_worked.txt: (primes, offsets, {table: mult [nb][4]}, [(table, window, rows)])."""
    as_int = lambda x: int(x, 0)
    primes, offsets, mult, cases = {}, {}, {}, []
    for r in read_golden("hash_worked.txt"):
        if r[0] == "prime":
            primes[int(r[1])], offsets[int(r[1])] = as_int(r[2]), as_int(r[3])
        elif r[0] == "mult":
            mult.setdefault(r[1], {})[int(r[2])] = [as_int(x) for x in r[3:7]]
        elif r[0] == "case":
            cases.append((r[1], [as_int(x) for x in r[2:6]], [as_int(x) for x in r[6:]]))
    nb = len(primes)
    tables = {k: np.array([v[b] for b in range(nb)], np.uint64) for k, v in mult.items()}
    return (np.array([primes[b] for b in range(nb)], np.uint64),
            np.array([offsets[b] for b in range(nb)], np.uint64), tables, cases)
