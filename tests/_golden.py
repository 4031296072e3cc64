"""Readers for the hand-derived fixtures in tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [c.strip() for c in line.split("|")]


def codes_from_rule(rule: str, K: int) -> np.ndarray:
    """One row of codes from a rule string (see pack_vectors.txt)."""
    v = np.arange(K)
    if rule.startswith("mod"):
        return (v % int(rule[3:])).astype(np.uint8)
    if rule == "zero":
        return np.zeros(K, np.uint8)
    if rule.startswith("all:"):
        return np.full(K, int(rule[4:]), np.uint8)
    if rule.startswith("set:"):
        out = np.zeros(K, np.uint8)
        for item in rule[4:].split(","):
            k, c = item.split("=")
            out[int(k)] = int(c)
        return out
    if rule.startswith("groups:"):
        vals = [int(c) for c in rule[7:].split(",")]
        assert len(vals) == K // 64
        return np.repeat(np.array(vals, np.uint8), 64)
    raise ValueError(rule)


def pack_vectors(name_of_file="pack_vectors.txt"):
    for name, bits, K, rule, words in _lines(name_of_file):
        K = int(K)
        yield (name, int(bits), K, codes_from_rule(rule, K),
               np.array([int(w, 16) for w in words.split()], dtype=np.uint32))


def x_from_rule(rule: str, K: int) -> np.ndarray:
    if rule == "ones":
        return np.ones(K)
    if rule == "alt":
        return np.where(np.arange(K) % 2 == 0, 1.0, -1.0)
    if rule.startswith("unit:"):
        x = np.zeros(K)
        x[int(rule[5:])] = 1.0
        return x
    raise ValueError(rule)


def matmul_examples():
    for name, bits, K, codes, scales, biases, xrule, y in _lines("matmul_examples.txt"):
        K = int(K)
        codes = np.stack([codes_from_rule(r, K) for r in codes.split(";")])
        scales = np.array([[float(v) for v in r.split(",")] for r in scales.split(";")])
        biases = np.array([[float(v) for v in r.split(",")] for r in biases.split(";")])
        yield (name, int(bits), K, codes, scales, biases, x_from_rule(xrule, K),
               np.array([float(v) for v in y.split(";")]))



def gate_up_examples():
    """(name, bits, K, gate, up, x, h): gate and up are (codes [1, K], scales
    [1, K/64], biases [1, K/64]) with one scale and one bias for every group."""
    for (name, bits, K, gcodes, gs, gb, ucodes, us, ub, xrule,
         h) in _lines("gate_up_examples.txt"):
        K = int(K)
        G = K // 64

        def w(codes, sc, bi):
            return (codes_from_rule(codes, K)[None, :], np.full((1, G), float(sc)),
                    np.full((1, G), float(bi)))
        yield (name, int(bits), K, w(gcodes, gs, gb), w(ucodes, us, ub), x_from_rule(xrule, K),
               float(h))
