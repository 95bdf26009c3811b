"""Readers for the fixtures under tests/golden (formulas printed on the pages)."""

import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def affine_fixture_shapes():
    rows = []
    with open(os.path.join(HERE, "affine_fixtures.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            m, n, k, tol = line.split()
            rows.append((int(m), int(n), int(k), float(tol)))
    return rows


def affine_fixture(m, n, k, group=32):
    """Codes ``[n, k]``, scales/biases ``[n, k/32]`` (float32) and ``x [m, k]`` (float32)."""
    i = np.arange(n * k)
    codes = ((i * 11 + 5) % 16).reshape(n, k).astype(np.int64)
    g = np.arange(n * (k // group))
    scales = (np.float32(0.05) + g.astype(np.float32) * np.float32(0.0017)).reshape(n, k // group)
    biases = (np.float32(-0.13) + g.astype(np.float32) * np.float32(0.0023)).reshape(n, k // group)
    xi = np.arange(m * k).astype(np.float32)
    x = (np.sin(xi * np.float32(0.013) - np.float32(0.4)) * np.float32(0.6)).astype(np.float32)
    return codes, scales.astype(np.float32), biases.astype(np.float32), x.reshape(m, k)
