"""Readers for the fixtures under tests/golden (formulas printed on the pages)."""

import os
from typing import NamedTuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


class AffineFixture(NamedTuple):
    name: str
    m: int
    n: int
    k: int
    cm: int
    ca: int
    s0: float
    ss: float
    b0: float
    bs: float
    f: str
    xa: float
    xf: float
    xp: float
    tol: float

    @property
    def derived(self) -> bool:
        """True for a shape that is not printed on the pages."""
        return self.name.startswith("derived:")


def affine_fixtures(include_derived=False):
    """Every fixture row of affine_fixtures.txt (page rows first)."""
    rows = []
    with open(os.path.join(HERE, "affine_fixtures.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c = line.split()
            fx = AffineFixture(c[0], int(c[1]), int(c[2]), int(c[3]), int(c[4]), int(c[5]),
                               float(c[6]), float(c[7]), float(c[8]), float(c[9]), c[10],
                               float(c[11]), float(c[12]), float(c[13]), float(c[14]))
            if fx.derived and not include_derived:
                continue
            rows.append(fx)
    return rows


def affine_fixture(fx: AffineFixture, group=32):
    """Codes ``[n, k]``, scales/biases ``[n, k/32]`` (float32) and ``x [m, k]``
    (float32) of one fixture, evaluated in float32 as the page's test does."""
    m, n, k = fx.m, fx.n, fx.k
    i = np.arange(n * k)
    codes = ((i * fx.cm + fx.ca) % 16).reshape(n, k).astype(np.int64)
    g = np.arange(n * (k // group)).astype(np.float32)
    scales = (np.float32(fx.s0) + g * np.float32(fx.ss)).reshape(n, k // group)
    biases = (np.float32(fx.b0) + g * np.float32(fx.bs)).reshape(n, k // group)
    xi = np.arange(m * k).astype(np.float32)
    fn = {"sin": np.sin, "cos": np.cos}[fx.f]
    x = (fn(xi * np.float32(fx.xf) + np.float32(fx.xp)) * np.float32(fx.xa)).astype(np.float32)
    return codes, scales.astype(np.float32), biases.astype(np.float32), x.reshape(m, k)
