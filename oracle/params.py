"""The per-(d, b, m, seed) constants of the method, built by the oracle's own routines.

TEST INFRASTRUCTURE (see ``oracle/__init__``).

Keys use a 2^(b-1)-level codebook (stage 1 has b-1 bits, stage 2 adds one sign bit per
projected coordinate); values use a 2^b-level codebook and no QJL stage ([BLOG] §1.2).
"""
from dataclasses import dataclass

import numpy as np

from . import codebook, rotation


@dataclass
class Params:
    d: int
    b: int
    m: int
    seed: int
    Pi: np.ndarray
    S: np.ndarray
    cb_k: tuple
    cb_v: tuple


def make(d, b, m=None, seed=0):
    m = d if m is None else m
    return Params(d=d, b=b, m=m, seed=seed,
                  Pi=rotation.haar_rotation(d, seed),
                  S=rotation.qjl_matrix(m, d, seed),
                  cb_k=codebook.codebook(d, 2 ** (b - 1)),
                  cb_v=codebook.codebook(d, 2 ** b))
