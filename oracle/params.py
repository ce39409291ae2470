"""The per-(d, b, m, seed) constants of the method, built by the oracle's own routines.

TEST INFRASTRUCTURE (see ``oracle/__init__``).

Keys use a 2^(b-1)-level codebook (stage 1 has b-1 bits, stage 2 adds one sign bit per
projected coordinate); values use a 2^b-level codebook and no QJL stage ([BLOG] §1.2).

``make_kv`` builds the generalised set of constants: separate key and value widths, and keys
with or without the QJL stage ([3BITS] "Python + HuggingFace": a cache object takes
key_bits and value_bits; a stage-1-only quantizer takes bits).  Reading: key_bits counts
every stored bit per key coordinate, so with QJL the Lloyd-Max book of the keys has
2^(key_bits-1) levels and the sign bit is the last bit (version 1 is key_bits = value_bits =
b with QJL); without QJL it has 2^key_bits levels.
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


@dataclass
class KVParams:
    d: int
    kb: int          # Lloyd-Max bits of the keys (number of key code planes)
    vb: int          # bits of the values
    m: int           # QJL projection size; 0 when keys have no QJL stage
    seed: int
    Pi: np.ndarray
    S: np.ndarray    # None when m = 0
    cb_k: tuple
    cb_v: tuple


def make_kv(d, key_bits, value_bits, qjl=True, m=None, seed=0):
    """Constants for keys of key_bits bits (with or without QJL) and values of value_bits."""
    kb = key_bits - 1 if qjl else key_bits
    if kb < 1 or value_bits < 1:
        raise ValueError("key and value books need at least one bit")
    m = (d if m is None else m) if qjl else 0
    return KVParams(d=d, kb=kb, vb=value_bits, m=m, seed=seed,
                    Pi=rotation.haar_rotation(d, seed),
                    S=rotation.qjl_matrix(m, d, seed) if m > 0 else None,
                    cb_k=codebook.codebook(d, 2 ** kb),
                    cb_v=codebook.codebook(d, 2 ** value_bits))
