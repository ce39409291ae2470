"""CPU checks of the algebra the tensor-core decode kernel relies on.

1. Each Lloyd-Max book (antisymmetric) is exactly 2 * sum_M alpha_M x_M(idx) - sum_M alpha_M
   over the odd subsets M of the code bits, x_M = XOR of those bits; even subsets vanish.
2. The e4m3 operand table: for bit position k of a byte, base_k and base_k | (1 << k) decode
   (by the OCP FP8 E4M3 definition) to beta_k and beta_k + gamma_k.
"""
import itertools

import numpy as np
import pytest

from oracle import codebook as ocb

BASE = [0x38, 0x38, 0x38, 0x30, 0x28, 0x18, 0x00, 0x38]
BETA = [1.0, 1.0, 1.0, 0.5, 0.25, 0.0625, 0.0, 1.0]
GAMMA = [0.125, 0.25, 0.5, 0.5, 0.75, 0.9375, 2.0, -2.0]


def e4m3(byte):
    """OCP 8-bit floating point, E4M3: bias 7, no infinities, S.1111.111 is NaN."""
    s = -1.0 if byte & 0x80 else 1.0
    e, m = (byte >> 3) & 0xF, byte & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * 2.0 ** -6 * m / 8.0
    return s * 2.0 ** (e - 7) * (1.0 + m / 8.0)


def odd_masks(n):
    return [m for m in range(1, 1 << n) if bin(m).count("1") % 2 == 1]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5])
def test_book_is_affine_in_xor_planes(d, bits):
    L = 2 ** bits
    c, _ = ocb.codebook(d, L)
    idx = np.arange(L)
    b = (idx[:, None] >> np.arange(bits)) & 1
    s = 2.0 * b - 1.0
    alphas = {}
    for r in range(bits + 1):
        for M in itertools.combinations(range(bits), r):
            mono = np.prod(s[:, list(M)], axis=1) if M else np.ones(L)
            alphas[M] = float(c @ mono) / L
            if r % 2 == 0:
                assert abs(alphas[M]) < 1e-15
    masks = odd_masks(bits)
    assert len(masks) == 2 ** (bits - 1)
    assert masks == sorted(masks) and masks[:4] == [1, 2, 4, 7][:len(masks)]
    recon = np.zeros(L)
    asum = 0.0
    for m in masks:
        M = tuple(q for q in range(bits) if (m >> q) & 1)
        x = np.bitwise_xor.reduce(b[:, list(M)], axis=1)
        recon += 2.0 * alphas[M] * x
        asum += alphas[M]
    assert np.max(np.abs(recon - asum - c)) < 1e-15


def test_e4m3_operand_table():
    for k in range(8):
        assert (BASE[k] >> k) & 1 == 0
        v0, v1 = e4m3(BASE[k]), e4m3(BASE[k] | (1 << k))
        assert v0 == BETA[k] and v1 - v0 == GAMMA[k]
    # the decoder itself against known encodings
    assert e4m3(0x7E) == 448.0 and e4m3(0x01) == 2.0 ** -9 and np.isnan(e4m3(0x7F))


def test_table_matches_torch_float8():
    torch = pytest.importorskip("torch")
    raw = torch.tensor([BASE[k] | (f << k) for k in range(8) for f in (0, 1)], dtype=torch.uint8)
    got = raw.view(torch.float8_e4m3fn).float().tolist()
    want = [BETA[k] + f * GAMMA[k] for k in range(8) for f in (0, 1)]
    assert got == want
