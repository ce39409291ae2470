"""Bit-exact packer / unpacker of the compressed KV page, format version 1 (oracle side).

TEST INFRASTRUCTURE (see ``oracle/__init__``).

The pages ask for a page-aligned compressed cache and note that quantized formats change
between releases, so the format is versioned.  This module restates the layout that the
library's public header defines, independently of the library code:

  cache = [batch][kv_head][page][page_bytes], P = 128 token slots per page.  A page holds
  six regions in this order (little-endian u32 words / f32):
    1. key codes   [b-1 planes][P tokens][d/32 words]   plane q holds bit q of each code
    2. key signs   [P tokens][m/32 words]               bit = sigma
    3. key norm    [P] f32                               n
    4. residual    [P] f32                               gamma = ||r||_2
    5. value codes [b planes][d coords][4 words]         plane q holds bit q of each code
    6. value norm  [P] f32

  Key codes and sign bits: within one token's words, coordinate j sits at
      kb = j>>5, h = (j>>4)&1, c = (j>>2)&3, e = j&3, s = c*(2*(D/32)) + 2*kb + h,
      word = s>>3, bit = (s&7) + 8*e                     (D = d for codes, m for signs)
  Value codes: within one coordinate's four words, token slot tau sits at
      kb = tau>>5, h = (tau>>4)&1, c = (tau>>2)&3, e = tau&3, word = c, bit = 2*kb+h+8*e
"""
import numpy as np

P = 128


def page_bytes(d, b, m):
    return P * ((b - 1) * d // 8 + m // 8 + 8 + b * d // 8 + 4)


def region_offsets(d, b, m):
    """Byte offsets of the six regions inside one page."""
    kc = 0
    sg = kc + (b - 1) * P * d // 8
    nk = sg + P * m // 8
    gm = nk + 4 * P
    vc = gm + 4 * P
    nv = vc + b * d * 4 * 4
    end = nv + 4 * P
    assert end == page_bytes(d, b, m)
    return dict(kcodes=kc, signs=sg, nk=nk, gamma=gm, vcodes=vc, nv=nv, end=end)


def coord_position(j, D):
    """(word, bit) of coordinate j inside one token's D/32 words (key codes, signs)."""
    j = np.asarray(j)
    kb, h, c, e = j >> 5, (j >> 4) & 1, (j >> 2) & 3, j & 3
    s = c * (2 * (D // 32)) + 2 * kb + h
    return s >> 3, (s & 7) + 8 * e


def token_position(tau):
    """(word, bit) of token slot tau inside one coordinate's 4 words (value codes)."""
    tau = np.asarray(tau)
    kb, h, c, e = tau >> 5, (tau >> 4) & 1, (tau >> 2) & 3, tau & 3
    return c, 2 * kb + h + 8 * e


def _pack_token_major(bits, D):
    """bits [P, D] in {0,1} -> words [P, D/32] (coordinate permutation above)."""
    words = np.zeros((bits.shape[0], D // 32), dtype=np.uint64)
    w, bpos = coord_position(np.arange(D), D)
    for j in range(D):
        words[:, w[j]] |= bits[:, j].astype(np.uint64) << np.uint64(bpos[j])
    return words.astype(np.uint32)


def _unpack_token_major(words, D):
    w, bpos = coord_position(np.arange(D), D)
    words = words.astype(np.uint64)
    out = np.zeros((words.shape[0], D), dtype=np.uint8)
    for j in range(D):
        out[:, j] = ((words[:, w[j]] >> np.uint64(bpos[j])) & np.uint64(1)).astype(np.uint8)
    return out


def pack_page(d, b, m, kidx, sigma, nk, gamma, vidx, nv):
    """One page from per-slot arrays of length P (kidx [P,d], sigma [P,m], vidx [P,d])."""
    off = region_offsets(d, b, m)
    buf = np.zeros(off["end"], dtype=np.uint8)
    kidx = np.asarray(kidx, dtype=np.int64)
    vidx = np.asarray(vidx, dtype=np.int64)
    # 1. key code planes
    planes = np.stack([_pack_token_major((kidx >> q) & 1, d) for q in range(b - 1)])
    buf[off["kcodes"]:off["signs"]] = planes.astype("<u4").view(np.uint8).ravel()
    # 2. sign plane
    buf[off["signs"]:off["nk"]] = _pack_token_major(np.asarray(sigma), m).astype("<u4").view(np.uint8).ravel()
    # 3, 4. key scalars
    buf[off["nk"]:off["gamma"]] = np.asarray(nk, dtype="<f4").view(np.uint8)
    buf[off["gamma"]:off["vcodes"]] = np.asarray(gamma, dtype="<f4").view(np.uint8)
    # 5. value code planes, coordinate-major over token slots
    vw = np.zeros((b, d, 4), dtype=np.uint64)
    wsl, bsl = token_position(np.arange(P))
    for q in range(b):
        bits = ((vidx >> q) & 1).astype(np.uint64)            # [P, d]
        for tau in range(P):
            vw[q, :, wsl[tau]] |= bits[tau, :] << np.uint64(bsl[tau])
    buf[off["vcodes"]:off["nv"]] = vw.astype("<u4").view(np.uint8).ravel()
    # 6. value norms
    buf[off["nv"]:off["end"]] = np.asarray(nv, dtype="<f4").view(np.uint8)
    return buf


def unpack_page(d, b, m, buf):
    """Inverse of ``pack_page``: dict(kidx, sigma, nk, gamma, vidx, nv) for all P slots."""
    off = region_offsets(d, b, m)
    buf = np.asarray(buf, dtype=np.uint8)
    kw = buf[off["kcodes"]:off["signs"]].view("<u4").reshape(b - 1, P, d // 32)
    kidx = np.zeros((P, d), dtype=np.int64)
    for q in range(b - 1):
        kidx |= _unpack_token_major(kw[q], d).astype(np.int64) << q
    sw = buf[off["signs"]:off["nk"]].view("<u4").reshape(P, m // 32)
    sigma = _unpack_token_major(sw, m)
    nk = buf[off["nk"]:off["gamma"]].view("<f4").copy()
    gamma = buf[off["gamma"]:off["vcodes"]].view("<f4").copy()
    vw = buf[off["vcodes"]:off["nv"]].view("<u4").reshape(b, d, 4).astype(np.uint64)
    wsl, bsl = token_position(np.arange(P))
    vidx = np.zeros((P, d), dtype=np.int64)
    for q in range(b):
        for tau in range(P):
            vidx[tau, :] |= (((vw[q, :, wsl[tau]] >> np.uint64(bsl[tau])) & np.uint64(1)).astype(np.int64) << q)
    nv = buf[off["nv"]:off["end"]].view("<f4").copy()
    return dict(kidx=kidx, sigma=sigma, nk=nk, gamma=gamma, vidx=vidx, nv=nv)


def unpack_tokens(d, b, m, cache_bytes, n_pages, batch, kv_head, n_tokens, kv_heads):
    """Per-token arrays for slots [0, n_tokens) of one (batch, kv_head) from a whole cache
    buffer laid out [batch][kv_head][n_pages][page]."""
    pb = page_bytes(d, b, m)
    base = ((batch * kv_heads) + kv_head) * n_pages * pb
    parts = []
    for p in range((n_tokens + P - 1) // P):
        parts.append(unpack_page(d, b, m, cache_bytes[base + p * pb: base + (p + 1) * pb]))
    out = {k: np.concatenate([pp[k] for pp in parts])[:n_tokens] for k in parts[0]} if parts else None
    return out
