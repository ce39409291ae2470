"""Bit-exact packer / unpacker of the compressed KV page (oracle side).

TEST INFRASTRUCTURE (see ``oracle/__init__``).

The pages ask for a page-aligned compressed cache and note that quantized formats change
between releases, so the format is versioned.  This module restates the layout that the
library's public header defines, independently of the library code.

Format version 1 (keys: b-1 Lloyd-Max bits + one QJL sign bit per projected coordinate;
values: b bits):

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

Paged pool (``paged_page_offset``, ``gather_paged``): the same pages kept in a pool of blocks
that sequences borrow in any order, as a PagedAttention-style serving engine holds its cache
([BLOG] 3.5, vLLM; [3BITS] "vLLM").  A block is the kv_heads pages of 128 consecutive token
slots, page (block, h) at byte (block * kv_heads + h) * page_bytes of the pool, and a table
row per sequence names the block of each of its logical pages.

Format version 2 (the ``*_kv`` functions) generalises version 1 to separate key and value
widths and to keys without the QJL stage ([3BITS] "Python + HuggingFace": a cache object
built with key_bits and value_bits, and a stage-1-only quantizer returning indices and
norms; the same page notes that the llama.cpp forks usually switch QJL off).  Its
parameters are the number of key code planes KB (Lloyd-Max bits of stage 1), the number of
value code planes VB and the projection size m, with m = 0 meaning no QJL stage: then
regions 2 (signs) and 4 (gamma) are empty and the other regions move up.  Every region keeps
the version-1 bit order, so version 1 is version 2 with KB = b-1, VB = b, m > 0, byte for
byte.
"""
import numpy as np

P = 128


def page_bytes_kv(d, kb, vb, m):
    """Bytes of one version-2 page: KB key planes, VB value planes, m sign bits (0: no QJL)."""
    qjl = P * (m // 8 + 4) if m > 0 else 0
    return P * (kb * d // 8 + 4 + vb * d // 8 + 4) + qjl


def region_offsets_kv(d, kb, vb, m):
    """Byte offsets of the six regions inside one version-2 page (empty regions have
    equal start and end)."""
    kc = 0
    sg = kc + kb * P * d // 8
    nk = sg + P * m // 8
    gm = nk + 4 * P
    vc = gm + (4 * P if m > 0 else 0)
    nv = vc + vb * d * 4 * 4
    end = nv + 4 * P
    assert end == page_bytes_kv(d, kb, vb, m)
    return dict(kcodes=kc, signs=sg, nk=nk, gamma=gm, vcodes=vc, nv=nv, end=end)


def page_bytes(d, b, m):
    """Bytes of one version-1 page."""
    return page_bytes_kv(d, b - 1, b, m)


def region_offsets(d, b, m):
    """Byte offsets of the six regions inside one version-1 page."""
    return region_offsets_kv(d, b - 1, b, m)


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


def pack_page_kv(d, kb, vb, m, kidx, sigma, nk, gamma, vidx, nv):
    """One version-2 page from per-slot arrays of length P (kidx [P,d], vidx [P,d]; sigma
    [P,m] and gamma [P] only when m > 0, ignored otherwise)."""
    off = region_offsets_kv(d, kb, vb, m)
    buf = np.zeros(off["end"], dtype=np.uint8)
    kidx = np.asarray(kidx, dtype=np.int64)
    vidx = np.asarray(vidx, dtype=np.int64)
    # 1. key code planes
    planes = np.stack([_pack_token_major((kidx >> q) & 1, d) for q in range(kb)])
    buf[off["kcodes"]:off["signs"]] = planes.astype("<u4").view(np.uint8).ravel()
    # 2. sign plane
    if m > 0:
        buf[off["signs"]:off["nk"]] = _pack_token_major(np.asarray(sigma), m).astype("<u4").view(np.uint8).ravel()
    # 3, 4. key scalars
    buf[off["nk"]:off["gamma"]] = np.asarray(nk, dtype="<f4").view(np.uint8)
    if m > 0:
        buf[off["gamma"]:off["vcodes"]] = np.asarray(gamma, dtype="<f4").view(np.uint8)
    # 5. value code planes, coordinate-major over token slots
    vw = np.zeros((vb, d, 4), dtype=np.uint64)
    wsl, bsl = token_position(np.arange(P))
    for q in range(vb):
        bits = ((vidx >> q) & 1).astype(np.uint64)            # [P, d]
        for tau in range(P):
            vw[q, :, wsl[tau]] |= bits[tau, :] << np.uint64(bsl[tau])
    buf[off["vcodes"]:off["nv"]] = vw.astype("<u4").view(np.uint8).ravel()
    # 6. value norms
    buf[off["nv"]:off["end"]] = np.asarray(nv, dtype="<f4").view(np.uint8)
    return buf


def unpack_page_kv(d, kb, vb, m, buf):
    """Inverse of ``pack_page_kv``: dict(kidx, sigma, nk, gamma, vidx, nv) for all P slots;
    sigma and gamma are None when m = 0."""
    off = region_offsets_kv(d, kb, vb, m)
    buf = np.asarray(buf, dtype=np.uint8)
    kw = buf[off["kcodes"]:off["signs"]].view("<u4").reshape(kb, P, d // 32)
    kidx = np.zeros((P, d), dtype=np.int64)
    for q in range(kb):
        kidx |= _unpack_token_major(kw[q], d).astype(np.int64) << q
    sigma = gamma = None
    if m > 0:
        sw = buf[off["signs"]:off["nk"]].view("<u4").reshape(P, m // 32)
        sigma = _unpack_token_major(sw, m)
        gamma = buf[off["gamma"]:off["vcodes"]].view("<f4").copy()
    nk = buf[off["nk"]:off["gamma"]].view("<f4").copy()
    vw = buf[off["vcodes"]:off["nv"]].view("<u4").reshape(vb, d, 4).astype(np.uint64)
    wsl, bsl = token_position(np.arange(P))
    vidx = np.zeros((P, d), dtype=np.int64)
    for q in range(vb):
        for tau in range(P):
            vidx[tau, :] |= (((vw[q, :, wsl[tau]] >> np.uint64(bsl[tau])) & np.uint64(1)).astype(np.int64) << q)
    nv = buf[off["nv"]:off["end"]].view("<f4").copy()
    return dict(kidx=kidx, sigma=sigma, nk=nk, gamma=gamma, vidx=vidx, nv=nv)


def pack_page(d, b, m, kidx, sigma, nk, gamma, vidx, nv):
    """One version-1 page from per-slot arrays of length P (kidx [P,d], sigma [P,m], vidx [P,d])."""
    return pack_page_kv(d, b - 1, b, m, kidx, sigma, nk, gamma, vidx, nv)


def unpack_page(d, b, m, buf):
    """Inverse of ``pack_page``: dict(kidx, sigma, nk, gamma, vidx, nv) for all P slots."""
    return unpack_page_kv(d, b - 1, b, m, buf)


def unpack_tokens_kv(d, kb, vb, m, cache_bytes, n_pages, batch, kv_head, n_tokens, kv_heads):
    """Per-token arrays for slots [0, n_tokens) of one (batch, kv_head) from a whole
    version-2 cache buffer laid out [batch][kv_head][n_pages][page]."""
    pb = page_bytes_kv(d, kb, vb, m)
    base = ((batch * kv_heads) + kv_head) * n_pages * pb
    parts = []
    for p in range((n_tokens + P - 1) // P):
        parts.append(unpack_page_kv(d, kb, vb, m, cache_bytes[base + p * pb: base + (p + 1) * pb]))
    if not parts:
        return None
    return {k: (None if parts[0][k] is None else np.concatenate([pp[k] for pp in parts])[:n_tokens])
            for k in parts[0]}


def unpack_tokens(d, b, m, cache_bytes, n_pages, batch, kv_head, n_tokens, kv_heads):
    """Per-token arrays for slots [0, n_tokens) of one (batch, kv_head) from a whole
    version-1 cache buffer laid out [batch][kv_head][n_pages][page]."""
    return unpack_tokens_kv(d, b - 1, b, m, cache_bytes, n_pages, batch, kv_head, n_tokens, kv_heads)


def paged_page_offset(block, kv_head, kv_heads, page_bytes):
    """Byte offset of the page of ``kv_head`` in ``block`` of a paged pool."""
    return (block * kv_heads + kv_head) * page_bytes


def gather_paged(pool_bytes, block_table, batch, kv_heads, page_bytes, n_pages):
    """The contiguous cache [batch][kv_head][n_pages][page] that a paged pool and its block
    table (int [batch][>= n_pages]) stand for: logical page p of (b, h) is the page of h in
    block block_table[b][p]."""
    out = np.zeros(batch * kv_heads * n_pages * page_bytes, dtype=np.uint8)
    for b in range(batch):
        for h in range(kv_heads):
            for p in range(n_pages):
                src = paged_page_offset(int(block_table[b][p]), h, kv_heads, page_bytes)
                dst = ((b * kv_heads + h) * n_pages + p) * page_bytes
                out[dst:dst + page_bytes] = pool_bytes[src:src + page_bytes]
    return out
