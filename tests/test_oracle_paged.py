"""Pins of the oracle's paged-pool address map (oracle.pagefmt.paged_page_offset / gather_paged).

A block is the kv_heads pages of 128 consecutive token slots; page (block, h) sits at byte
(block * kv_heads + h) * page_bytes of the pool, and row b of the block table names the block of
each logical page of sequence b ([BLOG] 3.5, vLLM and PagedAttention; [3BITS] "vLLM").
"""
import numpy as np

from oracle import pagefmt


def test_hand_derived_gather():
    # 4 blocks x 2 KV heads of 4-byte stand-in pages; pool byte i holds the value i
    pool = np.arange(32, dtype=np.uint8)
    table = [[2, 0], [1, 3]]
    got = pagefmt.gather_paged(pool, table, batch=2, kv_heads=2, page_bytes=4, n_pages=2)
    # (b, h, p) -> block table[b][p], head h -> bytes 4 * (2 * block + h) ...
    want = np.concatenate([
        np.arange(16, 20),   # b0 h0 p0: block 2, head 0 -> page index 4
        np.arange(0, 4),     # b0 h0 p1: block 0, head 0 -> page index 0
        np.arange(20, 24),   # b0 h1 p0: block 2, head 1 -> page index 5
        np.arange(4, 8),     # b0 h1 p1: block 0, head 1 -> page index 1
        np.arange(8, 12),    # b1 h0 p0: block 1, head 0 -> page index 2
        np.arange(24, 28),   # b1 h0 p1: block 3, head 0 -> page index 6
        np.arange(12, 16),   # b1 h1 p0: block 1, head 1 -> page index 3
        np.arange(28, 32),   # b1 h1 p1: block 3, head 1 -> page index 7
    ]).astype(np.uint8)
    assert np.array_equal(got, want)


def test_offsets_by_hand():
    assert pagefmt.paged_page_offset(0, 0, 8, 100) == 0
    assert pagefmt.paged_page_offset(0, 7, 8, 100) == 700
    assert pagefmt.paged_page_offset(3, 1, 8, 100) == 2500


def test_identity_table_is_the_contiguous_cache_for_one_head():
    # with one KV head and block b * n_pages + p, the pool is the contiguous cache itself
    rng = np.random.default_rng(0)
    batch, n_pages, pb = 3, 4, 16
    pool = rng.integers(0, 256, batch * n_pages * pb, dtype=np.uint8)
    table = [[b * n_pages + p for p in range(n_pages)] for b in range(batch)]
    assert np.array_equal(pagefmt.gather_paged(pool, table, batch, 1, pb, n_pages), pool)


def test_real_pages_round_trip_through_a_permuted_pool():
    # pack real version-1 pages, scatter them to a permuted pool, gather back and unpack
    rng = np.random.default_rng(1)
    d, b, m, batch, H, n_pages = 64, 3, 64, 2, 2, 3
    pb = pagefmt.page_bytes(d, b, m)
    pages = {}
    for bb in range(batch):
        for h in range(H):
            for p in range(n_pages):
                kidx = rng.integers(0, 1 << (b - 1), (pagefmt.P, d))
                sigma = rng.integers(0, 2, (pagefmt.P, m))
                vidx = rng.integers(0, 1 << b, (pagefmt.P, d))
                nk, gam, nv = (rng.random(pagefmt.P).astype(np.float32) for _ in range(3))
                pages[bb, h, p] = (kidx, sigma, nk, gam, vidx, nv)
    n_blocks = batch * n_pages + 2
    perm = rng.permutation(n_blocks)[:batch * n_pages]
    table = perm.reshape(batch, n_pages)
    pool = np.zeros(n_blocks * H * pb, dtype=np.uint8)
    for (bb, h, p), arrs in pages.items():
        off = pagefmt.paged_page_offset(int(table[bb, p]), h, H, pb)
        pool[off:off + pb] = pagefmt.pack_page(d, b, m, *arrs)
    cache = pagefmt.gather_paged(pool, table, batch, H, pb, n_pages)
    for (bb, h, p), (kidx, sigma, nk, gam, vidx, nv) in pages.items():
        base = ((bb * H + h) * n_pages + p) * pb
        got = pagefmt.unpack_page(d, b, m, cache[base:base + pb])
        assert np.array_equal(got["kidx"], kidx) and np.array_equal(got["vidx"], vidx)
        assert np.array_equal(got["sigma"], sigma) and np.array_equal(got["nv"], nv)
