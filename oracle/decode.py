"""Decode attention over the compressed KV cache (oracle, fp64).

TEST INFRASTRUCTURE (see ``oracle/__init__``).

The score of a cached key for a query q is the inner product with the reconstructed key:
the Lloyd-Max term n <Pi q, c[idx]> plus the QJL correction
gamma * sqrt(pi/2)/m * <S q, 2 sigma - 1> ([BLOG] §1.2: ||r||_2 is the reconstruction
scale of the sign sketch).  Softmax attention then weights the reconstructed values
n_v Pi^T c_v[idx_v].

Readings: logits are scaled by 1/sqrt(d); no mask other than t < seq_len; query head h
reads kv head floor(h / G) with G = Hq / Hkv (consecutive grouping); an empty sequence
(seq_len = 0) yields an all-zero output.

Keys without the QJL stage (tok_k["sigma"] is None; [3BITS] "Python + HuggingFace" and its
remark that the llama.cpp forks switch QJL off) score by the Lloyd-Max term alone.

Sparse V ([3BITS] llama.cpp section, the format list: positions with low attention weights
are skipped during decoding) is ``attend_sparse_v``.  The pages fix neither the threshold nor
the normalisation; the reading taken: with p_t = exp(l_t - max l), a position whose p_t is
below theta leaves the weighted sum of values, while the softmax denominator keeps every
position (the scores are computed either way; what is skipped is the value work).

Two routes are given.  Route A reconstructs every key and value in the original frame
(plain definition).  Route B works in the rotated frame (q~ = Pi q, q_s = S q, output
rotated back once by Pi^T); it is mathematically identical and serves as an internal
check of the algebra the GPU path relies on.
"""
import numpy as np

from . import quant


def _softmax(logits):
    mx = np.max(logits)
    e = np.exp(logits - mx)
    return e / np.sum(e)


def attend_route_a(q, tok_k, tok_v, Pi, S, cb_k, cb_v):
    """q [d] fp64; tok_k = dict(idx, n, sigma, gamma); tok_v = dict(idx, n).
    Returns (out [d], logits [T])."""
    d = Pi.shape[0]
    T = len(tok_k["n"])
    if T == 0:
        return np.zeros(d), np.zeros(0)
    khat = quant.reconstruct_keys_any(tok_k, Pi, S, cb_k[0])
    logits = khat @ np.asarray(q, dtype=np.float64) / np.sqrt(d)
    p = _softmax(logits)
    vhat = quant.reconstruct_values(tok_v["idx"], tok_v["n"], Pi, cb_v[0])
    return p @ vhat, logits


def attend_sparse_v(q, tok_k, tok_v, Pi, S, cb_k, cb_v, theta):
    """Sparse V: route A with the values of positions whose p_t = exp(l_t - max l) < theta
    dropped from the numerator only.  Returns (out [d], logits [T], skipped) where
    skipped = sum over dropped t of p_t ||v^_t|| / sum_t p_t bounds the change against the
    dense output, and against any evaluation that drops a subset of these positions."""
    d = Pi.shape[0]
    T = len(tok_k["n"])
    if T == 0:
        return np.zeros(d), np.zeros(0), 0.0
    khat = quant.reconstruct_keys_any(tok_k, Pi, S, cb_k[0])
    logits = khat @ np.asarray(q, dtype=np.float64) / np.sqrt(d)
    e = np.exp(logits - np.max(logits))
    keep = e >= theta
    vhat = quant.reconstruct_values(tok_v["idx"], tok_v["n"], Pi, cb_v[0])
    den = np.sum(e)
    out = (np.where(keep, e, 0.0) @ vhat) / den
    skipped = float(np.sum(np.where(keep, 0.0, e) * np.linalg.norm(vhat, axis=1)) / den)
    return out, logits, skipped


def ip_topk(q, tok_k, Pi, S, cb_k, k):
    """Compressed inner-product scan ([BLOG] 6.4: vector search over compressed indexes): the k
    cached keys with the largest estimated <q, k^_t> (the reconstructed key's inner product:
    the Lloyd-Max term plus, with QJL, the sign-sketch correction), equal estimates by lower
    slot.  Returns (slots [min(k, T)], estimates) in that order."""
    T = len(tok_k["n"])
    if T == 0:
        return np.zeros(0, dtype=np.int64), np.zeros(0)
    khat = quant.reconstruct_keys_any(tok_k, Pi, S, cb_k[0])
    # every row summed in the same order, so that equal keys get equal estimates
    est = np.sum(khat * np.asarray(q, dtype=np.float64)[None, :], axis=1)
    order = sorted(range(T), key=lambda t: (-est[t], t))[:k]
    order = np.asarray(order, dtype=np.int64)
    return order, est[order]


def attend_route_b(q, tok_k, tok_v, Pi, S, cb_k, cb_v):
    """Rotated-frame evaluation of the same quantities as ``attend_route_a``."""
    d = Pi.shape[0]
    T = len(tok_k["n"])
    if T == 0:
        return np.zeros(d), np.zeros(0)
    q = np.asarray(q, dtype=np.float64)
    qr = Pi @ q
    nk = np.asarray(tok_k["n"], dtype=np.float64)
    mse = nk * (np.asarray(cb_k[0])[tok_k["idx"]] @ qr)
    qjl = 0.0
    if tok_k.get("sigma") is not None:
        m = S.shape[0]
        qs = S @ q
        gm = np.asarray(tok_k["gamma"], dtype=np.float64)
        qjl = gm * quant.QJL_CONST / m * ((2.0 * np.asarray(tok_k["sigma"], dtype=np.float64) - 1.0) @ qs)
    logits = (mse + qjl) / np.sqrt(d)
    p = _softmax(logits)
    nv = np.asarray(tok_v["n"], dtype=np.float64)
    o_rot = (p * nv) @ np.asarray(cb_v[0])[tok_v["idx"]]
    return Pi.T @ o_rot, logits


def decode(q, tokens_for, kv_heads, Pi, S, cb_k, cb_v, route="a"):
    """Attention for every query head.  q [B, Hq, d]; tokens_for(b, kv_head) returns
    (tok_k, tok_v) for the slots t < seq_len[b].  Returns (out [B, Hq, d], logits[b][h])."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    G = Hq // kv_heads
    fn = attend_route_a if route == "a" else attend_route_b
    out = np.zeros((B, Hq, d))
    logits = [[None] * Hq for _ in range(B)]
    for b in range(B):
        for g in range(kv_heads):
            tk, tv = tokens_for(b, g)
            for h in range(g * G, (g + 1) * G):
                out[b, h], logits[b][h] = fn(q[b, h], tk, tv, Pi, S, cb_k, cb_v)
    return out, logits
