"""Pins for the oracle's resident caches beside an offloaded full cache (no GPU).

The retrieval drafter's rows packed into a buffer of their own, and the
streaming drafter's sinks + window packed likewise ("TriForce: Lossless
Acceleration of Long Sequence Generation with Hierarchical Speculative
Decoding", "Abstract (arXiv)": the offloading setting; "TriForce: Hierarchical
Speculative Decoding for LLMs", "The Three Forces of TriForce", Forces 1 and 2).
Pins: attention over a packed cache equals the already-pinned sparse and
window attention over the full cache; packed lengths against hand counts; the
row mapping against hand-written row lists.
"""

import numpy as np
import torch

from oracle import triforce as O


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def _rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _row_ids(Kc_bits, n):
    # rows of a cache whose row t holds the value t + 1 in every dim
    return [int(x) - 1 for x in O.bf16_to_f64(Kc_bits[:n, 0])]


def _position_cache(B, Hkv, Lmax, D):
    t = torch.arange(1, Lmax + 1, dtype=torch.float32)[None, None, :, None].expand(B, Hkv, Lmax, D)
    return _bits(t.contiguous().to(torch.bfloat16))  # integers <= 256 are exact in bf16


def test_packed_retrieval_cache_attends_like_the_sparse_call():
    B, Hq, Hkv, Lmax, D, chunk, kc = 3, 8, 2, 61, 128, 8, 4
    q = _bits(_rand_bf16((B, Hq, D), 1))
    K = _bits(_rand_bf16((B, Hkv, Lmax, D), 2, 2.0))
    V = _bits(_rand_bf16((B, Hkv, Lmax, D), 3))
    seq = np.array([61, 30, 0])
    idx = np.array([[[7, 0, 3, -1], [2, 2, 5, 9]],   # partial chunk 7 (rows 56..60); a repeated id; id 9 >= C
                    [[3, 1, -1, -1], [0, 1, 2, 3]],  # chunk 3 of a 30-token sequence holds rows 24..29
                    [[0, 1, 2, 3], [0, 0, 0, 0]]])   # L = 0: nothing is valid
    n_sel = np.array([[3, 4], [2, 4], [4, 0]])
    scale = D ** -0.5
    Kc, Vc, lens = O.compact_retrieval_cache(K, V, seq, idx, n_sel, chunk, kc)
    got = O.prefix_decode_attn(q, Kc, Vc, lens, scale)
    want = O.sparse_decode_attn(q, K, V, seq, idx, n_sel, chunk, scale)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)
    assert Kc.shape == (B, Hkv, kc * chunk, D)


def test_packed_lengths_and_rows_by_hand():
    B, Hkv, Lmax, D, chunk, kc = 1, 3, 21, 4, 8, 3
    K = _position_cache(B, Hkv, Lmax, D)
    V = K.copy()
    seq = np.array([21])  # chunks: 0 -> rows 0..7, 1 -> rows 8..15, 2 -> rows 16..20
    idx = np.array([[[2, 0, -1], [5, 2, 1], [1, 1, 0]]])
    n_sel = np.array([[2, 3, 3]])
    Kc, Vc, lens = O.compact_retrieval_cache(K, V, seq, idx, n_sel, chunk, kc)
    assert lens.tolist() == [[13, 13, 24]]
    assert _row_ids(Kc[0, 0], 13) == [16, 17, 18, 19, 20, 0, 1, 2, 3, 4, 5, 6, 7]
    assert _row_ids(Kc[0, 1], 13) == [16, 17, 18, 19, 20, 8, 9, 10, 11, 12, 13, 14, 15]
    assert _row_ids(Kc[0, 2], 24) == [8, 9, 10, 11, 12, 13, 14, 15, 8, 9, 10, 11, 12, 13, 14, 15,
                                      0, 1, 2, 3, 4, 5, 6, 7]
    assert np.array_equal(Kc, Vc)
    assert not Kc[0, 0, 13:].any() and not Kc[0, 1, 13:].any()
    # an empty selection packs nothing
    _, _, lens0 = O.compact_retrieval_cache(K, V, seq, idx, np.zeros((1, 3), int), chunk, kc)
    assert lens0.tolist() == [[0, 0, 0]]


def test_packed_window_attends_like_the_window_call():
    B, Hq, Hkv, Lmax, D = 4, 4, 4, 700, 128
    n_sink, window = 4, 252
    q = _bits(_rand_bf16((B, Hq, D), 4))
    K = _bits(_rand_bf16((B, Hkv, Lmax, D), 5, 2.0))
    V = _bits(_rand_bf16((B, Hkv, Lmax, D), 6))
    seq = np.array([700, 256, 100, 0])
    scale = D ** -0.5
    Kw, Vw, lens = O.window_cache(K, V, seq, n_sink, window)
    assert lens.tolist() == [256, 256, 100, 0]
    got = O.prefix_decode_attn(q, Kw, Vw, lens, scale)
    want = O.stream_window_attn(q, K, V, seq, n_sink, window, scale)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def test_packed_window_rows_by_hand():
    K = _position_cache(1, 1, 12, 4)
    Kw, _, lens = O.window_cache(K, K, np.array([12]), 2, 3)
    assert lens.tolist() == [5]
    assert _row_ids(Kw[0, 0], 5) == [0, 1, 9, 10, 11]
    Kw, _, lens = O.window_cache(K, K, np.array([4]), 2, 3)  # the context fits: every row once
    assert lens.tolist() == [4] and _row_ids(Kw[0, 0], 4) == [0, 1, 2, 3]


def test_packed_retrieval_cache_as_one_sequence_per_unit():
    # Viewing each (b, g) unit of the packed buffer as a sequence of its own
    # (one KV head, its G query heads, length = its packed count) turns the
    # per-unit prefix attention into the sparse call over consecutive chunk ids.
    B, Hq, Hkv, Lmax, D, chunk, kc = 2, 8, 4, 45, 128, 8, 3
    G = Hq // Hkv
    q = _bits(_rand_bf16((B, Hq, D), 7))
    K = _bits(_rand_bf16((B, Hkv, Lmax, D), 8, 2.0))
    V = _bits(_rand_bf16((B, Hkv, Lmax, D), 9))
    seq = np.array([45, 19])
    idx = np.array([[[5, 1, 0], [0, 2, 4], [3, 3, -1], [1, 2, 5]],
                    [[2, 0, 1], [1, 0, 7], [0, 0, 0], [2, 1, 0]]])
    n_sel = np.array([[3, 3, 2, 3], [3, 3, 0, 3]])
    scale = D ** -0.5
    Kc, Vc, lens = O.compact_retrieval_cache(K, V, seq, idx, n_sel, chunk, kc)
    assert any(int(n) % chunk for n in lens.ravel())  # some unit ends in a partial chunk
    units = B * Hkv
    ident = np.tile(np.arange(kc), (units, 1, 1))
    n_ident = -(-lens.reshape(units, 1) // chunk)
    got = O.sparse_decode_attn(q.reshape(units, G, D), Kc.reshape(units, 1, kc * chunk, D),
                               Vc.reshape(units, 1, kc * chunk, D), lens.reshape(units), ident, n_ident, chunk, scale)
    want = O.sparse_decode_attn(q, K, V, seq, idx, n_sel, chunk, scale)
    np.testing.assert_allclose(got.reshape(B, Hq, D), want, rtol=1e-13, atol=1e-13)
