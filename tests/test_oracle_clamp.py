"""Pins of the length clamp every call applies: seq_lens values outside
[0, Lmax] act as the nearest end of that range (the library contract stated in
the C header).  Each oracle function given raw lengths must equal the same
function given the lengths clamped by hand, and a negative length must leave
nothing to attend (zero outputs, empty selections, no packed rows)."""

import numpy as np
import pytest

from oracle import triforce as O

LMAX, D, CH = 45, 128, 8


def test_valid_len_hand_values():
    assert [O.valid_len(x, LMAX) for x in (-(2 ** 31), -1, 0, 1, 44, 45, 46, 2 ** 31 - 1)] == \
        [0, 0, 0, 1, 44, 45, 45, 45]
    assert O.valid_len(7, 0) == 0 and O.valid_len(-7, 0) == 0


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).__rshift__(16).astype(np.uint16)


@pytest.fixture(scope="module")
def case():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, T = 3, 4, 2, 3
    K = _bits(rng.standard_normal((B, Hkv, LMAX, D)))
    V = _bits(rng.standard_normal((B, Hkv, LMAX, D)))
    q = _bits(rng.standard_normal((B, Hq, D)))
    Q = _bits(rng.standard_normal((B, Hq, T, D)))
    raw = np.array([LMAX + 9, -4, 30])
    clamped = np.array([LMAX, 0, 30])
    return dict(K=K, V=V, q=q, Q=Q, raw=raw, cl=clamped, Hkv=Hkv, T=T)


def test_every_oracle_function_clamps(case):
    c = case
    K, V, q, Q, raw, cl, Hkv = c["K"], c["V"], c["q"], c["Q"], c["raw"], c["cl"], c["Hkv"]
    s = D ** -0.5
    kc = 3
    M_raw = O.build_chunk_means(K, raw, CH)
    M_cl = O.build_chunk_means(K, cl, CH)
    assert np.array_equal(M_raw, M_cl)
    assert np.all(M_raw[1] == 0)  # no valid token: all-zero means
    t_raw = O.chunk_scores_topk(q, M_raw, raw, LMAX, CH, kc, Hkv)
    t_cl = O.chunk_scores_topk(q, M_cl, cl, LMAX, CH, kc, Hkv)
    for a, b in zip(t_raw[:4], t_cl[:4]):
        assert np.array_equal(a, b)
    idx, n_sel = t_raw[0], t_raw[1]
    assert np.all(n_sel[1] == 0) and np.all(idx[1] == -1)
    for f in (lambda L: O.sparse_decode_attn(q, K, V, L, idx, n_sel, CH, s),
              lambda L: O.stream_window_attn(q, K, V, L, 4, 10, s),
              lambda L: O.verify_attn(Q, K, V, L, s),
              lambda L: O.tree_verify_attn(Q, K, V, L, np.tile([-1, 0, 0], (3, 1)), s),
              lambda L: O.sparse_verify_attn(Q, K, V, L, idx, n_sel, CH, s)):
        a, b = f(raw), f(cl)
        assert np.array_equal(a, b)
        assert np.all(a[1] == 0)  # a negative length attends to nothing
    full_idx = np.tile(np.arange(6), (3, Hkv, 1))
    p_raw = O.compact_retrieval_cache(K, V, raw, full_idx, np.full((3, Hkv), 6), CH, 6)
    p_cl = O.compact_retrieval_cache(K, V, cl, full_idx, np.full((3, Hkv), 6), CH, 6)
    for a, b in zip(p_raw, p_cl):
        assert np.array_equal(a, b)
    assert list(p_raw[2][:, 0]) == [LMAX, 0, 30]  # every valid row, no row, 30 rows
    w_raw, w_cl = O.window_cache(K, V, raw, 4, 10), O.window_cache(K, V, cl, 4, 10)
    for a, b in zip(w_raw, w_cl):
        assert np.array_equal(a, b)
    assert list(w_raw[2]) == [14, 0, 14]
