"""Float64 CPU oracle for the TriForce decode-step attention path.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously-correct
statement of what the CUDA library computes.  Only the tests, the smoke check
and the CPU-baseline leg of the benchmark may import it; the product path
never does.  It shares no code with the CUDA library and imports nothing from
the package.

Sources, cited by page title and section:

* "TriForce: Hierarchical Speculative Decoding for LLMs" (blog explainer),
  section "The Architecture", sub-section "The Three Forces of TriForce":
  Force 1 (streaming drafter over attention sinks plus a recent window of
  W = 256 tokens), Force 2 (the target model over a retrieval-sparse cache of
  the KV blocks that score highest under key-query similarity, top-k of the
  context), Force 3 (the target over the full cache, verifying all candidates
  in one pass).
* Same page, section "Dual Rejection Sampling: Mathematical Losslessness":
  accept a candidate x when min(1, target(x)/draft(x)) >= u with u ~ U(0, 1);
  on rejection resample from max(0, p - q) normalised; the two levels
  (r -> q, then q -> p) telescope to the target distribution.
* "TriForce: Lossless Acceleration of Long Sequence Generation with
  Hierarchical Speculative Decoding", "Abstract (arXiv)": the whole KV cache
  is read for every generated token; the retrieval-sparse cache serves as the
  middle draft level.

Where the pages leave a step open the oracle takes one plain reading; each is
named in the docstring of the function it affects (chunk means as the block
representation, the dot-product score summed over a GQA group, ties to the
lower chunk id, the chain-causal verify mask, the "u <= ratio" comparison, the
bonus token and the index-order inverse CDF).

Parity pins live in tests/test_oracle_*.py; every function here has at least
one pin that does not re-use the function's own formula.

Array conventions: bf16 tensors are passed as numpy uint16 bit patterns; all
arithmetic is float64.  Shapes: K, V [B, Hkv, Lmax, D]; chunk means
M [B, Hkv, Cmax, D]; decode query q [B, Hq, D]; verify queries Q [B, Hq, T, D];
logits [B, rows, Vocab].  Query head h belongs to KV head h // (Hq // Hkv).
"""

from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# bf16 <-> float64
# ---------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of each bf16 bit pattern (bf16 is the top half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16, nearest with ties to even; returns bit patterns.

    bf16 keeps 8 significant bits and the fp32 exponent range (smallest
    subnormal 2**-133).  For x in [2**e, 2**(e+1)) the spacing of bf16 values is
    2**(e-7); below 2**-126 it is the subnormal spacing 2**-133.  np.rint
    rounds half to even, which on the integer multiple of the spacing is
    exactly ties-to-even on the last kept bit.  Values that round past the
    largest finite bf16 become infinities.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat = x.reshape(-1)
    res = np.empty(flat.shape, dtype=np.float64)
    finite = np.isfinite(flat)
    xf = np.where(finite, flat, 0.0)
    _, e2 = np.frexp(np.abs(xf))  # |x| = m * 2**e2, m in [0.5, 1)
    e = e2.astype(np.int64) - 1  # |x| in [2**e, 2**(e+1))
    spacing_exp = np.maximum(e - 7, -133)
    spacing = np.ldexp(1.0, spacing_exp)
    rounded = np.rint(xf / spacing) * spacing
    res[:] = np.where(finite, rounded, flat)
    max_bf16 = float(np.ldexp(255.0, 120))  # (2 - 2**-7) * 2**127
    res = np.where(np.abs(res) > max_bf16, np.copysign(np.inf, res), res)
    f32 = res.astype(np.float32)  # exact: every bf16 value is an fp32 value
    u32 = f32.view(np.uint32)
    nan = np.isnan(flat)
    u32 = np.where(nan, np.uint32(0x7FC00000), u32)
    out.reshape(-1)[:] = (u32 >> np.uint32(16)).astype(np.uint16)
    return out


# ---------------------------------------------------------------------------
# a1: chunk-mean index
# ---------------------------------------------------------------------------


def valid_len(seq_len: int, Lmax: int) -> int:
    """Sequence lengths are clamped to [0, Lmax] before use (library contract)."""
    return int(min(max(int(seq_len), 0), Lmax))


def build_chunk_means(K_bits, seq_lens, chunk, c_begin=0, c_end=None):
    """Per-chunk key means, the retrieval index of the Force 2 drafter.

    The blog page's "The Three Forces of TriForce" says Force 2 picks the most
    relevant historical KV blocks by key-query similarity and the page's
    "Production Advantages" section calls its bookkeeping an on-demand sparse
    index.  Reading: a block is `chunk` consecutive tokens and is represented
    by the mean of its keys.  For chunk c of sequence b with n_c = number of
    valid tokens of the chunk (chunk, fewer for the partial last chunk):
        M[b, g, c, :] = bf16_rne( (1 / n_c) * sum_{t in chunk c, t < L_b} K[b, g, t, :] )
    A chunk with no valid token gets all-zero means.  Only chunks in
    [c_begin, c_end) are produced; the returned array holds zeros elsewhere.

    The sum of at most eight bf16 values is exact in float64 whenever their
    magnitudes span fewer than 2**42 (always, for the synthetic inputs), so the
    only rounding is the final one, as the definition says.
    """
    K = bf16_to_f64(K_bits)
    B, Hkv, Lmax, D = K.shape
    Cmax = -(-Lmax // chunk)
    if c_end is None:
        c_end = Cmax
    M = np.zeros((B, Hkv, Cmax, D), dtype=np.float64)
    for b in range(B):
        L = valid_len(seq_lens[b], Lmax)
        for c in range(c_begin, c_end):
            t0 = c * chunk
            n = min(max(L - t0, 0), chunk)
            if n == 0:
                continue
            M[b, :, c, :] = K[b, :, t0 : t0 + n, :].sum(axis=1) / n
    return f64_to_bf16_rne(M)


# ---------------------------------------------------------------------------
# a2 + a3: chunk scores and top-k selection
# ---------------------------------------------------------------------------


def chunk_scores(q_bits, M_bits, seq_lens, Lmax, chunk, Hkv):
    """Key-query similarity of every chunk, per (sequence, KV head).

    Reading of "Key-Query similarity matching" (blog page, "The Three Forces
    of TriForce", Force 2): the dot product of the query with the chunk's mean
    key, with the query heads of one GQA group summed first, so that all heads
    of a group share one selection:
        s[b, g, c] = sum_d ( sum_{h in group g} q[b, h, d] ) * M[b, g, c, d]
    The softmax scale is left out (it does not change the order).  Returns a
    list over b of float64 arrays [Hkv, C_b] with C_b = ceil(L_b / chunk).
    """
    q = bf16_to_f64(q_bits)
    M = bf16_to_f64(M_bits)
    B, Hq, D = q.shape
    G = Hq // Hkv
    qsum = q.reshape(B, Hkv, G, D).sum(axis=2)  # [B, Hkv, D]
    out = []
    for b in range(B):
        L = valid_len(seq_lens[b], Lmax)
        C = -(-L // chunk)
        out.append(np.einsum("gd,gcd->gc", qsum[b], M[b, :, :C, :]))
    return out


def topk_chunks(scores_b, kc):
    """Top-kc chunks of one (sequence, KV head) by score.

    Force 2 keeps a fixed budget of the highest-scoring blocks (blog page,
    "The Three Forces of TriForce": top-k tokens of the context).  Readings:
    ties go to the lower chunk id; the selected ids are returned in ascending
    order; with C <= kc every chunk is selected.  Returns (ids ascending,
    s_cut = smallest selected score, gap = s_cut minus the best unselected
    score, +inf when nothing is left out).
    """
    s = np.asarray(scores_b, dtype=np.float64)
    C = s.shape[0]
    if C == 0:
        return np.zeros(0, dtype=np.int64), -np.inf, np.inf
    ids = np.arange(C)
    order = np.lexsort((ids, -s))  # primary: score descending, then id ascending
    keep = order[: min(kc, C)]
    s_cut = float(s[keep[-1]])
    gap = float(s_cut - s[order[kc]]) if C > kc else np.inf
    return np.sort(keep), s_cut, gap


def chunk_scores_topk(q_bits, M_bits, seq_lens, Lmax, chunk, kc, Hkv):
    """The library call's full output: idx [B, Hkv, kc] (-1 padded), n_sel, s_cut, gap."""
    scores = chunk_scores(q_bits, M_bits, seq_lens, Lmax, chunk, Hkv)
    B = len(scores)
    idx = np.full((B, Hkv, kc), -1, dtype=np.int64)
    n_sel = np.zeros((B, Hkv), dtype=np.int64)
    s_cut = np.full((B, Hkv), -np.inf)
    gap = np.full((B, Hkv), np.inf)
    for b in range(B):
        for g in range(Hkv):
            sel, cut, gp = topk_chunks(scores[b][g], kc)
            idx[b, g, : len(sel)] = sel
            n_sel[b, g] = len(sel)
            s_cut[b, g] = cut
            gap[b, g] = gp
    return idx, n_sel, s_cut, gap, scores


# ---------------------------------------------------------------------------
# a4 / a6 / a7: attention over an explicit set of positions
# ---------------------------------------------------------------------------


def attend(q_rows, K_rows, V_rows, scale):
    """softmax(scale * q K^T) V for each query row; zero output for an empty key set.

    Plain definition; the row maximum is subtracted before exponentiation,
    which leaves the softmax unchanged.  q_rows [n, D], K_rows/V_rows [m, D].
    """
    q_rows = np.atleast_2d(q_rows)
    if K_rows.shape[0] == 0:
        return np.zeros((q_rows.shape[0], V_rows.shape[1]))
    s = scale * (q_rows @ K_rows.T)
    s = s - s.max(axis=1, keepdims=True)
    w = np.exp(s)
    w = w / w.sum(axis=1, keepdims=True)
    return w @ V_rows


def attend_partial(q_rows, K_rows, V_rows, scale):
    """Unnormalised partial state (m, l, o) of attention over a subset of keys.

    m = max score, l = sum exp(s - m), o = sum exp(s - m) V.  Empty subsets give
    (m=-inf, l=0, o=0).  Used with merge_partials to state the split-K identity.
    """
    q_rows = np.atleast_2d(q_rows)
    n = q_rows.shape[0]
    if K_rows.shape[0] == 0:
        return np.full(n, -np.inf), np.zeros(n), np.zeros((n, V_rows.shape[1]))
    s = scale * (q_rows @ K_rows.T)
    m = s.max(axis=1)
    w = np.exp(s - m[:, None])
    return m, w.sum(axis=1), w @ V_rows


def merge_partials(parts):
    """Log-sum-exp merge of partial states (the split-K identity behind FlashDecoding,
    named in the blog page's "Production Advantages"):
        m = max_s m_s,  l = sum_s e^{m_s - m} l_s,  o = sum_s e^{m_s - m} o_s / l."""
    ms = np.stack([p[0] for p in parts])
    ls = np.stack([p[1] for p in parts])
    os_ = np.stack([p[2] for p in parts])
    m = ms.max(axis=0)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    f = np.where(np.isfinite(ms), np.exp(ms - safe_m[None]), 0.0)
    l = (f * ls).sum(axis=0)
    o = (f[..., None] * os_).sum(axis=0)
    out = np.where(l[:, None] > 0, o / np.where(l > 0, l, 1.0)[:, None], 0.0)
    return out


def sparse_positions(idx_row, n_sel, L, chunk, Lmax):
    """Token positions covered by the selected chunks, in list order.

    Valid tokens only (t < L).  Entries outside [0, ceil(L / chunk)) are skipped
    (library contract); a repeated id is attended once per occurrence.
    """
    C = -(-L // chunk)
    pos = []
    for i in range(int(n_sel)):
        c = int(idx_row[i])
        if c < 0 or c >= C:
            continue
        pos.extend(range(c * chunk, min(c * chunk + chunk, L)))
    return np.asarray(pos, dtype=np.int64)


def sparse_decode_attn(q_bits, K_bits, V_bits, seq_lens, idx, n_sel, chunk, scale):
    """Force 2 decode attention over the retrieved chunks only.

    Blog page, "The Three Forces of TriForce", Force 2: the target model
    attends to a small retrieved subset of the KV cache.  For query head h of
    KV group g: o = softmax(scale * q_h K_S^T) V_S with S the valid tokens of
    the chunks idx[b, g, :n_sel[b, g]].  Returns float64 [B, Hq, D].
    """
    q = bf16_to_f64(q_bits)
    K = bf16_to_f64(K_bits)
    V = bf16_to_f64(V_bits)
    B, Hq, D = q.shape
    Hkv, Lmax = K.shape[1], K.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = valid_len(seq_lens[b], Lmax)
        for g in range(Hkv):
            pos = sparse_positions(idx[b, g], n_sel[b, g], L, chunk, Lmax)
            for h in range(g * G, (g + 1) * G):
                out[b, h] = attend(q[b, h], K[b, g, pos], V[b, g, pos], scale)[0]
    return out


def window_positions(L, n_sink, window):
    """StreamingLLM position set: the first n_sink tokens plus the last `window`.

    Blog page, "The Three Forces of TriForce", Force 1: attention sinks plus
    the most recent W tokens (W = 256 in total there; the configured split is
    4 sinks + 252 recent).  Reading: the two ranges are de-duplicated, i.e.
    P = [0, min(n_sink, L)) U [max(n_sink, L - window), L).
    """
    a = list(range(0, min(n_sink, L)))
    b = list(range(max(n_sink, L - window), L))
    return np.asarray(a + b, dtype=np.int64)


def stream_window_attn(q_bits, K_bits, V_bits, seq_lens, n_sink, window, scale):
    """Force 1 decode attention over sinks + recent window.  Returns [B, Hq, D]."""
    q = bf16_to_f64(q_bits)
    K = bf16_to_f64(K_bits)
    V = bf16_to_f64(V_bits)
    B, Hq, D = q.shape
    Hkv, Lmax = K.shape[1], K.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = valid_len(seq_lens[b], Lmax)
        pos = window_positions(L, n_sink, window)
        for h in range(Hq):
            g = h // G
            out[b, h] = attend(q[b, h], K[b, g, pos], V[b, g, pos], scale)[0]
    return out


def verify_positions(L, T, j):
    """Keys seen by verify query j (0 <= j < T): positions [0, L - T + j].

    Reading of Force 3 (blog page, "The Three Forces of TriForce": all
    candidates verified against the full cache in one pass): the cache already
    holds the T candidates' keys at positions L-T .. L-1 and the candidates
    form a chain, so query j sees the prefix and candidates 0..j (causal).
    """
    return np.arange(0, max(L - T + j + 1, 0), dtype=np.int64)


def verify_attn(Q_bits, K_bits, V_bits, seq_lens, scale):
    """Force 3 verification attention.  Q [B, Hq, T, D] -> float64 [B, Hq, T, D]."""
    Q = bf16_to_f64(Q_bits)
    K = bf16_to_f64(K_bits)
    V = bf16_to_f64(V_bits)
    B, Hq, T, D = Q.shape
    Hkv, Lmax = K.shape[1], K.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, T, D))
    for b in range(B):
        L = valid_len(seq_lens[b], Lmax)
        for h in range(Hq):
            g = h // G
            for j in range(T):
                pos = verify_positions(L, T, j)
                out[b, h, j] = attend(Q[b, h, j], K[b, g, pos], V[b, g, pos], scale)[0]
    return out


def tree_ancestors(parent_row, j):
    """Candidate j and its ancestors, following parent links towards the prefix.

    Reading of the candidate tree (blog page, "The Three Forces of TriForce":
    Force 2 arranges the surviving candidates as a tree, Force 3 checks it in
    one pass with tree attention): parent_row[j] is the candidate that j
    extends, -1 when j extends the prefix directly.  A link that does not point
    to an earlier candidate ends the walk (read as -1).
    """
    out = [j]
    x = j
    while True:
        px = int(parent_row[x])
        if px < 0 or px >= x:
            return out
        out.append(px)
        x = px


def tree_verify_positions(L, T, j, parent_row):
    """Keys seen by tree-verify query j: the prefix [0, L - T) and the positions
    L - T + i of candidate j's ancestors-or-self i (those inside [0, L))."""
    pre = list(range(0, max(L - T, 0)))
    cand = sorted(L - T + i for i in tree_ancestors(parent_row, j) if 0 <= L - T + i < L)
    return np.array(pre + cand, dtype=np.int64)


def tree_verify_attn(Q_bits, K_bits, V_bits, seq_lens, parent, scale):
    """Force 3 over a candidate tree.  parent [B, T] ints; Q [B, Hq, T, D] -> float64.

    Query j of head h attends to tree_verify_positions; with parent[b, j] = j - 1
    for every j this is verify_attn.
    """
    Q = bf16_to_f64(Q_bits)
    K = bf16_to_f64(K_bits)
    V = bf16_to_f64(V_bits)
    B, Hq, T, D = Q.shape
    Hkv, Lmax = K.shape[1], K.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, T, D))
    for b in range(B):
        L = valid_len(seq_lens[b], Lmax)
        for h in range(Hq):
            g = h // G
            for j in range(T):
                pos = tree_verify_positions(L, T, j, parent[b])
                out[b, h, j] = attend(Q[b, h, j], K[b, g, pos], V[b, g, pos], scale)[0]
    return out


def sparse_verify_positions(idx_row, n_sel, L, T, j, chunk, Lmax):
    """Keys seen by query j (0 <= j < T) of the retrieval drafter's verification.

    Reading of the level-1 check (blog page, "The Three Forces of TriForce":
    the retrieval drafter, i.e. the target model over the retrieved KV blocks,
    verifies the tiny drafter's candidates; "Dual Rejection Sampling:
    Mathematical Losslessness": the candidates are checked in one pass): the
    cache already holds the T candidates' keys at positions L-T .. L-1; the
    drafter's own cache is the retrieved chunks of the context before them, so
    query j sees the valid tokens of the selected chunks that lie before L-T,
    then candidates 0..j (chain-causal).  List order: selection, then candidates.
    """
    start = max(L - T, 0)
    pre = [t for t in sparse_positions(idx_row, n_sel, L, chunk, Lmax) if t < start]
    return np.array(pre + list(range(start, max(L - T + j + 1, start))), dtype=np.int64)


def sparse_verify_attn(Q_bits, K_bits, V_bits, seq_lens, idx, n_sel, chunk, scale):
    """Level-1 verification attention over the retrieval cache plus the candidates.

    Q [B, Hq, T, D] bf16 bits, idx [B, Hkv, kc], n_sel [B, Hkv] -> float64
    [B, Hq, T, D]; query j of head h attends to sparse_verify_positions.
    """
    Q = bf16_to_f64(Q_bits)
    K = bf16_to_f64(K_bits)
    V = bf16_to_f64(V_bits)
    B, Hq, T, D = Q.shape
    Hkv, Lmax = K.shape[1], K.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, T, D))
    for b in range(B):
        L = valid_len(seq_lens[b], Lmax)
        for g in range(Hkv):
            for j in range(T):
                pos = sparse_verify_positions(idx[b, g], n_sel[b, g], L, T, j, chunk, Lmax)
                for h in range(g * G, (g + 1) * G):
                    out[b, h, j] = attend(Q[b, h, j], K[b, g, pos], V[b, g, pos], scale)[0]
    return out


# ---------------------------------------------------------------------------
# resident caches beside an offloaded full cache
# ---------------------------------------------------------------------------


def compact_retrieval_cache(K_bits, V_bits, seq_lens, idx, n_sel, chunk, kc):
    """The retrieval drafter's cache as a buffer of its own.

    "TriForce: Lossless Acceleration of Long Sequence Generation with
    Hierarchical Speculative Decoding", "Abstract (arXiv)": the retrieval-sparse
    cache is the middle draft level, and the offloading setting keeps the full
    cache in host memory; project summary, "How It Works": the KV cache can be
    offloaded to CPU memory.  Reading: when the full cache is offloaded, the
    drafter keeps a copy of the rows it attends to on the GPU.  For each
    (b, g) those are the rows of sparse_positions (valid tokens of the selected
    chunks, list order, invalid ids skipped), packed from row 0 of a
    [B, Hkv, kc * chunk, D] buffer; rows past the packed count are zero.
    Returns (Kc_bits, Vc_bits, lens) with lens [B, Hkv] the packed counts.
    """
    B, Hkv, Lmax, D = K_bits.shape
    cap = kc * chunk
    Kc = np.zeros((B, Hkv, cap, D), dtype=np.uint16)
    Vc = np.zeros((B, Hkv, cap, D), dtype=np.uint16)
    lens = np.zeros((B, Hkv), dtype=np.int64)
    for b in range(B):
        L = valid_len(seq_lens[b], Lmax)
        for g in range(Hkv):
            pos = sparse_positions(idx[b, g], min(int(n_sel[b, g]), kc), L, chunk, Lmax)
            Kc[b, g, : len(pos)] = K_bits[b, g, pos]
            Vc[b, g, : len(pos)] = V_bits[b, g, pos]
            lens[b, g] = len(pos)
    return Kc, Vc, lens


def window_cache(K_bits, V_bits, seq_lens, n_sink, window):
    """The streaming drafter's cache as a buffer of its own: for each (b, g) the
    rows of window_positions packed from row 0 of a [B, Hkv, n_sink + window, D]
    buffer (blog page, "The Three Forces of TriForce", Force 1: the sinks and
    the recent window are all that drafter reads, so they can stay on the GPU
    when the full cache is offloaded).  Returns (Kw_bits, Vw_bits, lens [B])."""
    B, Hkv, Lmax, D = K_bits.shape
    cap = n_sink + window
    Kw = np.zeros((B, Hkv, cap, D), dtype=np.uint16)
    Vw = np.zeros((B, Hkv, cap, D), dtype=np.uint16)
    lens = np.zeros(B, dtype=np.int64)
    for b in range(B):
        pos = window_positions(valid_len(seq_lens[b], Lmax), n_sink, window)
        Kw[b, :, : len(pos)] = K_bits[b][:, pos]
        Vw[b, :, : len(pos)] = V_bits[b][:, pos]
        lens[b] = len(pos)
    return Kw, Vw, lens


def prefix_decode_attn(q_bits, Kc_bits, Vc_bits, lens, scale):
    """Decode attention over a packed cache: query head h of KV group g attends
    to rows [0, lens[b, g]) of its unit (lens [B, Hkv], or [B] for one length
    per sequence).  Returns float64 [B, Hq, D]."""
    q = bf16_to_f64(q_bits)
    K = bf16_to_f64(Kc_bits)
    V = bf16_to_f64(Vc_bits)
    B, Hq, D = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    lens = np.asarray(lens)
    if lens.ndim == 1:
        lens = np.repeat(lens[:, None], Hkv, axis=1)
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            n = int(lens[b, g])
            out[b, h] = attend(q[b, h], K[b, g, :n], V[b, g, :n], scale)[0]
    return out


# ---------------------------------------------------------------------------
# a8: lossless accept / resample
# ---------------------------------------------------------------------------


def softmax_rows(logits, temperature):
    """Row-wise softmax(logits / temperature) in float64."""
    z = np.asarray(logits, dtype=np.float64) / temperature
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def inverse_cdf(w, u):
    """Index-order inverse CDF: the first t with sum_{v <= t} w_v > u * sum_v w_v.

    Vectorised over leading axes (w [..., V], u [...]).  If rounding leaves no
    such t, the last index with w_t > 0 is taken.  Also returns the distance of
    u from the two CDF boundaries that enclose the chosen t (normalised CDF),
    used to count draws that sit on a decision boundary.
    """
    w = np.asarray(w, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    W = w.sum(axis=-1)
    F = np.cumsum(w, axis=-1)
    target = (u * W)[..., None]
    above = F > target
    has = above.any(axis=-1)
    first = np.argmax(above, axis=-1)
    Vn = w.shape[-1]
    last_pos = Vn - 1 - np.argmax((w > 0)[..., ::-1], axis=-1)
    t = np.where(has, first, last_pos)
    Fn = F / np.where(W > 0, W, 1.0)[..., None]
    hi = np.take_along_axis(Fn, t[..., None], axis=-1)[..., 0]
    lo = np.where(t > 0, np.take_along_axis(Fn, np.maximum(t - 1, 0)[..., None], axis=-1)[..., 0], 0.0)
    margin = np.minimum(np.abs(u - hi), np.abs(u - lo))
    return t, margin


def draft_length(drf_tokens, V):
    """Number of drafted tokens per sequence: the index of the first entry outside
    [0, V) (a negative entry ends the draft), else gamma."""
    x = np.asarray(drf_tokens)
    bad = (x < 0) | (x >= V)
    gamma = x.shape[-1]
    return np.where(bad.any(axis=-1), np.argmax(bad, axis=-1), gamma)


def spec_accept(tgt_logits, drf_logits, drf_tokens, u_acc, u_res, temperature=1.0):
    """Speculative accept / resample of one verification level.

    Blog page, "Dual Rejection Sampling: Mathematical Losslessness": with p the
    verifier's distribution and q the drafter's, candidate x at position i is
    accepted when min(1, p_i(x) / q_i(x)) >= u_i; at the first rejection the
    verifier resamples from max(0, p - q) normalised.  The same rule serves
    both levels (tiny drafter -> retrieval drafter, retrieval drafter ->
    target); only the arguments change.  Readings: u <= ratio accepts; a draft
    probability of zero accepts; when every candidate is accepted one bonus
    token is drawn from the verifier's next row p_g; an all-zero residual
    (p == q) falls back to sampling p_j; sampling is the index-order inverse
    CDF with the supplied uniform.

    Shapes: tgt_logits [B, gamma+1, V] (p rows), drf_logits [B, gamma, V]
    (q rows), drf_tokens [B, gamma] (an entry outside [0, V) ends the draft),
    u_acc [B, gamma], u_res [B].  Logit arrays may have a leading 1 to
    broadcast over B.  Returns dict with n_acc [B], next [B],
    out_tokens [B, gamma+1] (accepted drafts, then the next token, then -1)
    and the smallest decision margin per sequence (distance of a uniform from
    the boundary of any decision it took).
    """
    x = np.asarray(drf_tokens, dtype=np.int64)
    u_acc = np.asarray(u_acc, dtype=np.float64)
    u_res = np.asarray(u_res, dtype=np.float64)
    B, gamma = x.shape
    p = softmax_rows(tgt_logits, temperature)
    q = softmax_rows(drf_logits, temperature)
    Vn = p.shape[-1]
    p = np.broadcast_to(p, (B, gamma + 1, Vn))
    q = np.broadcast_to(q, (B, gamma, Vn)) if gamma > 0 else np.zeros((B, 0, Vn))
    g = draft_length(x, Vn)
    bidx = np.arange(B)

    n_acc = np.full(B, -1, dtype=np.int64)
    margin = np.full(B, np.inf)
    for i in range(gamma):
        live = (n_acc < 0) & (i < g)
        xi = np.clip(x[:, i], 0, Vn - 1)
        pi = p[bidx, i, xi]
        qi = q[bidx, i, xi]
        ratio = np.where(qi > 0, pi / np.where(qi > 0, qi, 1.0), np.inf)
        accept = u_acc[:, i] <= ratio
        dist = np.abs(u_acc[:, i] - ratio)
        margin = np.where(live, np.minimum(margin, dist), margin)
        reject_now = live & ~accept
        n_acc = np.where(reject_now, i, n_acc)
    all_acc = n_acc < 0
    n_acc = np.where(all_acc, g, n_acc)

    j = np.minimum(n_acc, gamma)  # row of p used for the next token
    pj = p[bidx, j]
    qj = q[bidx, np.minimum(j, max(gamma - 1, 0))] if gamma > 0 else np.zeros_like(pj)
    resid = np.maximum(pj - qj, 0.0)
    resid_ok = resid.sum(axis=-1) > 0
    w = np.where((~all_acc & resid_ok)[:, None], resid, pj)
    nxt, m2 = inverse_cdf(w, u_res)
    margin = np.minimum(margin, m2)

    col = np.arange(gamma + 1)[None, :]
    xpad = np.concatenate([x, np.full((B, 1), -1, dtype=np.int64)], axis=1)
    out_tokens = np.where(col < n_acc[:, None], xpad, -1)
    out_tokens = np.where(col == n_acc[:, None], nxt[:, None], out_tokens)
    return {"n_acc": n_acc, "next": nxt, "out_tokens": out_tokens, "margin": margin}


def tree_parent(parent_row, j):
    """Parent of candidate j as the tree calls read it: parent_row[j] when it
    points to an earlier candidate or is -1 (the prefix), else -1 (a link
    outside [-1, j) attaches the candidate to the prefix, as tree_ancestors
    ends a walk there)."""
    pj = int(parent_row[j])
    return pj if -1 <= pj < j else -1


def spec_accept_tree(tgt_logits, drf_logits, drf_tokens, parent, u_acc, u_res, temperature=1.0):
    """Lossless accept / resample over a tree of candidates.

    Blog page, "The Three Forces of TriForce": Force 2 arranges the surviving
    candidates as a tree and Force 3 verifies the tree in one pass, applying
    the speculative rejection rule; "Dual Rejection Sampling: Mathematical
    Losslessness" prints the rule for one candidate: keep x when
    min(1, p(x)/q(x)) >= u, otherwise draw from max(0, p - q) normalised.  The
    pages print no rule for several candidates that extend the same node.
    Reading (the printed rule applied to the siblings one at a time, the only
    steps it uses are the printed ones): the children of a node are
    independent draws from the drafter's distribution at that node; they are
    tested in index order against the current target distribution p', which
    starts as the verifier's distribution at the node; a child that passes is
    kept and the walk continues at it with the verifier's distribution there;
    a child that fails replaces p' by max(0, p' - q) normalised (kept as is
    when that residual is all zero, as the chain call falls back to p_j) and
    the next sibling is tested.  When a node has no child left, the next
    token is drawn from p' with the index-order inverse CDF: the residual
    after the last rejection, or the verifier's distribution at the node (the
    bonus token) when nothing there was rejected.  With parent[j] = j - 1 for
    every j this is spec_accept.

    Shapes (T candidates): tgt_logits [B, T+1, V], row 0 the verifier at the
    prefix and row 1+j the verifier after candidate j; drf_logits [B, T, V],
    row j the drafter distribution candidate j was drawn from (its parent's);
    drf_tokens [B, T] (an entry outside [0, V) removes the candidate and so its
    subtree); parent [B, T] (read by tree_parent); u_acc [B, T] (the uniform of
    candidate j's test); u_res [B].  Logit arrays may have a leading 1 to
    broadcast over B.

    Because a child's index exceeds its parent's, visiting j = 0 .. T-1 once
    and testing j exactly when its parent is the current node and j is in the
    draft takes every node's children in index order, each after the walk
    reached that node.  Returns dict with n_acc [B] (depth of the kept path),
    next [B], out_tokens [B, T+1] (the kept tokens, the next token, -1 pad),
    acc_nodes [B, T] (the kept candidates' indices, -1 pad) and the smallest
    decision margin per sequence (as in spec_accept).
    """
    x = np.asarray(drf_tokens, dtype=np.int64)
    par = np.asarray(parent, dtype=np.int64)
    u_acc = np.asarray(u_acc, dtype=np.float64)
    u_res = np.asarray(u_res, dtype=np.float64)
    B, T = x.shape
    p = softmax_rows(tgt_logits, temperature)
    Vn = p.shape[-1]
    p = np.broadcast_to(p, (B, T + 1, Vn))
    q = np.broadcast_to(softmax_rows(drf_logits, temperature), (B, T, Vn)) if T > 0 else np.zeros((B, 0, Vn))
    bidx = np.arange(B)

    node = np.full(B, -1, dtype=np.int64)
    w = p[:, 0].copy()  # p': the distribution the next test and the final draw use
    n_acc = np.zeros(B, dtype=np.int64)
    acc_nodes = np.full((B, T), -1, dtype=np.int64)
    out_tokens = np.full((B, T + 1), -1, dtype=np.int64)
    margin = np.full(B, np.inf)
    for j in range(T):
        pj = np.array([tree_parent(par[b], j) for b in range(B)], dtype=np.int64)
        valid = (x[:, j] >= 0) & (x[:, j] < Vn)
        test = valid & (pj == node)
        xj = np.clip(x[:, j], 0, Vn - 1)
        wx = w[bidx, xj]
        qx = q[bidx, j, xj]
        ratio = np.where(qx > 0, wx / np.where(qx > 0, qx, 1.0), np.inf)
        accept = u_acc[:, j] <= ratio
        margin = np.where(test, np.minimum(margin, np.abs(u_acc[:, j] - ratio)), margin)
        keep = test & accept
        drop = test & ~accept
        # kept: the walk moves to candidate j
        acc_nodes[bidx[keep], n_acc[keep]] = j
        out_tokens[bidx[keep], n_acc[keep]] = x[keep, j]
        n_acc = np.where(keep, n_acc + 1, n_acc)
        node = np.where(keep, j, node)
        w = np.where(keep[:, None], p[:, 1 + j], w)
        # rejected: the residual against this candidate's drafter distribution
        r = np.maximum(w - q[:, j], 0.0)
        rs = r.sum(axis=-1)
        upd = drop & (rs > 0)
        w = np.where(upd[:, None], r / np.where(rs > 0, rs, 1.0)[:, None], w)
    nxt, m2 = inverse_cdf(w, u_res)
    margin = np.minimum(margin, m2)
    out_tokens[bidx, n_acc] = nxt
    return {"n_acc": n_acc, "next": nxt, "out_tokens": out_tokens, "acc_nodes": acc_nodes, "margin": margin}
