"""Pins for the oracle's bf16 rounding and chunk-mean index (no GPU).

The chunk mean is the retrieval index of the Force 2 drafter ("TriForce:
Hierarchical Speculative Decoding for LLMs", "The Three Forces of TriForce").
Its definition is an exact mean rounded once to bf16; these tests pin the
oracle against exact rational arithmetic and against torch's own fp32->bf16
conversion, never against the oracle's formula retyped.
"""

from fractions import Fraction

import numpy as np
import torch

from oracle import triforce as O


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


def test_rne_matches_torch_fp32_to_bf16():
    g = torch.Generator().manual_seed(5)
    parts = [
        torch.randn(100000, generator=g) * 3,
        torch.randn(10000, generator=g) * 1e-39,  # fp32 subnormals
        torch.randn(10000, generator=g) * 1e38,
        torch.tensor([0.0, -0.0, 1.0, -1.0, 3.3895314e38, -3.3895314e38, 1e-45]),
    ]
    x = torch.cat(parts).float()
    # Exact bf16 midpoints (ties) in both directions of evenness.
    base = torch.randn(5000, generator=g).to(torch.bfloat16).float()
    mids = (base.view(torch.int32) + 0x8000).view(torch.float32)
    x = torch.cat([x, mids])
    want = _bits(x.to(torch.bfloat16))
    got = O.f64_to_bf16_rne(x.double().numpy())
    assert np.array_equal(got, want)


def test_bf16_decode_exact():
    g = torch.Generator().manual_seed(6)
    t = torch.randn(4096, generator=g).to(torch.bfloat16)
    assert np.array_equal(O.bf16_to_f64(_bits(t)), t.double().numpy())


def _exact_bf16_round(fr: Fraction) -> float:
    """Round an exact rational to bf16 by brute force: the nearest of the two
    neighbouring bf16 values, ties to the even bit pattern."""
    f = float(fr)  # within half an fp64 ulp: good enough to locate neighbours
    c = torch.tensor([f], dtype=torch.float64).float().to(torch.bfloat16)
    cand_bits = int(c.view(torch.int16).item()) & 0xFFFF
    cands = []
    for d in (-2, -1, 0, 1, 2):
        b = (cand_bits + d) & 0xFFFF
        v = float(O.bf16_to_f64(np.array([b], dtype=np.uint16))[0])
        if np.isfinite(v):
            cands.append((abs(Fraction(v) - fr), b & 1, b, v))
    cands.sort(key=lambda z: (z[0], z[1]))
    return cands[0][3]


def test_chunk_means_exact_rational_with_partial_chunks():
    g = torch.Generator().manual_seed(7)
    B, Hkv, Lmax, D, chunk = 2, 2, 29, 4, 8
    K = torch.randn((B, Hkv, Lmax, D), generator=g).to(torch.bfloat16)
    seq_lens = np.array([29, 13])
    M = O.bf16_to_f64(O.build_chunk_means(_bits(K), seq_lens, chunk))
    Kv = K.double().numpy()
    for b in range(B):
        L = seq_lens[b]
        for h in range(Hkv):
            for c in range(-(-Lmax // chunk)):
                rows = [t for t in range(c * chunk, c * chunk + chunk) if t < L]
                for d in range(D):
                    if not rows:
                        assert M[b, h, c, d] == 0.0
                        continue
                    fr = sum(Fraction(float(Kv[b, h, t, d])) for t in rows) / len(rows)
                    assert M[b, h, c, d] == _exact_bf16_round(fr), (b, h, c, d)


def test_chunk_mean_of_constant_chunk_is_constant():
    val = torch.tensor(-1.703125, dtype=torch.bfloat16)
    K = val.repeat(1, 1, 16, 128)
    M = O.bf16_to_f64(O.build_chunk_means(_bits(K), np.array([16]), 8))
    assert np.all(M[0, 0, :2] == float(val))


def test_chunk_mean_ties_round_to_even():
    # bf16 spacing just above 1.0 is 2**-7.  Two-token partial chunks whose
    # exact means are: a midpoint with the even neighbour below, a midpoint
    # with the even neighbour above, an exact bf16 value, and another midpoint.
    e7, e6 = 2.0**-7, 2.0**-6
    tok0 = [1.0, 1.0 + e7, 1.0, 1.0 + e6]
    tok1 = [1.0 + e7, 1.0 + e6, 1.0 + e6, 1.0 + 3 * e7]
    want = [1.0, 1.0 + e6, 1.0 + e7, 1.0 + e6]
    K = torch.tensor([tok0, tok1], dtype=torch.bfloat16).reshape(1, 1, 2, 4)
    assert K.double().flatten().tolist() == tok0 + tok1  # inputs are exact in bf16
    M = O.bf16_to_f64(O.build_chunk_means(_bits(K), np.array([2]), 8))[0, 0, 0]
    assert M.tolist() == want
