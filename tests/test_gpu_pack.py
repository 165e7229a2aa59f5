"""GPU parity of tf_pack_retrieval_cache (the retrieval drafter's rows packed into
a resident buffer) against the float64 oracle's packing, from device memory and
from pinned host memory, and of the attention over the packed buffer (viewed as
one sequence per (b, g) through tf_sparse_decode_attn) against the oracle's
sparse attention over the full cache.

Packing is a copy: the packed rows, their counts and the chunk counts are
compared bit for bit; attention within the usual tolerance.
"""

import numpy as np
import pytest
import torch

from hierarchical_speculative_decoding_gb300 import synth
from oracle import triforce as O
from test_gpu_parity import ATOL, bits, make_case, scale_for, small_workload

pytestmark = pytest.mark.gpu


def selection(w, seq_cpu, kc, seed):
    """Seeded chunk lists with the edge cases: ids past the context, negative
    ids, repeats, the partial last chunk, n_sel of 0 and above kc."""
    rng = np.random.default_rng(seed)
    Cmax = -(-w.L // w.chunk)
    idx = rng.integers(-1, Cmax + 2, (w.B, w.Hkv, kc)).astype(np.int32)
    n_sel = rng.integers(0, kc + 1, (w.B, w.Hkv)).astype(np.int32)
    for b in range(w.B):
        C = -(-int(seq_cpu[b]) // w.chunk)
        if C > 0:
            idx[b, 0, 0] = C - 1  # the last (possibly partial) chunk
        if kc > 2:
            idx[b, -1, :3] = idx[b, -1, 2]  # a repeated id
    n_sel[0, 0] = 0
    n_sel[-1, -1] = kc + 5  # clamped to kc
    return idx, n_sel


def check_packed(w, c, idx, n_sel, kc, Kc, Vc, lens, n_chunks):
    oK, oV, olens = O.compact_retrieval_cache(bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(), idx, n_sel,
                                              w.chunk, kc)
    got_lens = lens.cpu().numpy().reshape(w.B, w.Hkv)
    assert np.array_equal(got_lens, olens)
    assert np.array_equal(n_chunks.cpu().numpy(), -(-got_lens.reshape(-1) // w.chunk))
    gK, gV = bits(Kc), bits(Vc)
    for b in range(w.B):
        for g in range(w.Hkv):
            n = int(olens[b, g])
            assert np.array_equal(gK[b, g, :n], oK[b, g, :n]), (b, g)
            assert np.array_equal(gV[b, g, :n], oV[b, g, :n]), (b, g)


def attend_packed(cuda_lib, w, q, Kc, Vc, lens, n_chunks, kc):
    """The packed buffer as B*Hkv sequences of one KV head each, chunk ids 0.."""
    units, G = w.B * w.Hkv, w.Hq // w.Hkv
    ident = torch.arange(kc, dtype=torch.int32, device="cuda").repeat(units, 1, 1).contiguous()
    out = cuda_lib.tf_sparse_decode_attn(q.view(units, G, w.D), Kc.view(units, 1, kc * w.chunk, w.D),
                                         Vc.view(units, 1, kc * w.chunk, w.D), lens, ident,
                                         n_chunks.view(units, 1), scale_for(w.D))
    return out.view(w.B, w.Hq, w.D)


@pytest.mark.parametrize("w,kc", [
    (small_workload(L=1003, L_min=300), 20),                 # GQA 4:1, ragged, partial chunks
    (small_workload(B=3, Hq=8, Hkv=8, L=517, L_min=9), 7),   # MHA, short sequences
    (small_workload(B=1, Hq=32, Hkv=8, L=2048, ragged=False), 64),
], ids=["gqa-ragged", "mha-short", "gqa-exact"])
@pytest.mark.parametrize("source", ["device", "pinned-host"])
def test_pack_matches_oracle(cuda_lib, w, kc, source):
    c = make_case(w, fill_invalid=float("nan") if w.ragged else None)
    idx, n_sel = selection(w, c["seq_cpu"], kc, seed=kc)
    if source == "device":
        K, V = c["K"], c["V"]
    else:
        K, V = c["K_cpu"].contiguous().pin_memory(), c["V_cpu"].contiguous().pin_memory()
    Kc, Vc, lens, n_chunks = cuda_lib.tf_pack_retrieval_cache(K, V, c["seq"], torch.from_numpy(idx).cuda(),
                                                              torch.from_numpy(n_sel).cuda())
    torch.cuda.synchronize()
    check_packed(w, c, idx, n_sel, kc, Kc, Vc, lens, n_chunks)
    out = attend_packed(cuda_lib, w, c["q"], Kc, Vc, lens, n_chunks, kc)
    torch.cuda.synchronize()
    want = O.sparse_decode_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(), idx,
                                np.minimum(n_sel, kc), w.chunk, scale_for(w.D))
    assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL


def test_pack_rejects_pageable_host_memory(cuda_lib):
    w = small_workload(B=1, Hkv=2, L=64, ragged=False)
    c = make_case(w)
    idx = torch.zeros((1, 2, 4), dtype=torch.int32, device="cuda")
    n_sel = torch.ones((1, 2), dtype=torch.int32, device="cuda")
    lib = cuda_lib.load()
    Kc = torch.empty((1, 2, 32, 128), dtype=torch.bfloat16, device="cuda")
    lens = torch.empty(2, dtype=torch.int32, device="cuda")
    K_pageable = c["K_cpu"].contiguous()
    p = lambda t: t.data_ptr()
    st = torch.cuda.current_stream().cuda_stream
    status = lib.tf_pack_retrieval_cache(p(K_pageable), p(K_pageable), p(c["seq"]), p(idx), p(n_sel), 1, 2, 64, 128,
                                         8, 4, p(Kc), p(Kc), p(lens), p(lens), st)
    assert status == 1  # TF_ERR_INVALID_ARG, nothing launched


def test_pack_full_size_layer(cuda_lib):
    """Llama2-7B shape at 131072 tokens: the top-k call's selection packed from
    device memory and from pinned host memory; the packed buffers agree, and the
    attention over them equals the sparse call over the full cache."""
    w = synth.LLAMA2_7B_128K
    seq_cpu = synth.seq_lens_for(w)
    seq = seq_cpu.cuda()
    q, _ = synth.decode_queries(w, 0, device="cuda")
    K, V, _ = synth.kv_cache(w, 0, q, seq_cpu, device="cuda")
    M = torch.empty((w.B, w.Hkv, w.L // w.chunk, w.D), dtype=torch.bfloat16, device="cuda")
    cuda_lib.tf_build_chunk_means(K, seq, M)
    idx, n_sel = cuda_lib.tf_chunk_scores_topk(q, M, seq, w.L, w.kc)
    Kc, Vc, lens, n_chunks = cuda_lib.tf_pack_retrieval_cache(K, V, seq, idx, n_sel)
    K_host = torch.empty(K.shape, dtype=K.dtype, pin_memory=True).copy_(K)
    V_host = torch.empty(V.shape, dtype=V.dtype, pin_memory=True).copy_(V)
    Kh, Vh, lens_h, n_chunks_h = cuda_lib.tf_pack_retrieval_cache(K_host, V_host, seq, idx, n_sel)
    sp = cuda_lib.tf_sparse_decode_attn(q, K, V, seq, idx, n_sel, scale_for(w.D))
    torch.cuda.synchronize()
    assert torch.equal(lens, lens_h) and torch.equal(n_chunks, n_chunks_h)
    assert int(lens.min()) == int(lens.max()) == w.kc * w.chunk  # every selected chunk is full at 128K
    assert torch.equal(Kc.view(torch.int16), Kh.view(torch.int16))
    assert torch.equal(Vc.view(torch.int16), Vh.view(torch.int16))
    out = attend_packed(cuda_lib, w, q, Kc, Vc, lens, n_chunks, w.kc)
    torch.cuda.synchronize()
    assert (out - sp).abs().max().item() <= 1e-4
    # one unit against the oracle, row by row
    b, g = 0, w.Hkv - 1
    u = b * w.Hkv + g
    oK, oV, olens = O.compact_retrieval_cache(bits(K[b:b + 1, g:g + 1]), bits(V[b:b + 1, g:g + 1]),
                                              seq_cpu[b:b + 1].numpy(), idx[b:b + 1, g:g + 1].cpu().numpy(),
                                              n_sel[b:b + 1, g:g + 1].cpu().numpy(), w.chunk, w.kc)
    assert int(olens[0, 0]) == int(lens[u])
    assert np.array_equal(bits(Kc[b, g]), oK[0, 0]) and np.array_equal(bits(Vc[b, g]), oV[0, 0])
