"""GPU parity of tf_sparse_verify_attn (the retrieval drafter's check of the
tiny drafter's candidates) against the float64 oracle.

Query j sees the selected chunks' valid rows before the candidates and
candidates 0..j.  Tolerance: max abs error <= 2e-3 (bf16 inputs, fp32
accumulation, P split into two bf16 parts for the P V product).
"""

import numpy as np
import pytest
import torch

from hierarchical_speculative_decoding_gb300 import synth
from oracle import triforce as O

from test_gpu_parity import ATOL, bits, make_case, small_workload

pytestmark = pytest.mark.gpu


def run_case(cuda_lib, c, idx, nsel, scale, chunk=8):
    out = cuda_lib.tf_sparse_verify_attn(c["Q"], c["K"], c["V"], c["seq"],
                                         torch.from_numpy(idx.astype(np.int32)).cuda(),
                                         torch.from_numpy(nsel.astype(np.int32)).cuda(), scale)
    torch.cuda.synchronize()
    want = O.sparse_verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(), idx,
                                nsel, chunk, scale)
    got = out.cpu().double().numpy()
    return got, want


def topk_over_prefix(w, c, kc):
    """The selection the drafter would use: top-kc chunks by the oracle's scores
    of the prefix before the candidates."""
    seq = c["seq_cpu"].numpy()
    pre = np.maximum(seq - w.T, 0)
    M = O.build_chunk_means(bits(c["K_cpu"]), pre, w.chunk)
    idx, nsel, *_ = O.chunk_scores_topk(bits(c["q_cpu"]), M, pre, w.L, w.chunk, kc, w.Hkv)
    return idx, nsel


@pytest.mark.parametrize("w", [
    synth.TINY,
    small_workload(),
    small_workload(B=2, Hq=32, Hkv=8, L=3000, T=6, budget=8 * 40, L_min=500),
    small_workload(B=1, Hq=8, Hkv=8, L=20000, T=6, budget=4096, ragged=False),
    small_workload(B=4, Hq=32, Hkv=8, L=6000, T=6, budget=4096, ragged=False),
    small_workload(B=8, Hq=32, Hkv=8, L=6000, T=6, budget=4096, L_min=4500),
], ids=["tiny", "ragged-gqa", "gqa-24-rows", "mha-20k-kc512", "32-units-cluster-merge", "64-units-ragged"])
def test_sparse_verify_topk_selection(cuda_lib, w):
    c = make_case(w, fill_invalid=float("nan"))
    idx, nsel = topk_over_prefix(w, c, w.kc)
    got, want = run_case(cuda_lib, c, idx, nsel, w.D ** -0.5)
    assert np.abs(got - want).max() <= ATOL


def test_sparse_verify_edge_selections(cuda_lib):
    """Unordered ids, invalid ids, a chunk straddling the candidates, a repeated
    id, an empty selection and a full selection (which equals full verification)."""
    w = small_workload(B=3, Hq=4, Hkv=2, L=203, T=5, budget=8 * 30, ragged=False)
    c = make_case(w, fill_invalid=float("nan"))
    c["seq_cpu"] = torch.tensor([203, 197, 3], dtype=torch.int32)  # 3 < T: candidates only, partly absent
    c["seq"] = c["seq_cpu"].cuda()
    kc = 30
    idx = np.full((3, 2, kc), -1, dtype=np.int64)
    nsel = np.zeros((3, 2), dtype=np.int64)
    idx[0, 0, :6] = [24, 3, 25, 99, -7, 3]  # 198..202 are candidates: chunk 24 = 192..199 straddles
    nsel[0, 0] = 6
    nsel[0, 1] = 0  # empty selection
    C1 = -(-197 // 8)
    idx[1, 0, :C1] = np.arange(C1)[::-1]
    nsel[1, 0] = C1  # every chunk, reversed
    idx[1, 1, :C1] = np.arange(C1)
    nsel[1, 1] = C1
    idx[2, :, 0] = 0
    nsel[2] = 1
    got, want = run_case(cuda_lib, c, idx, nsel, 0.07)
    assert np.abs(got - want).max() <= ATOL
    full = cuda_lib.tf_verify_attn(c["Q"], c["K"], c["V"], c["seq"], 0.07)
    torch.cuda.synchronize()
    assert np.abs(got[1] - full.cpu().double().numpy()[1]).max() <= ATOL


def test_sparse_verify_two_calls_share_the_workspace(cuda_lib):
    w = small_workload(B=2, Hq=8, Hkv=2, L=5000, T=6, budget=8 * 64, L_min=3000)
    c = make_case(w)
    idx, nsel = topk_over_prefix(w, c, w.kc)
    ws = cuda_lib.workspace(cuda_lib.tf_sparse_verify_attn_workspace(w.B, w.Hq, w.Hkv, w.kc, w.T), "cuda")
    it = torch.from_numpy(idx.astype(np.int32)).cuda()
    nt = torch.from_numpy(nsel.astype(np.int32)).cuda()
    a = cuda_lib.tf_sparse_verify_attn(c["Q"], c["K"], c["V"], c["seq"], it, nt, 0.09, ws=ws)
    b = cuda_lib.tf_sparse_verify_attn(c["Q"], c["K"], c["V"], c["seq"], it, nt, 0.09, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert int(ws[:4].view(torch.int32)[0]) == 0  # status word: no timeout
