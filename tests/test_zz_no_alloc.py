"""The no-allocation sparse attention entry point matches the workspace one.

tf_sparse_decode_attn_noalloc serves callers that cannot allocate device
memory (an engine that owns every allocation, a latency-critical loop): it
keeps its scratch in a static per-device buffer of the library instead of a
caller workspace.  This file runs last so that a failure here never hides the
other tests; it passes alone in a fresh process too.
"""

import numpy as np
import pytest
import torch

from hierarchical_speculative_decoding_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL = 2e-3


def _case(w, seed_layer):
    seq = synth.seq_lens_for(w)
    q, _ = synth.decode_queries(w, seed_layer)
    K, V, _ = synth.kv_cache(w, seed_layer, q, seq)
    d = "cuda"
    # Selection from a seeded draw (any valid id list works for this comparison).
    g = torch.Generator().manual_seed(100 + seed_layer)
    C = -(-w.L // w.chunk)
    idx = torch.stack([torch.stack([torch.randperm(C, generator=g)[: w.kc].sort().values for _ in range(w.Hkv)])
                       for _ in range(w.B)]).to(torch.int32)
    n_sel = torch.full((w.B, w.Hkv), w.kc, dtype=torch.int32)
    n_sel[0, 0] = w.kc // 3  # a shorter list too
    return [t.to(d) for t in (q, K, V, seq, idx, n_sel)]


def test_noalloc_matches_workspace_entry_point_twice(cuda_lib):
    # Two calls in a row with different shapes: the second reuses the static
    # scratch the first one left behind.
    cases = [
        synth.Workload("noalloc-a", 2, 8, 2, 128, 5000, 1, 8, 1024, 4, 252, 6, 4, 100, 0.02, 31, True, 3000),
        synth.Workload("noalloc-b", 3, 32, 8, 128, 9000, 1, 8, 4096, 4, 252, 6, 4, 100, 0.01, 32),
    ]
    for i, w in enumerate(cases):
        q, K, V, seq, idx, n_sel = _case(w, i)
        scale = w.D ** -0.5
        want = cuda_lib.tf_sparse_decode_attn(q, K, V, seq, idx, n_sel, scale)
        out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
        cuda_lib.tf_sparse_decode_attn_noalloc(q, K, V, seq, idx, n_sel, scale, out)
        torch.cuda.synchronize()
        err = (out - want).abs().max().item()
        assert np.isfinite(err) and err <= ATOL, (w.name, err)


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_lib):
    import ctypes

    lib = cuda_lib.load()
    P = ctypes.c_void_p
    buf = torch.zeros(16, dtype=torch.int32, device="cuda")  # never read: the call is rejected first
    p = P(buf.data_ptr())
    # 64 sequences x 32 KV heads x 4 query heads per group at kc = 512 needs ~136 MB of partials.
    st = lib.tf_sparse_decode_attn_noalloc(p, p, p, p, p, p, 64, 128, 32, 4096, 128, 8, 512, 0.1, p, None)
    assert st == 5  # TF_ERR_SCRATCH_LIMIT
    assert b"static buffer" in lib.tf_status_string(5)
