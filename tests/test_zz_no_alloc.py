"""The no-allocation sparse attention entry point, against the oracle and the
workspace entry point.

tf_sparse_decode_attn_noalloc serves callers that cannot allocate device
memory (an engine that owns every allocation, a plugin inside one, a
latency-critical loop where an allocation and its synchronisation are not
allowed): it keeps its scratch in a static per-device buffer of the library
instead of a caller workspace.  Each case is checked element by element
against the float64 oracle and against tf_sparse_decode_attn (the same
tolerance: for grouped heads the workspace call runs the tensor-core kernel and
this one the CUDA-core gather kernel).  This file runs last so that a failure
here never hides the other tests; it passes alone in a fresh process too.
"""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from hierarchical_speculative_decoding_gb300 import synth
from oracle import triforce as O

pytestmark = pytest.mark.gpu

ATOL = 2e-3
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _case(w, seed_layer):
    seq = synth.seq_lens_for(w)
    q, _ = synth.decode_queries(w, seed_layer)
    K, V, _ = synth.kv_cache(w, seed_layer, q, seq, fill_invalid=float("nan"))
    # Selection from a seeded draw (any valid id list works for this comparison).
    g = torch.Generator().manual_seed(100 + seed_layer)
    C = -(-w.L // w.chunk)
    kc = min(w.kc, C)
    idx = torch.full((w.B, w.Hkv, w.kc), -1, dtype=torch.int32)
    for b in range(w.B):
        for h in range(w.Hkv):
            idx[b, h, :kc] = torch.randperm(C, generator=g)[:kc].sort().values.to(torch.int32)
    n_sel = torch.full((w.B, w.Hkv), kc, dtype=torch.int32)
    n_sel[0, 0] = kc // 3  # a shorter list too
    return q, K, V, seq, idx, n_sel


def _run_and_check(cuda_lib, w, seed_layer):
    q, K, V, seq, idx, n_sel = _case(w, seed_layer)
    scale = w.D ** -0.5
    d = [t.to("cuda") for t in (q, K, V, seq, idx, n_sel)]
    want_ws = cuda_lib.tf_sparse_decode_attn(*d, scale)
    out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.tf_sparse_decode_attn_noalloc(*d, scale, out)
    torch.cuda.synchronize()
    want = O.sparse_decode_attn(_bits(q), _bits(K), _bits(V), seq.numpy(), idx.numpy(), n_sel.numpy(), w.chunk,
                                scale)
    got = out.cpu().double().numpy()
    err_oracle = float(np.abs(got - want).max())
    err_ws = float((out - want_ws).abs().max().item())
    assert np.isfinite(got).all(), w.name
    assert err_oracle <= ATOL, (w.name, "oracle", err_oracle)
    assert err_ws <= ATOL, (w.name, "workspace call", err_ws)


# One query head per KV head (gather kernel with one row per CTA), two, and
# four (the mixed-batch workload's 32/8 heads); a ragged batch with NaN past
# each length; a batch of 9 x 8 KV heads whose 72 tickets fill more than the
# 256 bytes the earlier calls used.
CASES = [
    synth.Workload("noalloc-mha", 2, 8, 8, 128, 5000, 1, 8, 1024, 4, 252, 6, 4, 100, 0.02, 31, True, 3000),
    synth.Workload("noalloc-g2", 1, 16, 8, 128, 6000, 1, 8, 2048, 4, 252, 6, 4, 100, 0.02, 32),
    synth.Workload("noalloc-g4", 3, 32, 8, 128, 9000, 1, 8, 4096, 4, 252, 6, 4, 100, 0.01, 33),
    synth.Workload("noalloc-72-units", 9, 32, 8, 128, 1200, 1, 8, 512, 4, 252, 6, 4, 100, 0.02, 34, True, 600),
]


def test_noalloc_matches_oracle_and_workspace_call_twice(cuda_lib):
    # The cases run in a row and then the first one again: every call reuses
    # the static scratch the previous one left behind.
    for i, w in enumerate(CASES + CASES[:1]):
        _run_and_check(cuda_lib, w, i)


def test_noalloc_accepts_the_mixed_batch_shape(cuda_lib):
    # Batch 8 x 8 KV heads x 4 query heads per group at kc = 512 (the mixed
    # batch workload's attention shape; 17.2 MB of partials) fits the scratch.
    w = synth.Workload("noalloc-b8-kc512", 8, 32, 8, 128, 4200, 1, 8, 4096, 4, 252, 6, 4, 100, 0.01, 35, True, 3000)
    _run_and_check(cuda_lib, w, 5)


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_lib):
    import ctypes

    lib = cuda_lib.load()
    P = ctypes.c_void_p
    buf = torch.zeros(16, dtype=torch.int32, device="cuda")  # never read: the call is rejected first
    p = P(buf.data_ptr())
    # 64 sequences x 32 KV heads x 4 query heads per group at kc = 512 needs ~550 MB of partials.
    st = lib.tf_sparse_decode_attn_noalloc(p, p, p, p, p, p, 64, 128, 32, 4096, 128, 8, 512, 0.1, p, None)
    assert st == 5  # TF_ERR_SCRATCH_LIMIT
    assert b"static buffer" in lib.tf_status_string(5)
    # One past the stated limit at kc = 512 with four heads per group (B * Hkv = 125).
    st = lib.tf_sparse_decode_attn_noalloc(p, p, p, p, p, p, 125, 500, 125, 4096, 128, 8, 512, 0.1, p, None)
    assert st == 5


_FIRST_CALL_UNDER_CAPTURE = r"""
import sys, ctypes, torch
sys.path.insert(0, sys.argv[1])
from hierarchical_speculative_decoding_gb300 import binding as tf
lib = tf.load()
torch.cuda.set_device(0)
buf = torch.zeros(16, dtype=torch.int32, device="cuda")
p = ctypes.c_void_p(buf.data_ptr())
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
with torch.cuda.stream(s):
    g.capture_begin()
    st = lib.tf_sparse_decode_attn_noalloc(p, p, p, p, p, p, 1, 8, 8, 64, 128, 8, 4, 0.1, p,
                                           ctypes.c_void_p(s.cuda_stream))
    g.capture_end()
print("STATUS", st)
"""


def test_noalloc_first_call_under_capture_is_refused(cuda_lib):
    # In a fresh process the first call sets the scratch up; made while its
    # stream is being captured it is refused before touching the device.
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_UNDER_CAPTURE, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "STATUS 1" in r.stdout, r.stdout + r.stderr[-2000:]
