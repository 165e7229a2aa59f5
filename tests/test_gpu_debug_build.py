"""The checked build (TF_DEBUG): every call runs clean of bounds violations.

compute-sanitizer is not available here, so the library has a build in which
every kernel checks the data-dependent indices of its global-memory gathers
against the extents of their buffers, records a failure in a device word and
skips the access (tf_debug_status).  This test builds that variant and, in a
fresh process that loads it, runs the smoke sequence (every call against the
oracle) plus the calls that read through caller-given selections and host
memory, then requires that no check failed.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SCRIPT = r"""
import sys
sys.path.insert(0, sys.argv[1])
import numpy as np
import torch
import __graft_entry__ as entry
from hierarchical_speculative_decoding_gb300 import binding as tf
from hierarchical_speculative_decoding_gb300 import synth
assert tf.debug_variant() and tf.library_path().endswith("libtriforce_attn_debug.so")
tf.load()
st, flags = tf.tf_debug_status(clear=True)
assert st == 0, st
entry.smoke()  # every call, each checked against the oracle
# selections with ids past the context, negative ids and repeats (skipped by contract)
w = synth.Workload("dbg", 2, 8, 2, 128, 3000, 1, 8, 512, 4, 60, 6, 4, 100, 0.02, 9, True, 700)
seq = synth.seq_lens_for(w)
q, Q = synth.decode_queries(w, 0)
K, V, _ = synth.kv_cache(w, 0, q, seq)
d = "cuda"
rng = np.random.default_rng(1)
idx = torch.from_numpy(rng.integers(-2, 400, (2, 2, 64)).astype(np.int32)).to(d)
nsel = torch.full((2, 2), 64, dtype=torch.int32, device=d)
tf.tf_sparse_decode_attn(q.to(d), K.to(d), V.to(d), seq.to(d), idx, nsel, 0.088)
tf.tf_sparse_verify_attn(Q.to(d), K.to(d), V.to(d), seq.to(d), idx, nsel, 0.088)
tf.tf_pack_retrieval_cache(K.contiguous().pin_memory(), V.contiguous().pin_memory(), seq.to(d), idx, nsel)
out = torch.empty((2, 8, 128), dtype=torch.float32, device=d)
tf.tf_sparse_decode_attn_noalloc(q.to(d), K.to(d), V.to(d), seq.to(d), idx, nsel, 0.088, out)
torch.cuda.synchronize()
st, flags = tf.tf_debug_status()
print("FLAGS", st, flags)
"""


def test_checked_build_runs_every_call_without_violations(cuda_lib):
    env = dict(os.environ, TF_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", _SCRIPT, ROOT], env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    assert "smoke ok" in r.stdout
    assert "FLAGS 0 0" in r.stdout, r.stdout[-2000:]
