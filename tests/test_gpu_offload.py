"""GPU parity of the offloaded verify (K/V in pinned host memory, streamed in
segments through two device staging slots) against the float64 oracle and
against tf_verify_attn on a device-resident copy of the same cache.

Offloading changes where the cache lives, not what is computed, so the oracle
is the verify oracle itself; tolerance as for every attention output.
"""
import numpy as np
import pytest
import torch

from oracle import triforce as O
from test_gpu_parity import ATOL, bits, make_case, scale_for, small_workload

pytestmark = pytest.mark.gpu


def offload_case(w, seg_rows, copy_stream=True, fill_invalid=float("nan")):
    c = make_case(w, fill_invalid=fill_invalid if w.ragged else None)
    K_host = c["K_cpu"].contiguous().pin_memory()
    V_host = c["V_cpu"].contiguous().pin_memory()
    L_stream = int(c["seq_cpu"].max().item())
    return c, K_host, V_host, L_stream


def run_offload(cuda_lib, w, c, K_host, V_host, L_stream, seg_rows, copy_stream=None, ws=None):
    out = cuda_lib.tf_verify_attn_offload(c["Q"], K_host, V_host, c["seq"], L_stream, scale_for(w.D), ws=ws,
                                          seg_rows=seg_rows, copy_stream=copy_stream)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("w,seg_rows", [
    (small_workload(L=3000, L_min=700), 512),                          # several segments, ragged, partial last
    (small_workload(L=3000, L_min=700), 300),                          # segment not a multiple of the 128-key tile
    (small_workload(Hkv=8, T=6, L=2048, ragged=False), 1024),         # exact multiple: two full segments
    (small_workload(Hkv=8, T=1, L=1500, L_min=1000), 4096),           # one segment larger than the context
    (small_workload(B=1, Hq=32, Hkv=8, T=6, L=5000, L_min=4000), 777),  # GQA, 24 query rows
], ids=["ragged-512", "ragged-300", "mha-exact-1024", "t1-one-segment", "gqa-777"])
def test_offloaded_verify_matches_oracle_and_resident_verify(cuda_lib, w, seg_rows):
    c, K_host, V_host, L_stream = offload_case(w, seg_rows)
    side = torch.cuda.Stream()
    out = run_offload(cuda_lib, w, c, K_host, V_host, L_stream, seg_rows, copy_stream=side)
    want = O.verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(),
                         scale_for(w.D))
    assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL
    resident = cuda_lib.tf_verify_attn(c["Q"], c["K"], c["V"], c["seq"], scale_for(w.D))
    torch.cuda.synchronize()
    assert torch.allclose(out, resident, atol=1e-5, rtol=1e-5)


def test_offloaded_verify_on_one_stream_and_workspace_reuse(cuda_lib):
    w = small_workload(L=2500, L_min=900)
    seg_rows = 640
    c, K_host, V_host, L_stream = offload_case(w, seg_rows)
    nbytes = cuda_lib.tf_verify_attn_offload_workspace(w.B, w.Hq, w.Hkv, w.L, w.T, seg_rows)
    ws = cuda_lib.workspace(nbytes, "cuda")
    want = O.verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(),
                         scale_for(w.D))
    for _ in range(2):  # same stream for copies and kernels; the workspace reused
        out = run_offload(cuda_lib, w, c, K_host, V_host, L_stream, seg_rows, copy_stream=None, ws=ws)
        assert int(ws[:4].view(torch.int32).item()) == 0, "pipeline status word set"
        assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL


def test_offloaded_verify_context_shorter_than_candidates(cuda_lib):
    # L < T (and L = 0): rows with no visible position are zero, as in tf_verify_attn
    w = small_workload(B=2, ragged=False, L=16, T=6)
    c = make_case(w)
    c["seq"] = torch.tensor([3, 0], dtype=torch.int32, device="cuda")
    K_host = c["K_cpu"].contiguous().pin_memory()
    V_host = c["V_cpu"].contiguous().pin_memory()
    out = run_offload(cuda_lib, w, c, K_host, V_host, 3, 8)
    want = O.verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), np.array([3, 0]), scale_for(w.D))
    got = out.cpu().double().numpy()
    assert np.all(got[1] == 0) and np.all(got[0, :, :3] == 0)
    assert np.abs(got - want).max() <= ATOL
