"""tf_check_status on the GB300: a clean verify workspace reads TF_OK; a status
word set from the host (standing in for a kernel's timeout flag, which only a
hardware fault raises) reads TF_ERR_DEVICE_DATA, the whole workspace comes
back zeroed, and the next verify on it matches the oracle again."""

import numpy as np
import pytest
import torch

from oracle import triforce as O
from test_gpu_parity import ATOL, bits, make_case, scale_for, small_workload

pytestmark = pytest.mark.gpu


def test_status_word_round_trip(cuda_lib):
    w = small_workload(L=1500, L_min=600)
    c = make_case(w)
    nbytes = cuda_lib.tf_verify_attn_workspace(w.B, w.Hq, w.Hkv, w.L, w.T)
    ws = cuda_lib.workspace(nbytes, "cuda")
    want = O.verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(), scale_for(w.D))

    out = cuda_lib.tf_verify_attn(c["Q"], c["K"], c["V"], c["seq"], scale_for(w.D), ws=ws)
    assert cuda_lib.tf_check_status(ws) == 0
    assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL

    ws[:4].view(torch.int32).fill_(7)  # a flagged device error
    ws[-16:].fill_(0xAB)  # and left-over state elsewhere in the workspace
    assert cuda_lib.tf_check_status(ws) == cuda_lib.TF_ERR_DEVICE_DATA
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0

    out = cuda_lib.tf_verify_attn(c["Q"], c["K"], c["V"], c["seq"], scale_for(w.D), ws=ws)
    assert cuda_lib.tf_check_status(ws) == 0
    assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL
