"""The C-ABI library builds, loads and exports every declared symbol (no GPU).

Only calls that return before touching the GPU are made here: status strings,
the ABI version, workspace-size queries and host-side argument validation.
"""

import ctypes
import os
import re
import sys

import pytest

from hierarchical_speculative_decoding_gb300 import binding, build

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_symbols():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if fn.endswith(".h"):
            with open(os.path.join(HEADER_DIR, fn)) as f:
                names += re.findall(r"^TF_API\s+[\w\s\*]+?\b(tf_\w+)\s*\(", f.read(), flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load(build_if_needed=False)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(binding.exported_symbols())


def test_version_and_status_strings(lib):
    assert lib.tf_abi_version() == 101
    for s in range(7):
        assert len(lib.tf_status_string(s)) > 0
    assert lib.tf_status_string(99) == b"unknown status"


def test_workspace_sizes(lib):
    assert lib.tf_chunk_scores_topk_workspace(1, 32, 131072, 8) == 0  # selection stays on chip
    assert lib.tf_sparse_decode_attn_workspace(1, 32, 32, 512) > 0
    assert lib.tf_sparse_decode_attn_workspace(1, 32, 5, 512) == 0  # Hq % Hkv != 0
    assert lib.tf_stream_window_attn_workspace(4, 32, 8, 4, 252) > 0
    assert lib.tf_verify_attn_workspace(4, 32, 8, 131072, 6) > 0
    assert lib.tf_spec_accept_workspace(8, 5) >= 8 * 11 * 12
    # normalisers of 2T+1 rows and two vocabulary rows per sequence
    assert lib.tf_spec_accept_tree_workspace(8, 6, 32000) >= 8 * 13 * 12 + 8 * 2 * 32000 * 4
    assert lib.tf_spec_accept_tree_workspace(8, -1, 32000) == 0
    assert lib.tf_sparse_verify_attn_workspace(1, 32, 32, 512, 6) > 0
    assert lib.tf_verify_attn_offload_workspace(1, 32, 32, 131072, 6, 16384) > 0
    assert lib.tf_verify_attn_offload_workspace(1, 32, 32, 131072, 6, 0) == 0
    # the staging slots and the per-segment states grow with the segment count and size
    assert (lib.tf_verify_attn_offload_workspace(1, 32, 32, 131072, 6, 8192) <
            lib.tf_verify_attn_offload_workspace(1, 32, 32, 131072, 6, 16384))
    # workspace grows with the problem
    assert lib.tf_verify_attn_workspace(8, 32, 8, 131072, 6) > lib.tf_verify_attn_workspace(1, 32, 8, 131072, 6)


def test_host_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: every call below fails validation first
    odd = P(0x10008)  # not 16-byte aligned
    null = None
    INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3
    assert lib.tf_build_chunk_means(null, fake, 1, 1, 64, 128, 8, 0, 8, fake, None) == INVALID
    assert lib.tf_build_chunk_means(odd, fake, 1, 1, 64, 128, 8, 0, 8, fake, None) == INVALID
    assert lib.tf_build_chunk_means(fake, fake, 1, 1, 64, 64, 8, 0, 8, fake, None) == UNSUPPORTED
    assert lib.tf_build_chunk_means(fake, fake, 1, 1, 64, 128, 8, 0, 9, fake, None) == INVALID
    assert lib.tf_chunk_scores_topk(fake, fake, fake, 1, 6, 4, 64, 128, 8, 4, fake, fake, null, null, 0,
                                    None) == INVALID  # Hq % Hkv
    assert lib.tf_chunk_scores_topk(fake, fake, fake, 1, 8, 4, 64, 128, 8, 0, fake, fake, null, null, 0,
                                    None) == INVALID  # kc = 0
    assert lib.tf_sparse_decode_attn(fake, fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 4, 0.1, fake, null,
                                     0, None) == WORKSPACE
    assert lib.tf_sparse_decode_attn(fake, fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 16, 4, 0.1, fake, null,
                                     0, None) == UNSUPPORTED
    assert lib.tf_stream_window_attn(fake, fake, fake, fake, 1, 8, 2, 64, 128, -1, 4, 0.1, fake, null, 0,
                                     None) == INVALID
    assert lib.tf_verify_attn(fake, fake, fake, fake, 1, 8, 2, 64, 128, 0, 0.1, fake, null, 0, None) == INVALID
    assert lib.tf_verify_attn(fake, fake, fake, fake, 1, 8, 2, 64, 128, 17, 0.1, fake, null, 0, None) == UNSUPPORTED
    # fused retrieval drafter: q, M, K, V, seq_lens, B, Hq, Hkv, Lmax, D, chunk, kc, scale, idx, n_sel, s_cut, out
    assert lib.tf_retrieval_draft_attn(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 2049, 0.1, fake, fake, null,
                                       fake, None) == UNSUPPORTED  # kc above the on-chip list
    assert lib.tf_retrieval_draft_attn(fake, fake, fake, fake, fake, 1, 16, 2, 64, 128, 8, 64, 0.1, fake, fake, null,
                                       fake, None) == UNSUPPORTED  # 8 query heads per group
    assert lib.tf_retrieval_draft_attn(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 64, 0.1, fake, fake, null,
                                       null, None) == INVALID  # no output
    assert lib.tf_retrieval_draft_attn(fake, odd, fake, fake, fake, 1, 8, 2, 64, 128, 8, 64, 0.1, fake, fake, null,
                                       fake, None) == INVALID  # misaligned means
    assert lib.tf_retrieval_draft_attn(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 16, 64, 0.1, fake, fake, null,
                                       fake, None) == UNSUPPORTED  # chunk 16
    # verify + window in one launch: Q, q, K, V, seq, B, Hq, Hkv, Lmax, D, T, n_sink, window, scale, out, wout, ws, bytes, s
    vw = lib.tf_verify_window_attn
    assert vw(fake, null, fake, fake, fake, 1, 8, 2, 64, 128, 6, 4, 252, 0.1, fake, fake, fake, 1 << 30,
              None) == INVALID  # no window queries
    assert vw(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 6, 4, 252, 0.1, fake, null, fake, 1 << 30,
              None) == INVALID  # no window output
    assert vw(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 17, 4, 252, 0.1, fake, fake, fake, 1 << 30,
              None) == UNSUPPORTED  # T > 16
    assert vw(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 6, -1, 252, 0.1, fake, fake, fake, 1 << 30,
              None) == INVALID  # negative sink count
    assert vw(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 6, 4, 252, 0.1, fake, fake, fake, 0,
              None) == WORKSPACE
    # window rows in the verify launch when they fill padding rows: 4 x 6 verify rows -> 4 x 7 (24-row kernel)
    # and 8 x 5 -> 8 x 6 (two groups, 32-row kernel); not 4 x 6 -> 4 x 7 (24 -> 32 rows) nor 4 x 8 -> 4 x 9
    # (a second group): the window launched apart, its scratch after the verify's
    for G, T in ((4, 5), (8, 5), (1, 6), (1, 15)):  # the verify scratch of G * (T + 1) rows
        assert lib.tf_verify_window_attn_workspace(1, 2 * G, 2, 64, T, 4, 252) == \
            lib.tf_verify_attn_workspace(1, 2 * G, 2, 64, T + 1)
    for G, T in ((4, 6), (4, 8), (8, 4), (1, 8), (1, 16)):
        vsz = lib.tf_verify_attn_workspace(1, 2 * G, 2, 64, T)
        assert lib.tf_verify_window_attn_workspace(1, 2 * G, 2, 64, T, 4, 252) == \
            -(-vsz // 256) * 256 + lib.tf_stream_window_attn_workspace(1, 2 * G, 2, 4, 252)
    vsz = lib.tf_verify_attn_workspace(1, 8, 2, 64, 8)
    assert vw(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 4, 252, 0.1, fake, fake, fake, vsz,
              None) == WORKSPACE  # room for the verify scratch only
    assert vw(fake, fake, fake, fake, fake, 0, 8, 2, 64, 128, 6, 4, 252, 0.1, fake, fake, null, 0,
              None) == 0  # empty batch: nothing to do, nothing launched
    assert lib.tf_verify_window_attn_workspace(1, 8, 2, 64, 6, -1, 252) == 0
    # retrieval draft + window in one launch: ... scale, hint, n_sink, window, idx, n_sel, s_cut, out, wout, stream
    wd = lib.tf_retrieval_window_draft_attn
    assert wd(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 64, 0.1, null, 4, 252, fake, fake, null, fake,
              null, None) == INVALID  # no window output
    assert wd(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 64, 0.1, null, -1, 252, fake, fake, null, fake,
              fake, None) == INVALID  # negative sink count
    assert wd(fake, fake, fake, fake, fake, 1, 8, 8, 64, 128, 8, 64, 0.1, null, 4, 252, fake, fake, null, fake,
              fake, None) == UNSUPPORTED  # one query head: the window rides in the verify launch instead
    assert wd(fake, fake, fake, fake, fake, 1, 16, 2, 64, 128, 8, 64, 0.1, null, 4, 252, fake, fake, null, fake,
              fake, None) == UNSUPPORTED  # eight query heads per KV head
    assert wd(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 2020, 0.1, null, 4, 252, fake, fake, null, fake,
              fake, None) == UNSUPPORTED  # the chunk list cannot take kc chunks plus the window pieces
    # the same with a cut hint (before idx): required, and the same limits
    hd = lib.tf_retrieval_draft_attn_hinted
    assert hd(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 64, 0.1, null, fake, fake, null, fake,
              None) == INVALID  # no hint array
    assert hd(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 2049, 0.1, fake, fake, fake, null, fake,
              None) == UNSUPPORTED
    assert hd(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 64, 0.1, fake, fake, fake, null, null,
              None) == INVALID  # no output
    # sparse verification: Q, K, V, seq, idx, n_sel, B, Hq, Hkv, Lmax, D, chunk, kc, T, scale, out, ws, bytes, s
    sv = lib.tf_sparse_verify_attn
    big = 1 << 30
    assert sv(fake, fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 16, 17, 0.1, fake, fake, big,
              None) == UNSUPPORTED  # T > 16
    assert sv(fake, fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 16, 0, 0.1, fake, fake, big,
              None) == INVALID  # T = 0
    assert sv(fake, fake, fake, fake, null, fake, 1, 8, 2, 64, 128, 8, 16, 4, 0.1, fake, fake, big,
              None) == INVALID  # no ids
    assert sv(fake, fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 8, 16, 4, 0.1, fake, null, 0,
              None) == WORKSPACE
    # tree verify: Q, K, V, seq, parent, B, Hq, Hkv, Lmax, D, T, scale, out, ws, bytes, stream
    tv = lib.tf_verify_attn_tree
    assert tv(fake, fake, fake, fake, null, 1, 8, 2, 64, 128, 4, 0.1, fake, fake, big, None) == INVALID  # no tree
    assert tv(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 17, 0.1, fake, fake, big, None) == UNSUPPORTED
    assert tv(fake, fake, fake, fake, fake, 1, 8, 2, 64, 128, 4, 0.1, fake, null, 0, None) == WORKSPACE
    # offloaded verify: Q, K_host, V_host, seq, L_stream, B, Hq, Hkv, Lmax, D, T, scale, out, seg_rows,
    # ws, bytes, stream, copy_stream
    ov = lib.tf_verify_attn_offload
    assert ov(fake, fake, fake, fake, 65, 1, 8, 2, 64, 128, 4, 0.1, fake, 32, fake, big, None, None) == INVALID
    assert ov(fake, fake, fake, fake, 64, 1, 8, 2, 64, 128, 4, 0.1, fake, 0, fake, big, None, None) == INVALID
    assert ov(fake, null, fake, fake, 64, 1, 8, 2, 64, 128, 4, 0.1, fake, 32, fake, big, None, None) == INVALID
    assert ov(fake, fake, fake, fake, 64, 1, 8, 2, 64, 128, 17, 0.1, fake, 32, fake, big, None, None) == UNSUPPORTED
    assert ov(fake, fake, fake, fake, 64, 1, 8, 2, 64, 128, 4, 0.1, fake, 32, null, 0, None, None) == WORKSPACE
    assert lib.tf_spec_accept(fake, fake, fake, fake, fake, 1, 4, 100, 0.0, fake, fake, null, fake, 4096,
                              None) == INVALID
    assert lib.tf_spec_accept(fake, null, fake, fake, fake, 1, 4, 100, 1.0, fake, fake, null, fake, 4096,
                              None) == INVALID
    assert lib.tf_spec_accept(fake, fake, fake, fake, fake, 1, 4, 100, 1.0, fake, fake, null, null, 0,
                              None) == WORKSPACE
    # tree accept: tgt, drf, tokens, parent, u_acc, u_res, B, T, V, temperature, n_acc, next, out, nodes, ws, bytes
    ta = lib.tf_spec_accept_tree
    assert ta(fake, fake, fake, null, fake, fake, 1, 4, 100, 1.0, fake, fake, null, null, fake, big,
              None) == INVALID  # no tree
    assert ta(fake, fake, fake, fake, fake, fake, 1, 4, 100, 0.0, fake, fake, null, null, fake, big,
              None) == INVALID  # temperature
    assert ta(fake, fake, fake, fake, fake, fake, 1, -1, 100, 1.0, fake, fake, null, null, fake, big,
              None) == INVALID  # T < 0
    assert ta(fake, fake, fake, fake, fake, fake, 1, 4, 100, 1.0, fake, fake, null, null, fake,
              lib.tf_spec_accept_tree_workspace(1, 4, 100) - 1, None) == WORKSPACE
    assert ta(fake, fake, fake, fake, fake, fake, 0, 4, 100, 1.0, fake, fake, null, null, null, 0,
              None) == 0  # B = 0: no work
    pk = lib.tf_pack_retrieval_cache
    assert pk(null, fake, fake, fake, fake, 1, 2, 64, 128, 8, 4, fake, fake, fake, fake, None) == INVALID
    assert pk(fake, fake, fake, fake, fake, 1, 2, 64, 128, 8, 4, odd, fake, fake, fake, None) == INVALID
    assert pk(fake, fake, fake, fake, fake, 1, 0, 64, 128, 8, 4, fake, fake, fake, fake, None) == INVALID  # Hkv
    assert pk(fake, fake, fake, fake, fake, 1, 2, 64, 64, 8, 4, fake, fake, fake, fake, None) == UNSUPPORTED
    assert pk(fake, fake, fake, fake, fake, 1, 2, 64, 128, 8, 4097, fake, fake, fake, fake, None) == UNSUPPORTED
    assert pk(fake, fake, fake, fake, fake, 0, 2, 64, 128, 8, 4, fake, fake, fake, fake, None) == 0  # B = 0: no work
    # the release build keeps no bounds-check words
    flags = ctypes.c_uint32(7)
    assert lib.tf_debug_status(ctypes.byref(flags), 0) == UNSUPPORTED and flags.value == 0
    assert lib.tf_debug_status(null, 0) == INVALID
    # the status query reads nothing without a workspace of at least one word
    assert lib.tf_check_status(null, 4096, None) == INVALID
    assert lib.tf_check_status(fake, 3, None) == INVALID


def test_binding_rejects_cpu_tensors():
    import torch

    K = torch.zeros((1, 1, 8, 128), dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="CUDA"):
        binding.tf_build_chunk_means(K, torch.zeros(1, dtype=torch.int32), torch.zeros((1, 1, 1, 128),
                                                                                      dtype=torch.bfloat16))


def test_bench_mirrors_the_one_launch_rule(lib):
    """bench.py counts tf_verify_window_attn's launches with its own copy of the
    library's rule; the workspace query tells the two paths apart (one launch:
    the verify scratch of G*(T+1) rows; two: the verify scratch of G*T rows plus
    the window's)."""
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    for G in (1, 2, 3, 4, 5, 6, 8):
        for T in range(1, 17):
            one = lib.tf_verify_window_attn_workspace(1, 2 * G, 2, 64, T, 4, 252) == \
                lib.tf_verify_attn_workspace(1, 2 * G, 2, 64, T + 1)
            assert one == (bench.window_launches(G, T) == 1), (G, T)
    assert bench.window_launches(1, 6) == 1 and bench.window_launches(4, 6) == 2
