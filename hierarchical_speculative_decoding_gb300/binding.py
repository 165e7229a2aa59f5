"""Thin ctypes binding over libtriforce_attn.so (argument marshalling only).

Every function has the C entry point's name, checks dtypes/shapes/devices,
passes raw device pointers plus torch's current CUDA stream, and raises on a
non-zero status.  All arithmetic happens in the CUDA kernels; there is no CPU
path.  The library is built in-tree on first use (nvcc, sm_103a) and loading
fails loudly if it cannot be built or loaded.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_lib = None

_c = ctypes
_P = _c.c_void_p
_I = _c.c_int
_F = _c.c_float
_S = _c.c_size_t

_SIGS = {
    "tf_status_string": (_c.c_char_p, [_I]),
    "tf_check_status": (_I, [_P, _S, _P]),
    "tf_abi_version": (_I, []),
    "tf_build_chunk_means": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "tf_chunk_scores_topk_workspace": (_S, [_I, _I, _I, _I]),
    "tf_chunk_scores_topk": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _S, _P]),
    "tf_sparse_decode_attn_workspace": (_S, [_I, _I, _I, _I]),
    "tf_sparse_decode_attn": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _S, _P]),
    "tf_sparse_decode_attn_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P]),
    "tf_retrieval_draft_attn": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P]),
    "tf_verify_window_attn_workspace": (_S, [_I, _I, _I, _I, _I, _I, _I]),
    "tf_verify_window_attn": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _S, _P]),
    "tf_retrieval_draft_attn_hinted": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P,
                                            _P]),
    "tf_retrieval_window_draft_attn": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _I, _I, _P, _P,
                                            _P, _P, _P, _P]),
    "tf_stream_window_attn_workspace": (_S, [_I, _I, _I, _I, _I]),
    "tf_stream_window_attn": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _S, _P]),
    "tf_sparse_verify_attn_workspace": (_S, [_I, _I, _I, _I, _I]),
    "tf_sparse_verify_attn": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _S, _P]),
    "tf_verify_attn_workspace": (_S, [_I, _I, _I, _I, _I]),
    "tf_verify_attn": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _S, _P]),
    "tf_verify_attn_tree": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _S, _P]),
    "tf_verify_attn_offload_workspace": (_S, [_I, _I, _I, _I, _I, _I]),
    "tf_verify_attn_offload": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P, _S, _P, _P]),
    "tf_pack_retrieval_cache": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "tf_spec_accept_workspace": (_S, [_I, _I]),
    "tf_spec_accept": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _F, _P, _P, _P, _P, _S, _P]),
    "tf_debug_status": (_I, [_P, _I]),
    "tf_spec_accept_tree_workspace": (_S, [_I, _I, _I]),
    "tf_spec_accept_tree": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _F, _P, _P, _P, _P, _P, _S, _P]),
}


def debug_variant() -> bool:
    """TF_LIBRARY=debug in the environment selects the checked build of the
    library (every gather index checked, see tf_debug_status)."""
    return os.environ.get("TF_LIBRARY", "") == "debug"


def library_path() -> str:
    return _build.library(debug_variant())


def load(build_if_needed: bool = True):
    """Load (building first if needed) the CUDA library; raises if impossible."""
    global _lib
    if _lib is not None:
        return _lib
    dbg = debug_variant()
    path = _build.library(dbg)
    if build_if_needed and not _build.up_to_date(dbg):
        _build.build(debug=dbg)
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library missing: {path} (run build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def exported_symbols():
    return list(_SIGS)


class TFError(RuntimeError):
    pass


def _check(status: int, what: str):
    if status != 0:
        msg = load().tf_status_string(status).decode()
        raise TFError(f"{what} failed: status {status} ({msg})")


def _ptr(t: torch.Tensor | None):
    return None if t is None else _c.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return _c.c_void_p(s.cuda_stream)


def _need(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def _shape(t, shape, name):
    """The library reads and writes whole buffers from the sizes it is given,
    which it cannot check against the tensors: every buffer must have exactly
    the shape those sizes imply."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be {tuple(shape)}, got {tuple(t.shape)}")


def _kv_shapes(K, V, seq_lens, B, D):
    _shape(K, (B,) + tuple(K.shape[1:3]) + (D,), "K")
    _shape(V, tuple(K.shape), "V")
    _shape(seq_lens, (B,), "seq_lens")


def workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled scratch buffer (the library requires zeroed workspace once)."""
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device)


TF_ERR_DEVICE_DATA = 6


def tf_check_status(ws, stream=None) -> int:
    """Device-side status word of a verify workspace (tf_verify_attn, its tree
    and offloaded forms, tf_sparse_verify_attn).  Waits for the stream; returns
    0, or TF_ERR_DEVICE_DATA after zeroing the whole workspace again (the
    outputs computed with it since the last check are invalid)."""
    _need(ws, torch.uint8, "ws")
    status = load().tf_check_status(_ptr(ws), ws.numel(), _stream(stream))
    if status not in (0, TF_ERR_DEVICE_DATA):
        _check(status, "tf_check_status")
    return status


def tf_debug_status(clear: bool = False):
    """(status, flags): the bounds violations the checked build has recorded on
    the current device (0: none); status 2 (unsupported) from a release build."""
    flags = _c.c_uint32(0)
    status = load().tf_debug_status(_c.byref(flags), 1 if clear else 0)
    return status, int(flags.value)


def _ws(ws, need, device):
    if need == 0:
        return ws, 0
    if ws is None:
        ws = workspace(need, device)
    _need(ws, torch.uint8, "ws")
    return ws, ws.numel()


# ------------------------------------------------------------------ calls


def tf_build_chunk_means(K, seq_lens, M, chunk=8, c_begin=0, c_end=None, stream=None):
    _need(K, torch.bfloat16, "K", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(M, torch.bfloat16, "M", 4)
    B, Hkv, Lmax, D = K.shape
    Cmax = -(-Lmax // chunk)
    if tuple(M.shape) != (B, Hkv, Cmax, D):
        raise ValueError(f"M must be {(B, Hkv, Cmax, D)}")
    c_end = Cmax if c_end is None else c_end
    _check(load().tf_build_chunk_means(_ptr(K), _ptr(seq_lens), B, Hkv, Lmax, D, chunk, c_begin, c_end, _ptr(M),
                                       _stream(stream)), "tf_build_chunk_means")
    return M


def tf_chunk_scores_topk_workspace(B, Hkv, Lmax, chunk=8):
    return int(load().tf_chunk_scores_topk_workspace(B, Hkv, Lmax, chunk))


def tf_chunk_scores_topk(q, M, seq_lens, Lmax, kc, idx=None, n_sel=None, s_cut=None, ws=None, chunk=8,
                         stream=None):
    _need(q, torch.bfloat16, "q", 3)
    _need(M, torch.bfloat16, "M", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    Hkv = M.shape[1]
    if idx is None:
        idx = torch.empty((B, Hkv, kc), dtype=torch.int32, device=q.device)
    if n_sel is None:
        n_sel = torch.empty((B, Hkv), dtype=torch.int32, device=q.device)
    _need(idx, torch.int32, "idx", 3)
    _need(n_sel, torch.int32, "n_sel", 2)
    if s_cut is not None:
        _need(s_cut, torch.float32, "s_cut", 2)
    _shape(M, (B, Hkv, -(-Lmax // chunk), D), "M")
    _shape(seq_lens, (B,), "seq_lens")
    _shape(idx, (B, Hkv, kc), "idx")
    _shape(n_sel, (B, Hkv), "n_sel")
    _shape(s_cut, (B, Hkv), "s_cut")
    ws, nbytes = _ws(ws, tf_chunk_scores_topk_workspace(B, Hkv, Lmax, chunk), q.device)
    _check(load().tf_chunk_scores_topk(_ptr(q), _ptr(M), _ptr(seq_lens), B, Hq, Hkv, Lmax, D, chunk, kc, _ptr(idx),
                                       _ptr(n_sel), _ptr(s_cut), _ptr(ws), nbytes, _stream(stream)),
           "tf_chunk_scores_topk")
    return idx, n_sel


def tf_sparse_decode_attn_workspace(B, Hq, Hkv, kc):
    return int(load().tf_sparse_decode_attn_workspace(B, Hq, Hkv, kc))


def tf_sparse_decode_attn(q, K, V, seq_lens, idx, n_sel, scale, out=None, ws=None, chunk=8, stream=None):
    _need(q, torch.bfloat16, "q", 3)
    _need(K, torch.bfloat16, "K", 4)
    _need(V, torch.bfloat16, "V", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(idx, torch.int32, "idx", 3)
    _need(n_sel, torch.int32, "n_sel", 2)
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = K.shape
    kc = idx.shape[2]
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, "out", 3)
    _kv_shapes(K, V, seq_lens, B, D)
    _shape(idx, (B, Hkv, kc), "idx")
    _shape(n_sel, (B, Hkv), "n_sel")
    _shape(out, (B, Hq, D), "out")
    ws, nbytes = _ws(ws, tf_sparse_decode_attn_workspace(B, Hq, Hkv, kc), q.device)
    _check(load().tf_sparse_decode_attn(_ptr(q), _ptr(K), _ptr(V), _ptr(seq_lens), _ptr(idx), _ptr(n_sel), B, Hq,
                                        Hkv, Lmax, D, chunk, kc, float(scale), _ptr(out), _ptr(ws), nbytes,
                                        _stream(stream)), "tf_sparse_decode_attn")
    return out


def tf_pack_retrieval_cache(K, V, seq_lens, idx, n_sel, Kc=None, Vc=None, lens=None, n_chunks=None, chunk=8,
                            stream=None):
    """The retrieval drafter's rows packed into a resident buffer: for each
    (b, g) the valid tokens of the chunks idx[b, g, :n_sel[b, g]], in list
    order, from row 0 of Kc, Vc [B, Hkv, kc * chunk, D].  K and V may be CUDA
    tensors or pinned CPU tensors (read over the host link).  Returns
    (Kc, Vc, lens [B*Hkv], n_chunks [B*Hkv])."""
    for t, name in ((K, "K"), (V, "V")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 4:
            raise TypeError(f"{name} must be a 4-dim torch.bfloat16 tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not (t.is_cuda or t.is_pinned()):
            raise TypeError(f"{name} must be a CUDA tensor or pinned host memory (the library has no CPU path)")
    if V.shape != K.shape:
        raise ValueError("K and V must have the same shape")
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(idx, torch.int32, "idx", 3)
    _need(n_sel, torch.int32, "n_sel", 2)
    B, Hkv, Lmax, D = K.shape
    kc = idx.shape[2]
    dev = idx.device
    if Kc is None:
        Kc = torch.empty((B, Hkv, kc * chunk, D), dtype=torch.bfloat16, device=dev)
    if Vc is None:
        Vc = torch.empty((B, Hkv, kc * chunk, D), dtype=torch.bfloat16, device=dev)
    if lens is None:
        lens = torch.empty(B * Hkv, dtype=torch.int32, device=dev)
    if n_chunks is None:
        n_chunks = torch.empty(B * Hkv, dtype=torch.int32, device=dev)
    _need(Kc, torch.bfloat16, "Kc", 4)
    _need(Vc, torch.bfloat16, "Vc", 4)
    _need(lens, torch.int32, "lens", 1)
    _need(n_chunks, torch.int32, "n_chunks", 1)
    if Kc.shape != (B, Hkv, kc * chunk, D) or Vc.shape != Kc.shape:
        raise ValueError(f"Kc and Vc must be {(B, Hkv, kc * chunk, D)}")
    if lens.numel() != B * Hkv or n_chunks.numel() != B * Hkv:
        raise ValueError("lens and n_chunks hold one entry per (b, g)")
    _check(load().tf_pack_retrieval_cache(_ptr(K), _ptr(V), _ptr(seq_lens), _ptr(idx), _ptr(n_sel), B, Hkv, Lmax, D,
                                          chunk, kc, _ptr(Kc), _ptr(Vc), _ptr(lens), _ptr(n_chunks),
                                          _stream(stream)), "tf_pack_retrieval_cache")
    return Kc, Vc, lens, n_chunks


def tf_retrieval_draft_attn(q, M, K, V, seq_lens, kc, scale, idx=None, n_sel=None, s_cut=None, out=None, chunk=8,
                            stream=None, cut_hint=None):
    """Scores, top-k and sparse attention of the retrieval drafter in one launch.
    Returns (idx, n_sel, out); s_cut is filled when given.  cut_hint [B, Hkv]
    float32 (optional): lower bounds on the cut scores, which change only the
    time (tf_retrieval_draft_attn_hinted)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(M, torch.bfloat16, "M", 4)
    _need(K, torch.bfloat16, "K", 4)
    _need(V, torch.bfloat16, "V", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = K.shape
    if idx is None:
        idx = torch.empty((B, Hkv, kc), dtype=torch.int32, device=q.device)
    if n_sel is None:
        n_sel = torch.empty((B, Hkv), dtype=torch.int32, device=q.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(idx, torch.int32, "idx", 3)
    _need(n_sel, torch.int32, "n_sel", 2)
    _need(out, torch.float32, "out", 3)
    if s_cut is not None:
        _need(s_cut, torch.float32, "s_cut", 2)
    _kv_shapes(K, V, seq_lens, B, D)
    _shape(M, (B, Hkv, -(-Lmax // chunk), D), "M")
    _shape(idx, (B, Hkv, kc), "idx")
    _shape(n_sel, (B, Hkv), "n_sel")
    _shape(s_cut, (B, Hkv), "s_cut")
    _shape(out, (B, Hq, D), "out")
    if cut_hint is None:
        _check(load().tf_retrieval_draft_attn(_ptr(q), _ptr(M), _ptr(K), _ptr(V), _ptr(seq_lens), B, Hq, Hkv, Lmax,
                                              D, chunk, kc, float(scale), _ptr(idx), _ptr(n_sel), _ptr(s_cut),
                                              _ptr(out), _stream(stream)), "tf_retrieval_draft_attn")
    else:
        _need(cut_hint, torch.float32, "cut_hint", 2)
        if tuple(cut_hint.shape) != (B, Hkv):
            raise ValueError(f"cut_hint must be [B, Hkv] = {(B, Hkv)}, got {tuple(cut_hint.shape)}")
        _check(load().tf_retrieval_draft_attn_hinted(_ptr(q), _ptr(M), _ptr(K), _ptr(V), _ptr(seq_lens), B, Hq, Hkv,
                                                     Lmax, D, chunk, kc, float(scale), _ptr(cut_hint), _ptr(idx),
                                                     _ptr(n_sel), _ptr(s_cut), _ptr(out), _stream(stream)),
               "tf_retrieval_draft_attn_hinted")
    return idx, n_sel, out


def tf_retrieval_window_draft_attn(q, M, K, V, seq_lens, kc, scale, n_sink, window, idx=None, n_sel=None,
                                   s_cut=None, out=None, wout=None, chunk=8, stream=None, cut_hint=None):
    """The retrieval drafter (as tf_retrieval_draft_attn, cut_hint optional) and
    the sink + window attention of the same queries in one launch, for 2 to 4
    query heads per KV head.  Returns (idx, n_sel, out, wout [B, Hq, D])."""
    _need(q, torch.bfloat16, "q", 3)
    _need(M, torch.bfloat16, "M", 4)
    _need(K, torch.bfloat16, "K", 4)
    _need(V, torch.bfloat16, "V", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = K.shape
    if idx is None:
        idx = torch.empty((B, Hkv, kc), dtype=torch.int32, device=q.device)
    if n_sel is None:
        n_sel = torch.empty((B, Hkv), dtype=torch.int32, device=q.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if wout is None:
        wout = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(idx, torch.int32, "idx", 3)
    _need(n_sel, torch.int32, "n_sel", 2)
    _need(out, torch.float32, "out", 3)
    _need(wout, torch.float32, "wout", 3)
    if s_cut is not None:
        _need(s_cut, torch.float32, "s_cut", 2)
    if cut_hint is not None:
        _need(cut_hint, torch.float32, "cut_hint", 2)
    _kv_shapes(K, V, seq_lens, B, D)
    _shape(M, (B, Hkv, -(-Lmax // chunk), D), "M")
    _shape(idx, (B, Hkv, kc), "idx")
    _shape(n_sel, (B, Hkv), "n_sel")
    _shape(s_cut, (B, Hkv), "s_cut")
    _shape(cut_hint, (B, Hkv), "cut_hint")
    _shape(out, (B, Hq, D), "out")
    _shape(wout, (B, Hq, D), "wout")
    _check(load().tf_retrieval_window_draft_attn(_ptr(q), _ptr(M), _ptr(K), _ptr(V), _ptr(seq_lens), B, Hq, Hkv,
                                                 Lmax, D, chunk, kc, float(scale), _ptr(cut_hint), int(n_sink),
                                                 int(window), _ptr(idx), _ptr(n_sel), _ptr(s_cut), _ptr(out),
                                                 _ptr(wout), _stream(stream)), "tf_retrieval_window_draft_attn")
    return idx, n_sel, out, wout


def tf_sparse_verify_attn_workspace(B, Hq, Hkv, kc, T):
    return int(load().tf_sparse_verify_attn_workspace(B, Hq, Hkv, kc, T))


def tf_sparse_verify_attn(Q, K, V, seq_lens, idx, n_sel, scale, out=None, ws=None, chunk=8, stream=None):
    """Level-1 verification: T candidate queries over the retrieved chunks before
    the candidates plus the candidates themselves (chain-causal).  Q [B, Hq, T, D]."""
    _need(Q, torch.bfloat16, "Q", 4)
    _need(K, torch.bfloat16, "K", 4)
    _need(V, torch.bfloat16, "V", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(idx, torch.int32, "idx", 3)
    _need(n_sel, torch.int32, "n_sel", 2)
    B, Hq, T, D = Q.shape
    _, Hkv, Lmax, _ = K.shape
    kc = idx.shape[2]
    if out is None:
        out = torch.empty((B, Hq, T, D), dtype=torch.float32, device=Q.device)
    _need(out, torch.float32, "out", 4)
    _kv_shapes(K, V, seq_lens, B, D)
    _shape(idx, (B, Hkv, kc), "idx")
    _shape(n_sel, (B, Hkv), "n_sel")
    _shape(out, (B, Hq, T, D), "out")
    ws, nbytes = _ws(ws, tf_sparse_verify_attn_workspace(B, Hq, Hkv, kc, T), Q.device)
    _check(load().tf_sparse_verify_attn(_ptr(Q), _ptr(K), _ptr(V), _ptr(seq_lens), _ptr(idx), _ptr(n_sel), B, Hq,
                                        Hkv, Lmax, D, chunk, kc, T, float(scale), _ptr(out), _ptr(ws), nbytes,
                                        _stream(stream)), "tf_sparse_verify_attn")
    return out


def tf_sparse_decode_attn_noalloc(q, K, V, seq_lens, idx, n_sel, scale, out, chunk=8, stream=None):
    """tf_sparse_decode_attn for callers that cannot allocate: no workspace, the
    scratch is the library's static per-device buffer.  `out` must be given
    (preallocated by the caller); this wrapper allocates nothing either."""
    _need(q, torch.bfloat16, "q", 3)
    _need(K, torch.bfloat16, "K", 4)
    _need(V, torch.bfloat16, "V", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(idx, torch.int32, "idx", 3)
    _need(n_sel, torch.int32, "n_sel", 2)
    _need(out, torch.float32, "out", 3)
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = K.shape
    kc = idx.shape[2]
    _kv_shapes(K, V, seq_lens, B, D)
    _shape(idx, (B, Hkv, kc), "idx")
    _shape(n_sel, (B, Hkv), "n_sel")
    _shape(out, (B, Hq, D), "out")
    _check(load().tf_sparse_decode_attn_noalloc(_ptr(q), _ptr(K), _ptr(V), _ptr(seq_lens), _ptr(idx), _ptr(n_sel),
                                                B, Hq, Hkv, Lmax, D, chunk, kc, float(scale), _ptr(out),
                                                _stream(stream)), "tf_sparse_decode_attn_noalloc")
    return out


def tf_stream_window_attn_workspace(B, Hq, Hkv, n_sink, window):
    return int(load().tf_stream_window_attn_workspace(B, Hq, Hkv, n_sink, window))


def tf_stream_window_attn(q, K, V, seq_lens, n_sink, window, scale, out=None, ws=None, stream=None):
    _need(q, torch.bfloat16, "q", 3)
    _need(K, torch.bfloat16, "K", 4)
    _need(V, torch.bfloat16, "V", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = K.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, "out", 3)
    _kv_shapes(K, V, seq_lens, B, D)
    _shape(out, (B, Hq, D), "out")
    ws, nbytes = _ws(ws, tf_stream_window_attn_workspace(B, Hq, Hkv, n_sink, window), q.device)
    _check(load().tf_stream_window_attn(_ptr(q), _ptr(K), _ptr(V), _ptr(seq_lens), B, Hq, Hkv, Lmax, D, n_sink,
                                        window, float(scale), _ptr(out), _ptr(ws), nbytes, _stream(stream)),
           "tf_stream_window_attn")
    return out


def tf_verify_attn_workspace(B, Hq, Hkv, Lmax, T):
    return int(load().tf_verify_attn_workspace(B, Hq, Hkv, Lmax, T))


def tf_verify_attn(Q, K, V, seq_lens, scale, out=None, ws=None, stream=None):
    _need(Q, torch.bfloat16, "Q", 4)
    _need(K, torch.bfloat16, "K", 4)
    _need(V, torch.bfloat16, "V", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, T, D = Q.shape
    _, Hkv, Lmax, _ = K.shape
    if out is None:
        out = torch.empty((B, Hq, T, D), dtype=torch.float32, device=Q.device)
    _need(out, torch.float32, "out", 4)
    _kv_shapes(K, V, seq_lens, B, D)
    _shape(out, (B, Hq, T, D), "out")
    ws, nbytes = _ws(ws, tf_verify_attn_workspace(B, Hq, Hkv, Lmax, T), Q.device)
    _check(load().tf_verify_attn(_ptr(Q), _ptr(K), _ptr(V), _ptr(seq_lens), B, Hq, Hkv, Lmax, D, T, float(scale),
                                 _ptr(out), _ptr(ws), nbytes, _stream(stream)), "tf_verify_attn")
    return out


def tf_verify_window_attn_workspace(B, Hq, Hkv, Lmax, T, n_sink, window):
    return int(load().tf_verify_window_attn_workspace(B, Hq, Hkv, Lmax, T, n_sink, window))


def tf_verify_window_attn(Q, q, K, V, seq_lens, n_sink, window, scale, out=None, wout=None, ws=None, stream=None):
    """Verify attention of Q and the sink + window attention of the decode queries q
    in one call (one launch when the window rows fit the verify row groups).
    Returns (out [B, Hq, T, D], wout [B, Hq, D])."""
    _need(Q, torch.bfloat16, "Q", 4)
    _need(q, torch.bfloat16, "q", 3)
    _need(K, torch.bfloat16, "K", 4)
    _need(V, torch.bfloat16, "V", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, T, D = Q.shape
    _, Hkv, Lmax, _ = K.shape
    if tuple(q.shape) != (B, Hq, D):
        raise ValueError(f"q must be [B, Hq, D] = {(B, Hq, D)}, got {tuple(q.shape)}")
    if out is None:
        out = torch.empty((B, Hq, T, D), dtype=torch.float32, device=Q.device)
    if wout is None:
        wout = torch.empty((B, Hq, D), dtype=torch.float32, device=Q.device)
    _need(out, torch.float32, "out", 4)
    _need(wout, torch.float32, "wout", 3)
    _kv_shapes(K, V, seq_lens, B, D)
    _shape(out, (B, Hq, T, D), "out")
    _shape(wout, (B, Hq, D), "wout")
    ws, nbytes = _ws(ws, tf_verify_window_attn_workspace(B, Hq, Hkv, Lmax, T, n_sink, window), Q.device)
    _check(load().tf_verify_window_attn(_ptr(Q), _ptr(q), _ptr(K), _ptr(V), _ptr(seq_lens), B, Hq, Hkv, Lmax, D, T,
                                        int(n_sink), int(window), float(scale), _ptr(out), _ptr(wout), _ptr(ws),
                                        nbytes, _stream(stream)), "tf_verify_window_attn")
    return out, wout


def tf_verify_attn_tree(Q, K, V, seq_lens, parent, scale, out=None, ws=None, stream=None):
    """Verify attention over a candidate tree: parent [B, T] int32 (-1: the prefix)."""
    _need(Q, torch.bfloat16, "Q", 4)
    _need(K, torch.bfloat16, "K", 4)
    _need(V, torch.bfloat16, "V", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(parent, torch.int32, "parent", 2)
    B, Hq, T, D = Q.shape
    _, Hkv, Lmax, _ = K.shape
    if tuple(parent.shape) != (B, T):
        raise ValueError(f"parent must be [B, T] = [{B}, {T}], got {tuple(parent.shape)}")
    if out is None:
        out = torch.empty((B, Hq, T, D), dtype=torch.float32, device=Q.device)
    _need(out, torch.float32, "out", 4)
    _kv_shapes(K, V, seq_lens, B, D)
    _shape(out, (B, Hq, T, D), "out")
    ws, nbytes = _ws(ws, tf_verify_attn_workspace(B, Hq, Hkv, Lmax, T), Q.device)
    _check(load().tf_verify_attn_tree(_ptr(Q), _ptr(K), _ptr(V), _ptr(seq_lens), _ptr(parent), B, Hq, Hkv, Lmax, D,
                                      T, float(scale), _ptr(out), _ptr(ws), nbytes, _stream(stream)),
           "tf_verify_attn_tree")
    return out


def tf_verify_attn_offload_workspace(B, Hq, Hkv, Lmax, T, seg_rows):
    return int(load().tf_verify_attn_offload_workspace(B, Hq, Hkv, Lmax, T, seg_rows))


def tf_verify_attn_offload(Q, K_host, V_host, seq_lens, L_stream, scale, out=None, ws=None, seg_rows=16384,
                           stream=None, copy_stream=None):
    """tf_verify_attn with K and V [B, Hkv, Lmax, D] in host memory (pin it for
    asynchronous full-rate copies): positions [0, L_stream) stream through two
    device staging slots on copy_stream while the segments are attended."""
    _need(Q, torch.bfloat16, "Q", 4)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    for name, t in (("K_host", K_host), ("V_host", V_host)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 4:
            raise TypeError(f"{name} must be a 4-dim bfloat16 torch.Tensor")
        if t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous host tensor")
    B, Hq, T, D = Q.shape
    _, Hkv, Lmax, _ = K_host.shape
    if out is None:
        out = torch.empty((B, Hq, T, D), dtype=torch.float32, device=Q.device)
    _need(out, torch.float32, "out", 4)
    _kv_shapes(K_host, V_host, seq_lens, B, D)
    _shape(out, (B, Hq, T, D), "out")
    ws, nbytes = _ws(ws, tf_verify_attn_offload_workspace(B, Hq, Hkv, Lmax, T, seg_rows), Q.device)
    cs = _stream(stream)
    xs = cs if copy_stream is None else _stream(copy_stream)
    _check(load().tf_verify_attn_offload(_ptr(Q), _c.c_void_p(K_host.data_ptr()), _c.c_void_p(V_host.data_ptr()),
                                         _ptr(seq_lens), int(L_stream), B, Hq, Hkv, Lmax, D, T, float(scale), _ptr(out),
                                         int(seg_rows), _ptr(ws), nbytes, cs, xs), "tf_verify_attn_offload")
    return out


def tf_spec_accept_workspace(B, gamma):
    return int(load().tf_spec_accept_workspace(B, gamma))


def tf_spec_accept(tgt_logits, drf_logits, drf_tokens, u_acc, u_res, temperature=1.0, n_acc=None, next_token=None,
                   out_tokens=None, ws=None, stream=None):
    _need(tgt_logits, torch.float32, "tgt_logits", 3)
    B, g1, Vn = tgt_logits.shape
    gamma = g1 - 1
    _need(u_res, torch.float32, "u_res", 1)
    if gamma > 0:
        _need(drf_logits, torch.float32, "drf_logits", 3)
        _need(drf_tokens, torch.int32, "drf_tokens", 2)
        _need(u_acc, torch.float32, "u_acc", 2)
        if tuple(drf_logits.shape) != (B, gamma, Vn) or tuple(drf_tokens.shape) != (B, gamma):
            raise ValueError("draft shapes must be [B, gamma, V] and [B, gamma]")
        _shape(u_acc, (B, gamma), "u_acc")
    _shape(u_res, (B,), "u_res")
    dev = tgt_logits.device
    if n_acc is None:
        n_acc = torch.empty((B,), dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    for t, name, shape in ((n_acc, "n_acc", (B,)), (next_token, "next_token", (B,)),
                           (out_tokens, "out_tokens", (B, gamma + 1))):
        _need(t, torch.int32, name, len(shape))
        _shape(t, shape, name)
    ws, nbytes = _ws(ws, tf_spec_accept_workspace(B, gamma), dev)
    _check(load().tf_spec_accept(_ptr(tgt_logits), _ptr(drf_logits if gamma > 0 else None),
                                 _ptr(drf_tokens if gamma > 0 else None), _ptr(u_acc if gamma > 0 else None),
                                 _ptr(u_res), B, gamma, Vn, float(temperature), _ptr(n_acc), _ptr(next_token),
                                 _ptr(out_tokens), _ptr(ws), nbytes, _stream(stream)), "tf_spec_accept")
    return n_acc, next_token, out_tokens


def tf_spec_accept_tree_workspace(B, T, V):
    return int(load().tf_spec_accept_tree_workspace(B, T, V))


def tf_spec_accept_tree(tgt_logits, drf_logits, drf_tokens, parent, u_acc, u_res, temperature=1.0, n_acc=None,
                        next_token=None, out_tokens=None, acc_nodes=None, ws=None, stream=None):
    """Accept / resample over a candidate tree: tgt_logits [B, T+1, V] (row 1+j
    after candidate j), drf_logits [B, T, V] (row j the distribution candidate j
    was drawn from), drf_tokens / parent / u_acc [B, T], u_res [B].  Returns
    (n_acc, next_token, out_tokens [B, T+1], acc_nodes [B, T])."""
    _need(tgt_logits, torch.float32, "tgt_logits", 3)
    B, t1, Vn = tgt_logits.shape
    T = t1 - 1
    _need(u_res, torch.float32, "u_res", 1)
    if T > 0:
        _need(drf_logits, torch.float32, "drf_logits", 3)
        _need(drf_tokens, torch.int32, "drf_tokens", 2)
        _need(parent, torch.int32, "parent", 2)
        _need(u_acc, torch.float32, "u_acc", 2)
        if tuple(drf_logits.shape) != (B, T, Vn) or tuple(drf_tokens.shape) != (B, T) or \
                tuple(parent.shape) != (B, T) or tuple(u_acc.shape) != (B, T):
            raise ValueError("tree shapes must be [B, T, V] for drf_logits and [B, T] for tokens, parent, u_acc")
    dev = tgt_logits.device
    if n_acc is None:
        n_acc = torch.empty((B,), dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, T + 1), dtype=torch.int32, device=dev)
    if acc_nodes is None:
        acc_nodes = torch.empty((B, max(T, 1)), dtype=torch.int32, device=dev)
    _shape(u_res, (B,), "u_res")
    for t, name, shape in ((n_acc, "n_acc", (B,)), (next_token, "next_token", (B,)),
                           (out_tokens, "out_tokens", (B, T + 1)), (acc_nodes, "acc_nodes", (B, max(T, 1)))):
        _need(t, torch.int32, name, len(shape))
        _shape(t, shape, name)
    ws, nbytes = _ws(ws, tf_spec_accept_tree_workspace(B, T, Vn), dev)
    g = T > 0
    _check(load().tf_spec_accept_tree(_ptr(tgt_logits), _ptr(drf_logits if g else None),
                                      _ptr(drf_tokens if g else None), _ptr(parent if g else None),
                                      _ptr(u_acc if g else None), _ptr(u_res), B, T, Vn, float(temperature),
                                      _ptr(n_acc), _ptr(next_token), _ptr(out_tokens), _ptr(acc_nodes), _ptr(ws),
                                      nbytes, _stream(stream)), "tf_spec_accept_tree")
    return n_acc, next_token, out_tokens, acc_nodes
