"""Thin ctypes binding of libmsa.so: argument marshalling only.

Every function has the name of the C entry point it calls (include/msa.h), takes torch
tensors that already live on the GPU (bf16 for activations, fp32 for M/LSE, int32 for block
indices, int64 for cu_seqlens), checks dtypes/shapes/contiguity, and passes data pointers,
sizes and the current CUDA stream.  All arithmetic happens in the CUDA kernels; there is no
fallback of any kind: if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa.so")

STATUS = {0: "MSA_OK", 1: "MSA_ERR_INVALID_ARGUMENT", 2: "MSA_ERR_UNSUPPORTED",
          3: "MSA_ERR_WORKSPACE", 4: "MSA_ERR_CUDA", 5: "MSA_ERR_TIMEOUT"}


class MSAError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s returned %s" % (fn, STATUS.get(code, code)))
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libmsa.so not built (run __graft_entry__.build() or "
                          "python block_sparse_gqa_scores_gb300/_build.py)")
    L = ctypes.CDLL(LIB_PATH)
    P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.msa_status_string.argtypes = [i32]
    L.msa_status_string.restype = ctypes.c_char_p
    L.msa_index_block_scores.argtypes = [P, P, P, i64, i32, i32, i32, i64, i64, P]
    L.msa_select_blocks.argtypes = [P, P, i64, i32, i32, i32, i64, i64, P]
    L.msa_index_select.argtypes = [P, P, P, i64, i32, i32, i32, i32, i64, i64, P]
    L.msa_sparse_attn_fwd_workspace.argtypes = [i64, i32, i32, i32, i32]
    L.msa_sparse_attn_fwd_workspace.restype = sz
    L.msa_sparse_attn_fwd.argtypes = [P, P, P, P, P, P, i64, i32, i32, i32, i32, i32, P, sz, P]
    L.msa_sparse_attn_bwd_workspace.argtypes = [i64, i32, i32, i32, i32]
    L.msa_sparse_attn_bwd_workspace.restype = sz
    L.msa_sparse_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, i64, i32, i32, i32, i32, i32,
                                      P, sz, P]
    L.msa_sparse_decode_workspace.argtypes = [i32, i64, i32, i32, i32, i32, i32]
    L.msa_sparse_decode_workspace.restype = sz
    L.msa_sparse_decode.argtypes = [P, P, P, P, P, P, i32, i64, i32, i32, i32, i32, i32, i32, P, P,
                                    P, P, sz, P]
    L.msa_sparse_decode_noalloc.argtypes = [P, P, P, P, P, P, i32, i64, i32, i32, i32, i32, i32,
                                            i32, P, P, P, P]
    L.msa_sparse_decode_paged.argtypes = [P, P, P, P, P, P, P, i32, i64, i64, i64, i32, i32, i32,
                                          i32, i32, i32, P, P, P, P, sz, P]
    L.msa_prefill_varlen_workspace.argtypes = [P, i32, i32, i32, i32, i32]
    L.msa_prefill_varlen_workspace.restype = sz
    L.msa_prefill_varlen.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, P, P, P,
                                     P, sz, P]
    L.msa_kl_loss_fwd_workspace.argtypes = [i64, i32, i32]
    L.msa_kl_loss_fwd_workspace.restype = sz
    L.msa_kl_loss_fwd.argtypes = [P, P, P, P, P, P, P, P, P, i64, i32, i32, i32, i32, i32, i32, P,
                                  sz, P]
    L.msa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.msa_kl_loss_bwd_workspace.argtypes = [i64, i32, i32, i32]
    L.msa_kl_loss_bwd_workspace.restype = sz
    L.msa_kl_loss_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, i64, i32, i32, i32, i32, i32,
                                  i32, P, sz, P]
    for fn in ("msa_index_block_scores", "msa_select_blocks", "msa_index_select", "msa_sparse_attn_fwd",
               "msa_sparse_attn_bwd",
               "msa_sparse_decode", "msa_sparse_decode_noalloc", "msa_sparse_decode_paged",
               "msa_prefill_varlen",
               "msa_kl_loss_fwd", "msa_kl_loss_bwd",
               "msa_device_status", "msa_set_wait_limit_ns"):
        getattr(L, fn).restype = i32
    return L


lib = _load()

BLOCK = 64


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, code):
    if code != 0:
        raise MSAError(fn, code)


def _req(t, dtype, ndim, name, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype or t.dim() != ndim or not t.is_contiguous() or not t.is_cuda:
        raise ValueError("%s must be a contiguous %dD %s CUDA tensor, got %s %s %s" % (
            name, ndim, dtype, tuple(t.shape), t.dtype, t.device))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if device is not None and t.device != device:
        raise ValueError("%s must be on %s, got %s" % (name, device, t.device))


def _decode_outputs(q, q_idx, k, o, lse, idx_out, alloc):
    """Checks (or, with alloc, creates) the decode outputs: o like q, lse [S, H_q] fp32 and
    idx_out [S, H_kv, k] int32, all on q's device (a smaller buffer would be written past its
    end by the kernels)."""
    S, H_q, _ = q.shape
    H_kv = q_idx.shape[1]
    if alloc and o is None:
        o = torch.empty_like(q)
    if alloc and lse is None:
        lse = torch.empty((S, H_q), dtype=torch.float32, device=q.device)
    if alloc and idx_out is None:
        idx_out = torch.empty((S, H_kv, k), dtype=torch.int32, device=q.device)
    _req(o, torch.bfloat16, 3, "o", q.shape, q.device)
    _req(lse, torch.float32, 2, "lse", (S, H_q), q.device)
    if idx_out is not None:
        _req(idx_out, torch.int32, 3, "idx_out", (S, H_kv, k), q.device)
    return o, lse, idx_out


def msa_index_block_scores(q_idx, k_idx, M=None, q_start=0, q_count=None, block_size=BLOCK,
                           stream=None):
    """Block scores M [H_kv, q_count, ceil(N/64)] fp32 of rows [q_start, q_start+q_count)."""
    _req(q_idx, torch.bfloat16, 3, "q_idx")
    _req(k_idx, torch.bfloat16, 2, "k_idx")
    N, H_kv, d_idx = q_idx.shape
    q_count = N - q_start if q_count is None else q_count
    nblk = -(-N // block_size)
    if M is None:
        M = torch.empty((H_kv, q_count, nblk), dtype=torch.float32, device=q_idx.device)
    _req(M, torch.float32, 3, "M")
    _check("msa_index_block_scores", lib.msa_index_block_scores(
        _ptr(q_idx), _ptr(k_idx), _ptr(M), N, H_kv, d_idx, block_size, q_start, q_count,
        _stream(stream)))
    return M


def msa_select_blocks(M, N, k, idx=None, q_start=0, block_size=BLOCK, stream=None):
    """Selected blocks idx [H_kv, N, k] int32 (rows q_start..q_start+q_count-1 written)."""
    _req(M, torch.float32, 3, "M")
    H_kv, q_count, _ = M.shape
    if idx is None:
        idx = torch.full((H_kv, N, k), -2, dtype=torch.int32, device=M.device)
    _req(idx, torch.int32, 3, "idx")
    _check("msa_select_blocks", lib.msa_select_blocks(
        _ptr(M), _ptr(idx), N, H_kv, block_size, k, q_start, q_count, _stream(stream)))
    return idx


def msa_index_select(q_idx, k_idx, k, idx=None, q_start=0, q_count=None, block_size=BLOCK,
                     stream=None):
    """Selected blocks idx [H_kv, N, k] int32 straight from Q_idx, K_idx (no M); rows
    q_start..q_start+q_count-1 written."""
    _req(q_idx, torch.bfloat16, 3, "q_idx")
    _req(k_idx, torch.bfloat16, 2, "k_idx")
    N, H_kv, d_idx = q_idx.shape
    q_count = N - q_start if q_count is None else q_count
    if idx is None:
        idx = torch.full((H_kv, N, k), -2, dtype=torch.int32, device=q_idx.device)
    _req(idx, torch.int32, 3, "idx")
    _check("msa_index_select", lib.msa_index_select(
        _ptr(q_idx), _ptr(k_idx), _ptr(idx), N, H_kv, d_idx, block_size, k, q_start, q_count,
        _stream(stream)))
    return idx


def msa_sparse_attn_fwd_workspace(N, H_q, H_kv, d_h, k):
    return int(lib.msa_sparse_attn_fwd_workspace(N, H_q, H_kv, d_h, k))


def msa_sparse_attn_fwd(q, k, v, idx, o=None, lse=None, ws=None, block_size=BLOCK, stream=None):
    """Main branch: O [N, H_q, d_h] bf16 and LSE [H_q, N] fp32 over the selected blocks."""
    _req(q, torch.bfloat16, 3, "q")
    _req(k, torch.bfloat16, 3, "k")
    _req(v, torch.bfloat16, 3, "v")
    _req(idx, torch.int32, 3, "idx")
    N, H_q, d_h = q.shape
    H_kv = k.shape[1]
    kk = idx.shape[2]
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H_q, N), dtype=torch.float32, device=q.device)
    nws = msa_sparse_attn_fwd_workspace(N, H_q, H_kv, d_h, kk)
    if ws is None and nws:
        ws = torch.empty(nws, dtype=torch.uint8, device=q.device)
    _check("msa_sparse_attn_fwd", lib.msa_sparse_attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(o), _ptr(lse), N, H_q, H_kv, d_h, block_size,
        kk, _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))
    return o, lse


def msa_sparse_attn_bwd_workspace(N, H_q, H_kv, d_h, k):
    return int(lib.msa_sparse_attn_bwd_workspace(N, H_q, H_kv, d_h, k))


def msa_sparse_attn_bwd(q, k, v, idx, o, lse, d_o, dq=None, dk=None, dv=None, ws=None,
                        block_size=BLOCK, stream=None):
    """Main-branch gradients for upstream d_o: (dq [N,H_q,d_h], dk, dv [N,H_kv,d_h]) fp32, from
    the forward's o and lse on the same q, k, v, idx."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (d_o, "d_o")):
        _req(t, torch.bfloat16, 3, n, device=q.device)
    _req(idx, torch.int32, 3, "idx", device=q.device)
    N, H_q, d_h = q.shape
    H_kv = k.shape[1]
    kk = idx.shape[2]
    _req(o, torch.bfloat16, 3, "o", q.shape)
    _req(d_o, torch.bfloat16, 3, "d_o", q.shape)
    _req(lse, torch.float32, 2, "lse", (H_q, N), q.device)
    if dq is None:
        dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if dk is None:
        dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    if dv is None:
        dv = torch.empty(v.shape, dtype=torch.float32, device=q.device)
    _req(dq, torch.float32, 3, "dq", q.shape, q.device)
    _req(dk, torch.float32, 3, "dk", k.shape, q.device)
    _req(dv, torch.float32, 3, "dv", v.shape, q.device)
    if ws is None:
        ws = torch.empty(max(16, msa_sparse_attn_bwd_workspace(N, H_q, H_kv, d_h, kk)),
                         dtype=torch.uint8, device=q.device)
    _check("msa_sparse_attn_bwd", lib.msa_sparse_attn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(o), _ptr(lse), _ptr(d_o), _ptr(dq), _ptr(dk),
        _ptr(dv), N, H_q, H_kv, d_h, block_size, kk, _ptr(ws), ws.numel(), _stream(stream)))
    return dq, dk, dv


def msa_sparse_decode_workspace(S, max_len, H_q, H_kv, d_h, d_idx, k):
    return int(lib.msa_sparse_decode_workspace(S, max_len, H_q, H_kv, d_h, d_idx, k))


def msa_sparse_decode(q, q_idx, k_cache, v_cache, k_idx_cache, cu_seqlens, max_len, k,
                      o=None, lse=None, idx_out=None, ws=None, block_size=BLOCK, stream=None):
    """Decode one new query per sequence -> (O [S,H_q,d_h] bf16, LSE [S,H_q] fp32, idx)."""
    _req(q, torch.bfloat16, 3, "q")
    _req(q_idx, torch.bfloat16, 3, "q_idx")
    _req(k_cache, torch.bfloat16, 3, "k_cache")
    _req(v_cache, torch.bfloat16, 3, "v_cache")
    _req(k_idx_cache, torch.bfloat16, 2, "k_idx_cache")
    _req(cu_seqlens, torch.int64, 1, "cu_seqlens")
    S, H_q, d_h = q.shape
    H_kv, d_idx = q_idx.shape[1], q_idx.shape[2]
    for t, n in ((q_idx, "q_idx"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (k_idx_cache, "k_idx_cache"), (cu_seqlens, "cu_seqlens")):
        _req(t, t.dtype, t.dim(), n, device=q.device)
    o, lse, idx_out = _decode_outputs(q, q_idx, k, o, lse, idx_out, alloc=True)
    nws = msa_sparse_decode_workspace(S, max_len, H_q, H_kv, d_h, d_idx, k)
    if ws is None:
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=q.device)
    _check("msa_sparse_decode", lib.msa_sparse_decode(
        _ptr(q), _ptr(q_idx), _ptr(k_cache), _ptr(v_cache), _ptr(k_idx_cache), _ptr(cu_seqlens),
        S, max_len, H_q, H_kv, d_h, d_idx, block_size, k, _ptr(o), _ptr(lse), _ptr(idx_out),
        _ptr(ws), ws.numel(), _stream(stream)))
    return o, lse, idx_out


def msa_sparse_decode_noalloc(q, q_idx, k_cache, v_cache, k_idx_cache, cu_seqlens, max_len, k,
                              o, lse, idx_out=None, block_size=BLOCK, stream=None):
    """msa_sparse_decode for callers that cannot allocate where they decode: the library's fixed
    device scratch replaces the workspace, and the outputs o [S,H_q,d_h] bf16 and
    lse [S,H_q] fp32 (and optionally idx_out [S,H_kv,k] int32) must be passed in.  Calls that
    overlap on the GPU share that scratch and must be serialised."""
    _req(q, torch.bfloat16, 3, "q")
    _req(q_idx, torch.bfloat16, 3, "q_idx")
    _req(k_cache, torch.bfloat16, 3, "k_cache")
    _req(v_cache, torch.bfloat16, 3, "v_cache")
    _req(k_idx_cache, torch.bfloat16, 2, "k_idx_cache")
    _req(cu_seqlens, torch.int64, 1, "cu_seqlens")
    S, H_q, d_h = q.shape
    H_kv, d_idx = q_idx.shape[1], q_idx.shape[2]
    for t, n in ((q_idx, "q_idx"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (k_idx_cache, "k_idx_cache"), (cu_seqlens, "cu_seqlens")):
        _req(t, t.dtype, t.dim(), n, device=q.device)
    o, lse, idx_out = _decode_outputs(q, q_idx, k, o, lse, idx_out, alloc=False)
    _check("msa_sparse_decode_noalloc", lib.msa_sparse_decode_noalloc(
        _ptr(q), _ptr(q_idx), _ptr(k_cache), _ptr(v_cache), _ptr(k_idx_cache), _ptr(cu_seqlens),
        S, max_len, H_q, H_kv, d_h, d_idx, block_size, k, _ptr(o), _ptr(lse), _ptr(idx_out),
        _stream(stream)))
    return o, lse, idx_out


def msa_prefill_varlen_workspace(cu_seqlens, H_q, H_kv, d_h, kk):
    """Workspace bytes of msa_prefill_varlen for this batch (cu_seqlens: CPU int64 [nseq+1])."""
    if cu_seqlens.dtype != torch.int64 or cu_seqlens.is_cuda or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous int64 CPU tensor")
    return int(lib.msa_prefill_varlen_workspace(ctypes.c_void_p(cu_seqlens.data_ptr()),
                                                cu_seqlens.numel() - 1, H_q, H_kv, d_h, kk))


def msa_prefill_varlen(q, k, v, q_idx, k_idx, cu_seqlens, kk, o=None, lse=None, idx=None,
                       ws=None, block_size=BLOCK, stream=None):
    """Prefill of packed independent sequences (cu_seqlens: a CPU int64 tensor [nseq+1]) ->
    (O [T,H_q,d_h], LSE flat fp32 (sequence s: [H_q, N_s] at H_q*cu[s]), idx flat int32
    (sequence s: [H_kv, N_s, k] at H_kv*k*cu[s]))."""
    for t, n, nd in ((q, "q", 3), (k, "k", 3), (v, "v", 3), (q_idx, "q_idx", 3)):
        _req(t, torch.bfloat16, nd, n)
    _req(k_idx, torch.bfloat16, 2, "k_idx")
    if cu_seqlens.dtype != torch.int64 or cu_seqlens.is_cuda or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous int64 CPU tensor")
    T, H_q, d_h = q.shape
    H_kv, d_idx = k.shape[1], q_idx.shape[2]
    nseq = cu_seqlens.numel() - 1
    cu_ptr = ctypes.c_void_p(cu_seqlens.data_ptr())
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(T * H_q, dtype=torch.float32, device=q.device)
    if idx is None:
        idx = torch.empty(T * H_kv * kk, dtype=torch.int32, device=q.device)
    nws = int(lib.msa_prefill_varlen_workspace(cu_ptr, nseq, H_q, H_kv, d_h, kk))
    if ws is None:
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=q.device)
    _check("msa_prefill_varlen", lib.msa_prefill_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx), cu_ptr, nseq, H_q, H_kv, d_h, d_idx,
        block_size, kk, _ptr(idx), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))
    return o, lse, idx


def msa_sparse_decode_paged(q, q_idx, k_pages, v_pages, k_idx_pages, page_table, seq_lens,
                            max_len, k, o=None, lse=None, idx_out=None, ws=None, block_size=BLOCK,
                            stream=None):
    """Decode from 64-token pages -> (O [S,H_q,d_h] bf16, LSE [S,H_q] fp32, idx [S,H_kv,k])."""
    _req(q, torch.bfloat16, 3, "q")
    _req(q_idx, torch.bfloat16, 3, "q_idx")
    _req(k_pages, torch.bfloat16, 4, "k_pages")
    _req(v_pages, torch.bfloat16, 4, "v_pages")
    _req(k_idx_pages, torch.bfloat16, 3, "k_idx_pages")
    _req(page_table, torch.int32, 2, "page_table")
    _req(seq_lens, torch.int64, 1, "seq_lens")
    S, H_q, d_h = q.shape
    H_kv, d_idx = q_idx.shape[1], q_idx.shape[2]
    num_pages, max_pages = k_pages.shape[0], page_table.shape[1]
    if page_table.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("page_table must be [S, max_pages] and seq_lens [S], S = %d" % S)
    o, lse, idx_out = _decode_outputs(q, q_idx, k, o, lse, idx_out, alloc=True)
    nws = msa_sparse_decode_workspace(S, max_len, H_q, H_kv, d_h, d_idx, k)
    if ws is None:
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=q.device)
    _check("msa_sparse_decode_paged", lib.msa_sparse_decode_paged(
        _ptr(q), _ptr(q_idx), _ptr(k_pages), _ptr(v_pages), _ptr(k_idx_pages), _ptr(page_table),
        _ptr(seq_lens), S, max_pages, num_pages, max_len, H_q, H_kv, d_h, d_idx, block_size, k,
        _ptr(o), _ptr(lse), _ptr(idx_out), _ptr(ws), ws.numel(), _stream(stream)))
    return o, lse, idx_out


def msa_kl_loss_fwd_workspace(N, H_kv, k):
    return int(lib.msa_kl_loss_fwd_workspace(N, H_kv, k))


def msa_kl_loss_fwd(q, k, q_idx, k_idx, idx, lse, kl=None, ws=None, block_size=BLOCK,
                    stream=None, lse_idx=None, p_sum=None):
    """KL alignment loss per (group, row): KL [H_kv, N] fp32, teacher from the forward's LSE.
    lse_idx / p_sum ([H_kv, N] fp32, optional) receive what msa_kl_loss_bwd needs."""
    _req(q, torch.bfloat16, 3, "q")
    _req(k, torch.bfloat16, 3, "k")
    _req(q_idx, torch.bfloat16, 3, "q_idx")
    _req(k_idx, torch.bfloat16, 2, "k_idx")
    _req(idx, torch.int32, 3, "idx")
    _req(lse, torch.float32, 2, "lse")
    N, H_q, d_h = q.shape
    H_kv, d_idx = k.shape[1], q_idx.shape[2]
    kk = idx.shape[2]
    if kl is None:
        kl = torch.empty((H_kv, N), dtype=torch.float32, device=q.device)
    nws = msa_kl_loss_fwd_workspace(N, H_kv, kk)
    if ws is None and nws:
        ws = torch.empty(nws, dtype=torch.uint8, device=q.device)
    _check("msa_kl_loss_fwd", lib.msa_kl_loss_fwd(
        _ptr(q), _ptr(k), _ptr(q_idx), _ptr(k_idx), _ptr(idx), _ptr(lse), _ptr(kl), _ptr(lse_idx),
        _ptr(p_sum), N, H_q, H_kv, d_h, d_idx, block_size, kk, _ptr(ws),
        0 if ws is None else ws.numel(), _stream(stream)))
    return kl


def msa_kl_loss_bwd_workspace(N, H_kv, d_idx, k):
    return int(lib.msa_kl_loss_bwd_workspace(N, H_kv, d_idx, k))


def msa_kl_loss_bwd(q, k, q_idx, k_idx, idx, lse, lse_idx, p_sum, grad_kl, dq_idx=None,
                    dk_idx=None, ws=None, block_size=BLOCK, stream=None):
    """Index-branch gradient of sum(grad_kl * KL), teacher fixed -> (dq_idx [N,H_kv,d_idx],
    dk_idx [N,d_idx]) fp32."""
    for t, n in ((lse_idx, "lse_idx"), (p_sum, "p_sum"), (grad_kl, "grad_kl")):
        _req(t, torch.float32, 2, n)
    N, H_q, d_h = q.shape
    H_kv, d_idx = k.shape[1], q_idx.shape[2]
    kk = idx.shape[2]
    if dq_idx is None:
        dq_idx = torch.empty((N, H_kv, d_idx), dtype=torch.float32, device=q.device)
    if dk_idx is None:
        dk_idx = torch.empty((N, d_idx), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = torch.empty(msa_kl_loss_bwd_workspace(N, H_kv, d_idx, kk), dtype=torch.uint8,
                         device=q.device)
    _check("msa_kl_loss_bwd", lib.msa_kl_loss_bwd(
        _ptr(q), _ptr(k), _ptr(q_idx), _ptr(k_idx), _ptr(idx), _ptr(lse), _ptr(lse_idx),
        _ptr(p_sum), _ptr(grad_kl), _ptr(dq_idx), _ptr(dk_idx), N, H_q, H_kv, d_h, d_idx,
        block_size, kk, _ptr(ws), ws.numel(), _stream(stream)))
    return dq_idx, dk_idx


def msa_device_status():
    """Reads and clears the device status words; raises on a recorded timeout."""
    _check("msa_device_status", lib.msa_device_status())


def msa_set_wait_limit_ns(ns):
    """Time limit of the index-branch kernel's pipeline waits on the current device (default
    2e9 ns; 0 makes a wait that is not already satisfied give up at once)."""
    _check("msa_set_wait_limit_ns", lib.msa_set_wait_limit_ns(int(ns)))
