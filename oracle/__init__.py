"""CPU oracle of MSA block-sparse GQA attention (TEST INFRASTRUCTURE ONLY).

A plain C (OpenMP, fp64) restatement of the formulas in «MiniMax-M3：MSA 技术报告速读»,
section 核心机制 (index branch eq. S^idx / M^idx, TopK eq. I^(r)_i with the forced local
block, main branch eq. O^(h)_i, LSE from section Kernel; the KL alignment loss of section
训练, eq. P^idx / P / L_KL).  Only tests, the smoke check
and the bench's CPU-baseline leg import this package; the CUDA library never does, and
the two share no code.

Every function takes numpy arrays: bf16 tensors as uint16 bit patterns (see
``gen.to_bits``), int32/int64 index arrays, and returns numpy arrays.

Pins (what this oracle is checked against, in tests/test_oracle_pins.py):
  block scores  -- brute-force dense fp64 matmul, reshaped per block and max-reduced;
                   hand-worked golden case (tests/golden).
  selection     -- brute-force stable argsort; constant-score closed form; invariants.
  main branch   -- dense masked fp64 attention; k >= #blocks equals the library routine
                   torch.nn.functional.scaled_dot_product_attention (causal, fp64);
                   Q = 0 closed form (LSE = ln|T|, O = mean of V over T).
  decode        -- equals the prefill row L-1 on the same tokens.
  main-branch gradient -- torch.autograd (fp64) through a dense masked attention; k >= #blocks
                   equals torch.autograd through scaled_dot_product_attention (causal).
  KL gradient   -- torch.autograd (fp64) through a dense masked restatement of the loss; central
                   finite differences of the oracle's own kl_loss; the uniform-teacher closed
                   form; sum over the index keys of dK_idx . K_idx equals sum of dQ_idx . Q_idx.
  KL loss       -- k >= #blocks equals scipy.stats.entropy of torch.softmax distributions
                   (causal); sparse selections equal the same library routines on a mask
                   built by brute force; uniform-teacher and uniform-student closed forms;
                   KL = 0 when the student's scores equal the teacher's; KL >= 0.
  bf16 rounding -- exhaustive agreement with torch's fp32->bf16 RNE on fp32-representable
                   values plus hand-picked tie cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIB = os.path.join(_HERE, "libmsa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP) into oracle/libmsa_oracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-Wall", "-Wno-unknown-pragmas", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        L.msa_oracle_block_scores.argtypes = [P, P, i64, i32, i32, i32, i64, i64, P, P]
        L.msa_oracle_select_blocks.argtypes = [P, i64, i32, i32, i32, i64, i64, P]
        L.msa_oracle_sparse_attn.argtypes = [P, P, P, P, i64, i32, i32, i32, i32, i32, P, i64,
                                             P, P, P]
        L.msa_oracle_sparse_attn_rows.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, i64,
                                                  P, P, P]
        L.msa_oracle_prefill_rows.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i32, i32, i32,
                                              P, i64, P, P, P, P, P]
        L.msa_oracle_decode.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, P,
                                        i32, P, P, i64, P, P, P]
        L.msa_oracle_kl_loss.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, i64, P]
        L.msa_oracle_kl_loss_grad.argtypes = [P, P, P, P, P, P, i64, i32, i32, i32, i32, i32,
                                               i32, P, P, P, P]
        L.msa_oracle_sparse_attn_grad.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i32, i32, P,
                                                   P, P]
        L.msa_oracle_set_threads.argtypes = [i32]
        L.msa_oracle_get_threads.restype = i32
        L.msa_oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        L.msa_oracle_f64_to_bf16.restype = ctypes.c_uint16
        L.msa_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.msa_oracle_bf16_to_f64.restype = ctypes.c_double
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def set_threads(n: int) -> None:
    lib().msa_oracle_set_threads(int(n))


def get_threads() -> int:
    return int(lib().msa_oracle_get_threads())


def f64_to_bf16(x: float) -> int:
    return int(lib().msa_oracle_f64_to_bf16(float(x)))


def block_scores(q_idx, k_idx, block_size=64, q_start=0, q_count=None):
    """Index-branch block scores M [H_kv, q_count, nblk] -> (M64 float64, M32 float32)."""
    q_idx, k_idx = _u16(q_idx), _u16(k_idx)
    N, H_kv, d_idx = q_idx.shape
    if q_count is None:
        q_count = N - q_start
    nblk = -(-N // block_size)
    M64 = np.empty((H_kv, q_count, nblk), np.float64)
    M32 = np.empty((H_kv, q_count, nblk), np.float32)
    lib().msa_oracle_block_scores(_p(q_idx), _p(k_idx), N, H_kv, d_idx, block_size, q_start,
                                  q_count, _p(M64), _p(M32))
    return M64, M32


def select_blocks(M32, N, k, block_size=64, q_start=0, I=None):
    """Selection from fp32 block scores [H_kv, q_count, nblk] -> I [H_kv, N, k] int32
    (rows outside [q_start, q_start+q_count) are left as given / -2)."""
    M32 = np.ascontiguousarray(M32, dtype=np.float32)
    H_kv, q_count, _ = M32.shape
    if I is None:
        I = np.full((H_kv, N, k), -2, np.int32)
    lib().msa_oracle_select_blocks(_p(M32), N, H_kv, block_size, k, q_start, q_count, _p(I))
    return I


def sparse_attn(q, k, v, I, block_size=64, rows=None, compact=False):
    """Main branch over a given selection I [H_kv, N, kk] -> (O64, O16 bits, LSE64).
    compact=True: q and I hold only the listed rows ([n,H_q,d_h] and [H_kv,n,kk], row t is
    query position rows[t]); k and v are the whole sequence."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    I = np.ascontiguousarray(I, dtype=np.int32)
    if compact:
        rows_a = np.ascontiguousarray(rows, dtype=np.int64)
        n, H_q, d_h = q.shape
        H_kv = k.shape[1]
        assert I.shape[:2] == (H_kv, n) and len(rows_a) == n
        I_rows = np.ascontiguousarray(I.transpose(1, 0, 2))
        O64 = np.empty((n, H_q, d_h), np.float64)
        O16 = np.empty((n, H_q, d_h), np.uint16)
        LSE = np.empty((n, H_q), np.float64)
        lib().msa_oracle_sparse_attn_rows(_p(q), _p(k), _p(v), _p(I_rows), H_q, H_kv, d_h,
                                          block_size, I.shape[2], _p(rows_a), n, _p(O64),
                                          _p(O16), _p(LSE))
        return O64, O16, LSE
    N, H_q, d_h = q.shape
    H_kv = k.shape[1]
    kk = I.shape[2]
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = N if rows_a is None else len(rows_a)
    O64 = np.empty((n, H_q, d_h), np.float64)
    O16 = np.empty((n, H_q, d_h), np.uint16)
    LSE = np.empty((n, H_q), np.float64)
    lib().msa_oracle_sparse_attn(_p(q), _p(k), _p(v), _p(I), N, H_q, H_kv, d_h, block_size, kk,
                                 _p(rows_a), n, _p(O64), _p(O16), _p(LSE))
    return O64, O16, LSE


def prefill(q, k, v, q_idx, k_idx, kk, block_size=64, rows=None, want_m=False, compact=False):
    """Whole prefill path on the given rows (None: all) ->
    dict(I [n,H_kv,kk], O64, O16, LSE [n,H_q], M32 [n,H_kv,nblk] if want_m).
    compact=True: q and q_idx hold only the listed rows ([n,H_q,d_h], [n,H_kv,d_idx])."""
    q, k, v, q_idx, k_idx = map(_u16, (q, k, v, q_idx, k_idx))
    N, H_kv, d_h = k.shape
    H_q, d_idx = q.shape[1], q_idx.shape[2]
    rows_a = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    n = len(rows_a)
    if not compact:
        q, q_idx = np.ascontiguousarray(q[rows_a]), np.ascontiguousarray(q_idx[rows_a])
    assert q.shape[0] == n and q_idx.shape[0] == n
    nblk = -(-N // block_size)
    I = np.empty((n, H_kv, kk), np.int32)
    M32 = np.empty((n, H_kv, nblk), np.float32) if want_m else None
    O64 = np.empty((n, H_q, d_h), np.float64)
    O16 = np.empty((n, H_q, d_h), np.uint16)
    LSE = np.empty((n, H_q), np.float64)
    lib().msa_oracle_prefill_rows(_p(q), _p(k), _p(v), _p(q_idx), _p(k_idx), N, H_q, H_kv, d_h,
                                  d_idx, block_size, kk, _p(rows_a), n, _p(I), _p(M32), _p(O64),
                                  _p(O16), _p(LSE))
    out = dict(rows=rows_a, I=I, O64=O64, O16=O16, LSE=LSE)
    if want_m:
        out["M32"] = M32
    return out


def decode(q, q_idx, k_cache, v_cache, k_idx_cache, cu_seqlens, kk, block_size=64, seqs=None,
           want_m=False):
    """Decode path (query = last cache row of each sequence) ->
    dict(I [n,H_kv,kk], O64, O16, LSE [n,H_q], M32 [n,H_kv,max_nblk] if want_m)."""
    q, q_idx, k_cache, v_cache, k_idx_cache = map(_u16, (q, q_idx, k_cache, v_cache, k_idx_cache))
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    S, H_q, d_h = q.shape
    H_kv, d_idx = q_idx.shape[1], q_idx.shape[2]
    seqs_a = None if seqs is None else np.ascontiguousarray(seqs, dtype=np.int32)
    n = S if seqs_a is None else len(seqs_a)
    max_len = int((cu[1:] - cu[:-1]).max())
    stride = -(-max_len // block_size)
    I = np.empty((n, H_kv, kk), np.int32)
    M32 = np.empty((n, H_kv, stride), np.float32) if want_m else None
    O64 = np.empty((n, H_q, d_h), np.float64)
    O16 = np.empty((n, H_q, d_h), np.uint16)
    LSE = np.empty((n, H_q), np.float64)
    lib().msa_oracle_decode(_p(q), _p(q_idx), _p(k_cache), _p(v_cache), _p(k_idx_cache), _p(cu),
                            S, H_q, H_kv, d_h, d_idx, block_size, kk, _p(seqs_a), n, _p(I),
                            _p(M32), stride, _p(O64), _p(O16), _p(LSE))
    out = dict(I=I, O64=O64, O16=O16, LSE=LSE)
    if want_m:
        out["M32"] = M32
    return out


def kl_loss(q, k, q_idx, k_idx, I, block_size=64, rows=None, compact=False):
    """KL alignment loss over a given selection -> KL [n, H_kv] float64, row t = query rows[t]
    (all N rows when rows is None).  I is [H_kv, N, kk]; compact=True: q, q_idx and I hold only
    the listed rows ([n,H_q,d_h], [n,H_kv,d_idx], [H_kv,n,kk])."""
    q, k, q_idx, k_idx = map(_u16, (q, k, q_idx, k_idx))
    N, H_kv, d_h = k.shape
    H_q, d_idx = q.shape[1], q_idx.shape[2]
    rows_a = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    I = np.asarray(I, dtype=np.int32)
    if not compact:
        q, q_idx, I = q[rows_a], q_idx[rows_a], I[:, rows_a]
    q, q_idx = np.ascontiguousarray(q), np.ascontiguousarray(q_idx)
    I_rows = np.ascontiguousarray(I.transpose(1, 0, 2))
    n = len(rows_a)
    assert q.shape[0] == n and q_idx.shape[0] == n and I_rows.shape[:2] == (n, H_kv)
    KL = np.empty((n, H_kv), np.float64)
    lib().msa_oracle_kl_loss(_p(q), _p(k), _p(q_idx), _p(k_idx), _p(I_rows), H_q, H_kv, d_h,
                             d_idx, block_size, I_rows.shape[2], _p(rows_a), n, _p(KL))
    return KL


def kl_loss_grad(q, k, q_idx, k_idx, I, g_kl, block_size=64):
    """Index-branch gradient of sum(g_kl * KL) (teacher fixed) over all rows ->
    dict(dq_idx [N,H_kv,d_idx], dk_idx [N,d_idx], lse_idx [H_kv,N], psum [H_kv,N]) float64."""
    q, k, q_idx, k_idx = map(_u16, (q, k, q_idx, k_idx))
    I = np.ascontiguousarray(I, dtype=np.int32)
    g_kl = np.ascontiguousarray(g_kl, dtype=np.float64)
    N, H_q, d_h = q.shape
    H_kv, d_idx = k.shape[1], q_idx.shape[2]
    out = dict(dq_idx=np.empty((N, H_kv, d_idx)), dk_idx=np.empty((N, d_idx)),
               lse_idx=np.empty((H_kv, N)), psum=np.empty((H_kv, N)))
    lib().msa_oracle_kl_loss_grad(_p(q), _p(k), _p(q_idx), _p(k_idx), _p(I), _p(g_kl), N, H_q,
                                  H_kv, d_h, d_idx, block_size, I.shape[2], _p(out["dq_idx"]),
                                  _p(out["dk_idx"]), _p(out["lse_idx"]), _p(out["psum"]))
    return out


def sparse_attn_grad(q, k, v, dO, I, block_size=64):
    """Main-branch gradient for upstream dO [N,H_q,d_h] (bf16 bits) over a given selection ->
    dict(dq [N,H_q,d_h], dk [N,H_kv,d_h], dv [N,H_kv,d_h]) float64."""
    q, k, v, dO = map(_u16, (q, k, v, dO))
    I = np.ascontiguousarray(I, dtype=np.int32)
    N, H_q, d_h = q.shape
    H_kv = k.shape[1]
    out = dict(dq=np.empty((N, H_q, d_h)), dk=np.empty((N, H_kv, d_h)),
               dv=np.empty((N, H_kv, d_h)))
    lib().msa_oracle_sparse_attn_grad(_p(q), _p(k), _p(v), _p(dO), _p(I), N, H_q, H_kv, d_h,
                                      block_size, I.shape[2], _p(out["dq"]), _p(out["dk"]),
                                      _p(out["dv"]))
    return out
