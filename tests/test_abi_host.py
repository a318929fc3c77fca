"""Host-side checks of the C ABI (no GPU needed): the library builds for sm_103a, loads,
exports every entry point include/msa.h declares, and rejects bad arguments before any
CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    return ctypes.CDLL(path)


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "msa.h")).read()
    return sorted(set(re.findall(r"^\w[\w\s\*]*?\b(msa_\w+)\s*\(", text, re.M)))


def test_header_declares_the_api():
    syms = declared_symbols()
    for name in ("msa_index_block_scores", "msa_select_blocks", "msa_index_select",
                 "msa_sparse_attn_fwd", "msa_sparse_attn_fwd_workspace", "msa_sparse_decode",
                 "msa_sparse_decode_workspace", "msa_sparse_decode_paged", "msa_prefill_varlen",
                 "msa_prefill_varlen_workspace", "msa_kl_loss_fwd", "msa_kl_loss_bwd",
                 "msa_kl_loss_bwd_workspace",
                 "msa_kl_loss_fwd_workspace", "msa_sparse_attn_bwd", "msa_sparse_attn_bwd_workspace",
                 "msa_status_string", "msa_device_status"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    lib.msa_status_string.restype = ctypes.c_char_p
    names = [lib.msa_status_string(i).decode() for i in range(6)]
    assert names == ["MSA_OK", "MSA_ERR_INVALID_ARGUMENT", "MSA_ERR_UNSUPPORTED",
                     "MSA_ERR_WORKSPACE", "MSA_ERR_CUDA", "MSA_ERR_TIMEOUT"]
    assert lib.msa_status_string(99) == b"MSA_ERR_UNKNOWN"


# Fake, 16-byte aligned pointer values: every call below must return before touching them.
P = ctypes.c_void_p(0x10000)
MIS = ctypes.c_void_p(0x10002)
NUL = ctypes.c_void_p(0)
i64 = ctypes.c_int64


def scores(lib, q=P, k=P, M=P, N=1024, H_kv=4, d_idx=64, B=64, qs=0, qc=1024):
    return lib.msa_index_block_scores(q, k, M, i64(N), H_kv, d_idx, B, i64(qs), i64(qc), NUL)


def select(lib, M=P, idx=P, N=1024, H_kv=4, B=64, k=16, qs=0, qc=1024):
    return lib.msa_select_blocks(M, idx, i64(N), H_kv, B, k, i64(qs), i64(qc), NUL)


def index_select(lib, q=P, k=P, idx=P, N=1024, H_kv=4, d_idx=64, B=64, kk=16, qs=0, qc=1024):
    return lib.msa_index_select(q, k, idx, i64(N), H_kv, d_idx, B, kk, i64(qs), i64(qc), NUL)


def attn(lib, q=P, k=P, v=P, idx=P, o=P, lse=P, N=1024, H_q=32, H_kv=4, d_h=128, B=64, kk=16,
         ws=P, wsb=1 << 40):
    return lib.msa_sparse_attn_fwd(q, k, v, idx, o, lse, i64(N), H_q, H_kv, d_h, B, kk, ws,
                                   ctypes.c_size_t(wsb), NUL)


def decode(lib, q=P, S=4, max_len=1000, H_q=32, H_kv=4, d_h=128, d_idx=64, B=64, k=16, ws=P,
           wsb=1 << 40, cu=P, idx_out=NUL):
    return lib.msa_sparse_decode(q, P, P, P, P, cu, S, i64(max_len), H_q, H_kv, d_h, d_idx, B, k,
                                 P, P, idx_out, ws, ctypes.c_size_t(wsb), NUL)


def kl(lib, q=P, k=P, qi=P, ki=P, idx=P, lse=P, out=P, N=1024, H_q=32, H_kv=4, d_h=128, d_idx=64,
       B=64, kk=16, ws=P, wsb=1 << 40):
    return lib.msa_kl_loss_fwd(q, k, qi, ki, idx, lse, out, NUL, NUL, i64(N), H_q, H_kv, d_h, d_idx,
                               B, kk,
                               ws, ctypes.c_size_t(wsb), NUL)


INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3


@pytest.mark.parametrize("kw", [dict(q=NUL), dict(k=MIS), dict(M=NUL), dict(N=0), dict(B=32),
                                dict(qs=-1), dict(qc=0), dict(qs=1000, qc=100), dict(H_kv=0)])
def test_scores_invalid(lib, kw):
    assert scores(lib, **kw) == INVALID


@pytest.mark.parametrize("kw", [dict(H_kv=3), dict(H_kv=16), dict(d_idx=48), dict(d_idx=128)])
def test_scores_unsupported(lib, kw):
    assert scores(lib, **kw) == UNSUPPORTED


@pytest.mark.parametrize("kw", [dict(M=NUL), dict(idx=NUL), dict(k=0), dict(k=65), dict(B=128),
                                dict(qs=1024, qc=1), dict(N=-5)])
def test_select_invalid(lib, kw):
    assert select(lib, **kw) == INVALID


@pytest.mark.parametrize("kw", [dict(q=NUL), dict(k=MIS), dict(idx=NUL), dict(N=0), dict(B=32),
                                dict(kk=0), dict(kk=65), dict(qs=-1), dict(qc=0),
                                dict(qs=1000, qc=100), dict(H_kv=0)])
def test_index_select_invalid(lib, kw):
    assert index_select(lib, **kw) == INVALID


@pytest.mark.parametrize("kw", [dict(H_kv=3), dict(H_kv=16), dict(d_idx=48), dict(kk=33),
                                dict(kk=64)])
def test_index_select_unsupported(lib, kw):
    assert index_select(lib, **kw) == UNSUPPORTED


@pytest.mark.parametrize("kw", [dict(q=NUL), dict(o=MIS), dict(N=0), dict(H_q=30), dict(kk=0),
                                dict(kk=100), dict(B=16), dict(ws=NUL), dict(ws=MIS)])
def test_attn_invalid(lib, kw):
    assert attn(lib, **kw) == INVALID


@pytest.mark.parametrize("kw", [dict(d_h=96), dict(d_h=256), dict(H_q=64, H_kv=4),
                                dict(H_q=12, H_kv=4)])
def test_attn_unsupported(lib, kw):
    assert attn(lib, **kw) == UNSUPPORTED


@pytest.mark.parametrize("kw", [dict(q=NUL), dict(S=0), dict(max_len=0), dict(cu=NUL),
                                dict(cu=ctypes.c_void_p(0x10004)), dict(k=0), dict(ws=NUL),
                                dict(idx_out=MIS)])
def test_decode_invalid(lib, kw):
    assert decode(lib, **kw) == INVALID


def test_decode_workspace_checked(lib):
    lib.msa_sparse_decode_workspace.restype = ctypes.c_size_t
    need = lib.msa_sparse_decode_workspace(4, i64(1000), 32, 4, 128, 64, 16)
    assert need > 0
    assert decode(lib, wsb=need - 1) == WORKSPACE
    assert decode(lib, d_h=80) == UNSUPPORTED


def test_workspace_sizes(lib):
    lib.msa_sparse_decode_workspace.restype = ctypes.c_size_t
    lib.msa_sparse_attn_fwd_workspace.restype = ctypes.c_size_t
    S, L, H_q, H_kv, d_h, k = 32, 262144, 32, 4, 128, 16
    need = lib.msa_sparse_decode_workspace(S, i64(L), H_q, H_kv, d_h, 64, k)
    # block scores + selections
    nblk = L // 64
    floor = 4 * S * H_kv * nblk + 4 * S * H_kv * k
    assert floor <= need <= floor + 2 * 256
    # main branch: per query chunk (<= 32768 rows) the bucket arrays, the entries, the plan's
    # (bucket, rank, entry) scratch and its per-tile counts, each tile's shared-block list and
    # private-slot masks, and the private partials (bf16 O + fp32 LSE per selection, at fixed
    # (row, slot) positions)
    need = lib.msa_sparse_attn_fwd_workspace(i64(1024), 8, 2, 64, 4)
    sel = 2 * 1024 * 4
    tiles = 2 * 1024 // 16                       # 16-query tiles: shared-block lists, masks
    floor = (4 * sel + 12 * sel + 4 * tiles + sel * 4 * (64 * 2 + 4) + 3 * 4 * (2 * 16 + 1) +
             4 * tiles * (512 + 1) + 8 * tiles * 16)
    assert floor <= need <= floor + 10 * 256
    assert attn(lib, N=1024, H_q=8, H_kv=2, d_h=64, kk=4, wsb=need - 1) == WORKSPACE


@pytest.mark.parametrize("kw", [dict(q=NUL), dict(qi=MIS), dict(ki=NUL), dict(idx=NUL),
                                dict(lse=ctypes.c_void_p(0x10001)), dict(out=NUL), dict(N=0),
                                dict(H_q=30), dict(kk=0), dict(kk=65), dict(B=32), dict(ws=NUL),
                                dict(ws=MIS)])
def test_kl_invalid(lib, kw):
    assert kl(lib, **kw) == INVALID


@pytest.mark.parametrize("kw", [dict(d_h=96), dict(d_idx=128), dict(H_q=64, H_kv=4),
                                dict(H_q=12, H_kv=4), dict(N=(1 << 21) + 1)])
def test_kl_unsupported(lib, kw):
    assert kl(lib, **kw) == UNSUPPORTED


def test_kl_workspace(lib):
    lib.msa_kl_loss_fwd_workspace.restype = ctypes.c_size_t
    need = lib.msa_kl_loss_fwd_workspace(i64(131072), 4, 16)
    sel = 4 * 131072 * 16
    floor = 20 * sel + 4 * 4 * (4 * 2048 + 1)           # entries + partials, four bucket arrays
    assert floor <= need <= floor + 6 * 256
    assert lib.msa_kl_loss_fwd_workspace(i64(0), 4, 16) == 0
    assert kl(lib, N=1000, wsb=lib.msa_kl_loss_fwd_workspace(i64(1000), 4, 16) - 1) == WORKSPACE


def paged(lib, pt=P, sl=ctypes.c_void_p(0x10008), S=4, max_pages=16, num_pages=64, max_len=1000,
          H_q=32, H_kv=4, d_h=128, d_idx=64, B=64, k=16, ws=P, wsb=1 << 40, kp=P):
    return lib.msa_sparse_decode_paged(P, P, kp, P, P, pt, sl, S, i64(max_pages), i64(num_pages),
                                       i64(max_len), H_q, H_kv, d_h, d_idx, B, k, P, P, NUL, ws,
                                       ctypes.c_size_t(wsb), NUL)


@pytest.mark.parametrize("kw", [dict(pt=NUL), dict(pt=ctypes.c_void_p(0x10002)), dict(sl=NUL),
                                dict(sl=ctypes.c_void_p(0x10004)), dict(kp=MIS), dict(S=0),
                                dict(max_pages=15), dict(num_pages=0), dict(max_len=0),
                                dict(k=0), dict(B=32), dict(ws=NUL)])
def test_decode_paged_invalid(lib, kw):
    assert paged(lib, **kw) == INVALID


def test_decode_paged_unsupported_and_workspace(lib):
    assert paged(lib, d_h=96) == UNSUPPORTED
    assert paged(lib, d_idx=48) == UNSUPPORTED
    lib.msa_sparse_decode_workspace.restype = ctypes.c_size_t
    need = lib.msa_sparse_decode_workspace(4, i64(1000), 32, 4, 128, 64, 16)
    assert paged(lib, wsb=need - 1) == WORKSPACE


def varlen(lib, cu=(0, 100, 1100), q=P, k=16, ws=P, wsb=1 << 40, H_q=32, H_kv=4, d_h=128,
           d_idx=64, B=64, idx=P):
    arr = None if cu is None else (ctypes.c_int64 * len(cu))(*cu)
    n = 0 if cu is None else len(cu) - 1
    return lib.msa_prefill_varlen(q, P, P, P, P, arr, n, H_q, H_kv, d_h, d_idx, B, k, idx, P, P,
                                  ws, ctypes.c_size_t(wsb), NUL)


@pytest.mark.parametrize("kw", [dict(cu=None), dict(cu=(1, 100)), dict(cu=(0, 100, 100)),
                                dict(q=NUL), dict(idx=ctypes.c_void_p(0x10002)), dict(k=0),
                                dict(B=32), dict(ws=NUL)])
def test_prefill_varlen_invalid(lib, kw):
    assert varlen(lib, **kw) == INVALID


def test_prefill_varlen_unsupported_and_workspace(lib):
    assert varlen(lib, k=33) == UNSUPPORTED
    assert varlen(lib, d_h=96) == UNSUPPORTED
    lib.msa_prefill_varlen_workspace.restype = ctypes.c_size_t
    lib.msa_sparse_attn_fwd_workspace.restype = ctypes.c_size_t
    # one launch per stage over a virtual row space where each sequence starts on a multiple of
    # 128 rows: 100, 40000, 900 -> 128 + 40064 + 1024 = 41216 rows.  Workspace: the main
    # branch's for 41216 rows, the selections and LSEs over the virtual rows, and (lengths not
    # multiples of 128) virtual copies of q, k, v, q_idx, k_idx and o; d_idx is sized at 64.
    cu = (ctypes.c_int64 * 4)(0, 100, 40100, 41000)
    need = lib.msa_prefill_varlen_workspace(cu, 3, 32, 4, 128, 16)
    tv = 41216
    floor = (lib.msa_sparse_attn_fwd_workspace(i64(tv), 32, 4, 128, 16) + 4 * 4 * tv * 16 +
             4 * 32 * tv + 2 * tv * (32 * 128 + 2 * 4 * 128 + 4 * 64 + 64 + 32 * 128))
    assert floor <= need <= floor + 12 * 256 + 2 * 8 * 4 + 4 * tv // 128
    assert varlen(lib, cu=(0, 100, 40100, 41000), wsb=need - 1) == WORKSPACE
    # lengths that are multiples of 128: the packed rows are the virtual rows, nothing is copied
    cu2 = (ctypes.c_int64 * 3)(0, 2048, 4096)
    need2 = lib.msa_prefill_varlen_workspace(cu2, 2, 32, 4, 128, 16)
    floor2 = (lib.msa_sparse_attn_fwd_workspace(i64(4096), 32, 4, 128, 16) + 4 * 4 * 4096 * 16 +
              4 * 32 * 4096)
    assert floor2 <= need2 <= floor2 + 6 * 256 + 2 * 8 * 3 + 4 * 32


def klb(lib, gk=P, dq=P, dk=P, N=1024, H_q=32, H_kv=4, d_h=128, d_idx=64, B=64, kk=16, ws=P,
        wsb=1 << 40):
    return lib.msa_kl_loss_bwd(P, P, P, P, P, P, P, P, gk, dq, dk, i64(N), H_q, H_kv, d_h, d_idx,
                               B, kk, ws, ctypes.c_size_t(wsb), NUL)


@pytest.mark.parametrize("kw", [dict(gk=NUL), dict(dq=MIS), dict(dk=NUL), dict(N=0), dict(kk=0),
                                dict(B=32), dict(ws=NUL), dict(H_q=30)])
def test_kl_bwd_invalid(lib, kw):
    assert klb(lib, **kw) == INVALID


def test_kl_bwd_unsupported_and_workspace(lib):
    assert klb(lib, H_q=48) == UNSUPPORTED          # G = 12: the pass is built for G in {1,2,4,8}
    assert klb(lib, d_idx=48) == UNSUPPORTED
    lib.msa_kl_loss_bwd_workspace.restype = ctypes.c_size_t
    lib.msa_kl_loss_fwd_workspace.restype = ctypes.c_size_t
    need = lib.msa_kl_loss_bwd_workspace(i64(1024), 4, 64, 16)
    assert need >= lib.msa_kl_loss_fwd_workspace(i64(1024), 4, 16) + 4 * 4 * 1024 * 16 * 64
    assert klb(lib, wsb=need - 1) == WORKSPACE


def test_device_status_and_wait_limit_without_a_device(lib):
    """The status word and the wait-limit knob live in device memory of the current device; with
    no usable device both calls report MSA_ERR_CUDA instead of failing in another way."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    assert lib.msa_device_status() == 4
    lib.msa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    assert lib.msa_set_wait_limit_ns(ctypes.c_uint64(0)) == 4
