"""msa_sparse_decode_noalloc: decode for callers that cannot allocate device memory where they
decode (a runtime whose pool owns all device memory, or a loop that must not call
cudaMalloc/cudaFree).  It keeps its temporaries in a fixed array inside the library instead of a
caller-supplied workspace, so it must give the same results as msa_sparse_decode -- including on
back-to-back calls of different sizes, where the second call finds the first call's leftovers in
that shared array.  Collected last so that a failure here comes after every other test ran."""
import ctypes

import pytest
import torch

import gen
from msa_testutil import LSE_TOL, O_TOL

pytestmark = pytest.mark.gpu

msa = pytest.importorskip("block_sparse_gqa_scores_gb300")


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def call_noalloc(d, cfg, max_len, o, lse, idx):
    """Straight through the C ABI (libmsa.so via ctypes); returns the status code."""
    return msa.msa.lib.msa_sparse_decode_noalloc(
        _p(d["q"]), _p(d["q_idx"]), _p(d["k_cache"]), _p(d["v_cache"]), _p(d["k_idx_cache"]),
        _p(d["cu_seqlens"]), d["q"].shape[0], max_len, cfg.H_q, cfg.H_kv, cfg.d_h, cfg.d_idx, 64,
        cfg.k, _p(o), _p(lse), _p(idx), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def compare_once(cfg, seed, S, lo, hi):
    d = gen.decode_inputs(cfg, seed=seed, device="cuda", S=S, len_lo=lo, len_hi=hi)
    max_len = hi
    o_ref, lse_ref, idx_ref = msa.msa_sparse_decode(d["q"], d["q_idx"], d["k_cache"],
                                                    d["v_cache"], d["k_idx_cache"],
                                                    d["cu_seqlens"], max_len, cfg.k)
    o = torch.full_like(o_ref, float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    idx = torch.full_like(idx_ref, -7)
    assert call_noalloc(d, cfg, max_len, o, lse, idx) == 0
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_ref)
    assert (o.float() - o_ref.float()).abs().max().item() <= O_TOL
    assert (lse - lse_ref).abs().max().item() <= LSE_TOL


def test_noalloc_decode_matches_workspace_decode_twice():
    cfg = gen.CONFIGS["decode"]
    # two calls in a row; the second is smaller, so stale scratch from the first would show
    compare_once(cfg, seed=3, S=32, lo=65536, hi=262144)
    compare_once(cfg, seed=4, S=5, lo=1, hi=9000)


def test_noalloc_decode_rejects_sizes_beyond_its_scratch():
    cfg = gen.CONFIGS["decode"]
    d = gen.decode_inputs(cfg, seed=5, device="cuda", S=2, len_lo=100, len_hi=200)
    big = 1 << 25                                   # block scores alone exceed the fixed array
    assert msa.msa_sparse_decode_workspace(2, big, cfg.H_q, cfg.H_kv, cfg.d_h, cfg.d_idx,
                                           cfg.k) > (8 << 20)
    o = torch.empty_like(d["q"])
    lse = torch.empty((2, cfg.H_q), dtype=torch.float32, device="cuda")
    assert call_noalloc(d, cfg, big, o, lse, None) == 3        # MSA_ERR_WORKSPACE
