"""Full-size parity on the benchmark's own workloads, in the benchmark's launch configuration
(the same C-ABI calls on the full tensors), checked on sampled query rows / sequences that the
oracle recomputes one by one: 32K and 128K prefill, the 32-sequence decode batch (packed and
paged), 1M prefill (query-chunked index scores) and the packed varlen batch.

Every sampled row is checked twice: its selection against the oracle's (exact up to near-ties,
1e-3 relative), and its O and LSE against the oracle's main branch evaluated on the GPU's own
selection (O max-abs <= 2e-2, LSE <= 1e-3), so rows inside the near-tie band are covered too.
Row counts: 512 at 32K, 1024 at 128K, 4096 random rows at 1M (plus edge rows), every decode
sequence."""
import numpy as np
import pytest
import torch

import gen
import oracle
from msa_testutil import check_decode_seqs, check_prefill_rows, to_pages, unpage

pytestmark = pytest.mark.gpu

msa = pytest.importorskip("block_sparse_gqa_scores_gb300")


def sample_rows(N, n, seed):
    rng = np.random.default_rng(seed)
    edge = [0, 1, 63, 64, 65, N // 2, N - 65, N - 64, N - 1]
    rows = np.unique(np.concatenate([rng.choice(N, min(n, N), replace=False),
                                     [e for e in edge if 0 <= e < N]]))
    return rows.astype(np.int64)


def unfused_index(x, cfg, chunk=None):
    """Block scores then selection, query-chunked so that M stays bounded."""
    N = cfg.N
    idx = torch.empty((cfg.H_kv, N, cfg.k), dtype=torch.int32, device="cuda")
    chunk = chunk or N
    M = None
    for q0 in range(0, N, chunk):
        qc = min(chunk, N - q0)
        M = msa.msa_index_block_scores(x["q_idx"], x["k_idx"], M=M if M is not None and
                                       M.shape[1] == qc else None, q_start=q0, q_count=qc)
        msa.msa_select_blocks(M, N, cfg.k, idx=idx, q_start=q0)
    del M
    return idx


def run_prefill(x, cfg):
    """The benchmark's path: fused index branch over all rows, then the main branch."""
    idx = msa.msa_index_select(x["q_idx"], x["k_idx"], cfg.k)
    o, lse = msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], idx)
    torch.cuda.synchronize()
    msa.msa_device_status()
    return idx, o, lse


@pytest.mark.parametrize("name,n_rows", [("p32k", 512), ("p128k", 1024)])
def test_fullsize_prefill(name, n_rows):
    cfg = gen.CONFIGS[name]
    x = gen.prefill_inputs(cfg, seed=0, device="cuda")
    idx, o, lse = run_prefill(x, cfg)
    # the fused index branch selects exactly what block scores + selection select
    assert torch.equal(idx, unfused_index(x, cfg))
    check_prefill_rows(x, cfg.k, idx, o, lse, sample_rows(cfg.N, n_rows, seed=1))


def test_fullsize_kl_loss():
    """The KL alignment loss at 128K, in the benchmark's launch sequence (fused index branch,
    main branch, KL forward), on sampled rows the oracle recomputes on the GPU's selection."""
    cfg = gen.CONFIGS["p128k"]
    x = gen.prefill_inputs(cfg, seed=0, device="cuda")
    idx, _, lse = run_prefill(x, cfg)
    kl = msa.msa_kl_loss_fwd(x["q"], x["k"], x["q_idx"], x["k_idx"], idx, lse)
    torch.cuda.synchronize()
    msa.msa_device_status()
    rows = sample_rows(cfg.N, 256, seed=3)
    rows_t = torch.from_numpy(rows).cuda()
    ref = oracle.kl_loss(gen.to_bits(x["q"][rows_t]), gen.to_bits(x["k"]),
                         gen.to_bits(x["q_idx"][rows_t]), gen.to_bits(x["k_idx"]),
                         idx[:, rows_t].cpu().numpy(), rows=rows, compact=True)
    got = kl[:, rows_t].cpu().numpy().T.astype(np.float64)
    assert np.isfinite(kl.cpu().numpy()).all() and float(kl.min()) >= -1e-3
    assert (np.abs(got - ref) <= 5e-4 + 1e-3 * np.abs(ref)).all(), float(np.abs(got - ref).max())


def test_fullsize_prefill_1m():
    """1M tokens: the whole index array against the unfused path, and 4096 random query rows
    (plus edge rows) against the oracle."""
    cfg = gen.CONFIGS["p1m"]
    x = gen.prefill_inputs(cfg, seed=0, device="cuda")
    idx, o, lse = run_prefill(x, cfg)
    ref = unfused_index(x, cfg, chunk=16384)
    assert torch.equal(idx, ref)
    del ref
    check_prefill_rows(x, cfg.k, idx, o, lse, sample_rows(cfg.N, 4096, seed=2))


def test_fullsize_decode():
    """Every sequence of the 32-sequence batch against the oracle."""
    cfg = gen.CONFIGS["decode"]
    d = gen.decode_inputs(cfg, seed=0, device="cuda")
    o, lse, idx = msa.msa_sparse_decode(d["q"], d["q_idx"], d["k_cache"], d["v_cache"],
                                        d["k_idx_cache"], d["cu_seqlens"], cfg.len_hi, cfg.k)
    torch.cuda.synchronize()
    msa.msa_device_status()
    check_decode_seqs(d, cfg.k, o, lse, idx)


def test_fullsize_decode_paged():
    """The 32-sequence batch from a paged cache (shuffled 64-token pages): bit-equal to the packed
    decode, and every sequence against the oracle on the tokens gathered back from the pages."""
    cfg = gen.CONFIGS["decode"]
    d = gen.decode_inputs(cfg, seed=0, device="cuda")
    o, lse, idx = msa.msa_sparse_decode(d["q"], d["q_idx"], d["k_cache"], d["v_cache"],
                                        d["k_idx_cache"], d["cu_seqlens"], cfg.len_hi, cfg.k)
    kp, vp, kip, pt, sl = to_pages(d, seed=1)
    del d["k_cache"], d["v_cache"], d["k_idx_cache"]
    o2, lse2, idx2 = msa.msa_sparse_decode_paged(d["q"], d["q_idx"], kp, vp, kip, pt, sl,
                                                 min(cfg.len_hi, 64 * pt.shape[1]), cfg.k)
    torch.cuda.synchronize()
    msa.msa_device_status()
    assert torch.equal(idx2, idx) and torch.equal(o2, o) and torch.equal(lse2, lse)
    del o, lse, idx
    kc, vc, kic, cu = unpage((kp, vp, kip), pt, sl)
    del kp, vp, kip
    dd = dict(q=d["q"], q_idx=d["q_idx"], k_cache=kc, v_cache=vc, k_idx_cache=kic, cu_seqlens=cu)
    check_decode_seqs(dd, cfg.k, o2, lse2, idx2)


def test_fullsize_prefill_varlen():
    """The benchmark's varlen batch (the 128K workload cut into 10 independent sequences) on
    sampled rows of every sequence against the oracle on that sequence alone."""
    cfg = gen.CONFIGS["p128k"]
    x = gen.prefill_inputs(cfg, seed=0, device="cuda")
    lens = [65536, 32768, 16384, 8192, 4096, 2048, 1024, 512, 256, 256]
    cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lens), 0)
    o, lse, idx = msa.msa_prefill_varlen(x["q"], x["k"], x["v"], x["q_idx"], x["k_idx"], cu,
                                         cfg.k)
    torch.cuda.synchronize()
    msa.msa_device_status()
    for s, n in enumerate(lens):
        t0 = int(cu[s])
        sl = slice(t0, t0 + n)
        xs = {k_: x[k_][sl] for k_ in ("q", "k", "v", "q_idx", "k_idx")}
        idx_s = idx[t0 * cfg.H_kv * cfg.k:(t0 + n) * cfg.H_kv * cfg.k].view(cfg.H_kv, n, cfg.k)
        lse_s = lse[t0 * cfg.H_q:(t0 + n) * cfg.H_q].view(cfg.H_q, n)
        check_prefill_rows(xs, cfg.k, idx_s, o[sl], lse_s, sample_rows(n, 96, seed=10 + s))
