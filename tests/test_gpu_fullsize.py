"""Full-size parity on the benchmark's own workloads, in the benchmark's launch configuration
(the same C-ABI calls on the full tensors), checked on sampled query rows / sequences that the
oracle recomputes one by one: 32K and 128K prefill, the 32-sequence decode batch, and 1M prefill
(query-chunked index scores).  Selections must match the oracle up to near-ties; O and LSE are
compared on rows whose selection matches exactly."""
import numpy as np
import pytest
import torch

import gen
import oracle
from msa_testutil import LSE_TOL, O_TOL, selection_mismatches, to_pages

pytestmark = pytest.mark.gpu

msa = pytest.importorskip("block_sparse_gqa_scores_gb300")


def sample_rows(N, n, seed):
    rng = np.random.default_rng(seed)
    edge = [0, 1, 63, 64, 65, N // 2, N - 65, N - 64, N - 1]
    rows = np.unique(np.concatenate([rng.choice(N, n, replace=False), [e for e in edge if e < N]]))
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


def check_rows(x, cfg, idx, o, lse, rows, M_last=None, chunk_start=None):
    b = {n: gen.to_bits(x[n]) for n in ("k", "v", "k_idx")}
    rows_t = torch.from_numpy(rows).cuda()
    qr = gen.to_bits(x["q"][rows_t])
    qir = gen.to_bits(x["q_idx"][rows_t])
    ref = oracle.prefill(qr, b["k"], b["v"], qir, b["k_idx"], cfg.k, rows=rows, want_m=True,
                         compact=True)
    I_gpu = idx[:, rows_t].cpu().numpy()                       # [H_kv, n, k]
    I_ref = ref["I"].transpose(1, 0, 2)
    differ, bad = selection_mismatches(I_gpu, I_ref, ref["M32"].transpose(1, 0, 2), cfg.k, rows=rows)
    assert not bad, bad[:5]
    same = (I_gpu == I_ref).all(axis=(0, 2))                   # rows with all groups identical
    assert same.mean() >= 0.9
    o_s = o[rows_t].float().cpu().numpy()
    l_s = lse[:, rows_t].cpu().numpy().T
    err_o = np.abs(o_s - ref["O64"]).max(axis=(1, 2))[same]
    err_l = np.abs(l_s - ref["LSE"]).max(axis=1)[same]
    assert err_o.max() <= O_TOL and err_l.max() <= LSE_TOL
    return differ


@pytest.mark.parametrize("name,n_rows", [("p32k", 48), ("p128k", 40)])
def test_fullsize_prefill(name, n_rows):
    cfg = gen.CONFIGS[name]
    x = gen.prefill_inputs(cfg, seed=0, device="cuda")
    idx, o, lse = run_prefill(x, cfg)
    # the fused index branch selects exactly what block scores + selection select
    assert torch.equal(idx, unfused_index(x, cfg))
    check_rows(x, cfg, idx, o, lse, sample_rows(cfg.N, n_rows, seed=1))


def test_fullsize_kl_loss():
    """The KL alignment loss at 128K, in the benchmark's launch sequence (fused index branch,
    main branch, KL forward), on sampled rows the oracle recomputes on the GPU's selection."""
    cfg = gen.CONFIGS["p128k"]
    x = gen.prefill_inputs(cfg, seed=0, device="cuda")
    idx, _, lse = run_prefill(x, cfg)
    kl = msa.msa_kl_loss_fwd(x["q"], x["k"], x["q_idx"], x["k_idx"], idx, lse)
    torch.cuda.synchronize()
    msa.msa_device_status()
    rows = sample_rows(cfg.N, 40, seed=3)
    rows_t = torch.from_numpy(rows).cuda()
    ref = oracle.kl_loss(gen.to_bits(x["q"][rows_t]), gen.to_bits(x["k"]),
                         gen.to_bits(x["q_idx"][rows_t]), gen.to_bits(x["k_idx"]),
                         idx[:, rows_t].cpu().numpy(), rows=rows, compact=True)
    got = kl[:, rows_t].cpu().numpy().T.astype(np.float64)
    assert np.isfinite(kl.cpu().numpy()).all() and float(kl.min()) >= -1e-3
    assert (np.abs(got - ref) <= 5e-4 + 1e-3 * np.abs(ref)).all(), float(np.abs(got - ref).max())


def test_fullsize_prefill_1m():
    cfg = gen.CONFIGS["p1m"]
    x = gen.prefill_inputs(cfg, seed=0, device="cuda")
    idx, o, lse = run_prefill(x, cfg)
    ref = unfused_index(x, cfg, chunk=16384)
    assert torch.equal(idx, ref)
    del ref
    check_rows(x, cfg, idx, o, lse, sample_rows(cfg.N, 8, seed=2))


def test_fullsize_decode():
    cfg = gen.CONFIGS["decode"]
    d = gen.decode_inputs(cfg, seed=0, device="cuda")
    o, lse, idx = msa.msa_sparse_decode(d["q"], d["q_idx"], d["k_cache"], d["v_cache"],
                                        d["k_idx_cache"], d["cu_seqlens"], cfg.len_hi, cfg.k)
    torch.cuda.synchronize()
    msa.msa_device_status()
    cu = d["cu_seqlens"].cpu().numpy()
    for s in (0, 13, 31):
        sl = slice(int(cu[s]), int(cu[s + 1]))
        L = int(cu[s + 1] - cu[s])
        sub = lambda n: gen.to_bits(d[n][sl])
        ref = oracle.decode(gen.to_bits(d["q"][s:s + 1]), gen.to_bits(d["q_idx"][s:s + 1]),
                            sub("k_cache"), sub("v_cache"), sub("k_idx_cache"),
                            np.array([0, L], np.int64), cfg.k, want_m=True)
        I_gpu = idx[s:s + 1].cpu().numpy()
        differ, bad = selection_mismatches(I_gpu.transpose(1, 0, 2), ref["I"].transpose(1, 0, 2),
                                           ref["M32"].transpose(1, 0, 2), cfg.k, rows=[L - 1])
        assert not bad
        if np.array_equal(I_gpu, ref["I"]):
            assert np.abs(o[s].float().cpu().numpy() - ref["O64"][0]).max() <= O_TOL
            assert np.abs(lse[s].cpu().numpy() - ref["LSE"][0]).max() <= LSE_TOL


def test_fullsize_decode_paged():
    """The 32-sequence decode batch from a paged cache (shuffled 64-token pages) equals the packed
    decode bit for bit."""
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
