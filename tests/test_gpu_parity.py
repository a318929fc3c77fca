"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded
inputs, at sizes that span several tiles plus ragged tails, and on the degenerate cases.

Bars:  block scores -- exact on small-integer inputs at d_idx=64 (fp32 dot products exact,
       scale 1/8 exact), <= 1 ulp at d_idx=32 (scale rounded once), fp32-accumulation
       tolerance on Gaussian inputs;  selection -- bit-exact when both sides see the same
       fp32 block scores; end to end, exact on integer inputs and exact up to near-ties
       (< 1e-3 relative) on Gaussian inputs;  O max-abs <= 2e-2, LSE abs <= 1e-3 against the
       oracle evaluated on the GPU's own selection."""
import numpy as np
import pytest
import torch

import gen
import oracle
from msa_testutil import (LSE_TOL, O_TOL, bits, check_decode_seqs, check_prefill_rows, cuda,
                          max_abs, selection_mismatches, to_pages, unpage)

pytestmark = pytest.mark.gpu

msa = pytest.importorskip("block_sparse_gqa_scores_gb300")


def cfg_of(name, **kw):
    base = gen.CONFIGS[name]
    return gen.PrefillConfig(**{**base.__dict__, **kw}) if kw else base


def fresh(cfg, N=None, seed=0, variant="gauss"):
    x = gen.prefill_inputs(cfg, seed=seed, device="cuda", variant=variant, N=N)
    return x, bits(x)


def sync_ok():
    torch.cuda.synchronize()
    msa.msa_device_status()


# ---------------------------------------------------------------- block scores --

SCORE_CASES = [
    ("tiny", 1024, "gauss", 0), ("tiny", 1024, "gauss", 1), ("tiny", 1024, "gauss", 2),
    ("tiny", 1024, "int", 0), ("tiny", 777, "int", 3),
    ("p32k", 1, "gauss", 0), ("p32k", 63, "gauss", 0), ("p32k", 64, "gauss", 0),
    ("p32k", 65, "int", 0), ("p32k", 1000, "gauss", 0), ("p32k", 3000, "int", 1),
    ("p32k", 4099, "gauss", 2),
]


@pytest.mark.parametrize("name,N,variant,seed", SCORE_CASES)
def test_block_scores(name, N, variant, seed):
    cfg = cfg_of(name)
    x, b = fresh(cfg, N, seed, variant)
    M = msa.msa_index_block_scores(x["q_idx"], x["k_idx"])
    sync_ok()
    M = M.cpu().numpy()
    _, ref = oracle.block_scores(b["q_idx"], b["k_idx"])
    assert np.array_equal(np.isneginf(M), np.isneginf(ref))
    fin = np.isfinite(ref)
    if variant == "int":
        if cfg.d_idx == 64:
            assert np.array_equal(M[fin], ref[fin])
        else:
            ulp = np.abs(M[fin].view(np.int32).astype(np.int64) - ref[fin].view(np.int32))
            assert ulp.max() <= 1
    else:
        np.testing.assert_allclose(M[fin], ref[fin], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("q_start,q_count", [(0, 1), (100, 333), (2999, 1), (64, 1000), (1, 2998)])
def test_block_scores_query_range(q_start, q_count):
    cfg = cfg_of("p32k")
    x, b = fresh(cfg, 3000, 5, "int")
    M = msa.msa_index_block_scores(x["q_idx"], x["k_idx"], q_start=q_start, q_count=q_count)
    sync_ok()
    _, ref = oracle.block_scores(b["q_idx"], b["k_idx"], q_start=q_start, q_count=q_count)
    assert np.array_equal(M.cpu().numpy(), ref)


# ------------------------------------------------------------------- selection --

def synthetic_scores(H_kv, N, q_start, q_count, kind, seed):
    """Block-score tensors with -inf after each row's own block: Gaussian, small integers
    (many ties) or all equal (ties everywhere)."""
    rng = np.random.default_rng(seed)
    nblk = -(-N // 64)
    if kind == "gauss":
        M = rng.standard_normal((H_kv, q_count, nblk)).astype(np.float32)
    elif kind == "intM":
        M = rng.integers(0, 4, (H_kv, q_count, nblk)).astype(np.float32)
    else:
        M = np.zeros((H_kv, q_count, nblk), np.float32)
    l = (np.arange(q_start, q_start + q_count) // 64)[None, :, None]
    M[np.broadcast_to(np.arange(nblk)[None, None, :] > l, M.shape)] = -np.inf
    return M


SELECT_CASES = [
    (2, 1024, 0, 1024, 4, "gauss"), (2, 1024, 0, 1024, 4, "intM"), (4, 5000, 0, 5000, 16, "gauss"),
    (4, 5000, 0, 5000, 16, "intM"), (4, 5000, 0, 5000, 16, "const"), (4, 5000, 0, 5000, 1, "gauss"),
    (4, 5000, 0, 5000, 2, "intM"), (4, 5000, 0, 5000, 33, "gauss"), (4, 5000, 0, 5000, 64, "intM"),
    (4, 70000, 60000, 2000, 16, "gauss"), (4, 70000, 60000, 2000, 16, "intM"),
    (4, 70000, 65000, 300, 64, "const"), (8, 20000, 19000, 1000, 16, "gauss"),
    (1, 300000, 299000, 1000, 16, "gauss"),
]


@pytest.mark.parametrize("H_kv,N,q_start,q_count,k,kind", SELECT_CASES)
def test_select_bit_exact(H_kv, N, q_start, q_count, k, kind):
    M = synthetic_scores(H_kv, N, q_start, q_count, kind, seed=N + k)
    ref = oracle.select_blocks(M, N, k, q_start=q_start)
    idx = msa.msa_select_blocks(torch.from_numpy(M).cuda(), N, k, q_start=q_start)
    sync_ok()
    assert np.array_equal(idx.cpu().numpy(), ref)


# ------------------------------------------------------------------ main branch --

ATTN_CASES = [
    ("tiny", {}, 1024, 4), ("tiny", {}, 1024, 1), ("tiny", {}, 1024, 64),
    ("p32k", {}, 1, 16), ("p32k", {}, 63, 16), ("p32k", {}, 64, 16), ("p32k", {}, 65, 16),
    ("p32k", {}, 1000, 16), ("p32k", {}, 1000, 64), ("p32k", {}, 2500, 16),
    ("p32k", dict(H_q=4, H_kv=4), 700, 8), ("p32k", dict(H_q=8, H_kv=4), 700, 8),
    ("p32k", dict(H_q=16, H_kv=4), 700, 8), ("p32k", dict(H_q=8, H_kv=1), 700, 5),
    ("p32k", dict(d_h=64), 900, 16), ("tiny", dict(d_h=128), 900, 4),
]


@pytest.mark.parametrize("name,over,N,k", ATTN_CASES)
def test_sparse_attention(name, over, N, k):
    cfg = cfg_of(name, k=k, **over)
    x, b = fresh(cfg, N, seed=11)
    _, M32 = oracle.block_scores(b["q_idx"], b["k_idx"])
    I = oracle.select_blocks(M32, N, k)
    O64, _, L = oracle.sparse_attn(b["q"], b["k"], b["v"], I)
    o, lse = msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], torch.from_numpy(I).cuda())
    sync_ok()
    assert max_abs(o.float().cpu().numpy(), O64) <= O_TOL
    assert max_abs(lse.cpu().numpy().T, L) <= LSE_TOL


def test_sparse_attention_zero_query_closed_form():
    """Q = 0: LSE = ln|T| and O = mean of V over T, on the GPU."""
    cfg = cfg_of("p32k")
    x, b = fresh(cfg, 1500, seed=3, variant="zero_q")
    _, M32 = oracle.block_scores(b["q_idx"], b["k_idx"])
    I = oracle.select_blocks(M32, 1500, 16)
    _, lse = msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], torch.from_numpy(I).cuda())
    sync_ok()
    i = np.arange(1500)
    T = np.minimum(i + 1, 15 * 64 + i % 64 + 1)
    assert np.abs(lse.cpu().numpy() - np.log(T)[None, :]).max() <= 1e-4


# ---------------------------------------------------------- fused index branch --
# msa_index_select must write exactly what msa_select_blocks writes from the block scores of
# msa_index_block_scores (same fp32 scores, same ordering), and so match the oracle wherever
# the unfused path does.

FUSED_CASES = [
    ("tiny", {}, 1024, "gauss", 0, 4, 0, None), ("tiny", {}, 1024, "int", 0, 4, 0, None),
    ("tiny", {}, 777, "int", 3, 2, 0, None), ("tiny", {}, 1024, "gauss", 1, 1, 0, None),
    ("tiny", {"H_kv": 1}, 1000, "gauss", 0, 4, 0, None),
    ("tiny", {"H_kv": 8}, 1000, "int", 0, 5, 0, None),
    ("tiny", {"d_idx": 64}, 1024, "gauss", 2, 4, 0, None),
    ("p32k", {}, 1, "gauss", 0, 16, 0, None), ("p32k", {}, 63, "gauss", 0, 16, 0, None),
    ("p32k", {}, 65, "int", 0, 16, 0, None), ("p32k", {}, 3000, "gauss", 0, 16, 0, None),
    ("p32k", {}, 4099, "int", 1, 32, 0, None), ("p32k", {}, 4099, "gauss", 2, 16, 0, None),
    ("p32k", {}, 4099, "gauss", 0, 16, 1000, 2000), ("p32k", {}, 3000, "int", 0, 16, 2999, 1),
    ("p128k", {}, 4500, "gauss", 0, 16, 0, None), ("p32k", {}, 32768, "gauss", 0, 16, 0, None),
]


@pytest.mark.parametrize("name,over,N,variant,seed,k,q_start,q_count", FUSED_CASES)
def test_index_select_equals_scores_then_select(name, over, N, variant, seed, k, q_start, q_count):
    if "H_kv" in over:
        over = {**over, "H_q": 8 * over["H_kv"]}
    cfg = cfg_of(name, **over)
    x, b = fresh(cfg, N, seed, variant)
    qc = N - q_start if q_count is None else q_count
    fused = msa.msa_index_select(x["q_idx"], x["k_idx"], k, q_start=q_start, q_count=qc)
    M = msa.msa_index_block_scores(x["q_idx"], x["k_idx"], q_start=q_start, q_count=qc)
    ref = msa.msa_select_blocks(M, N, k, q_start=q_start)
    sync_ok()
    assert torch.equal(fused, ref)
    if variant == "int" and N <= 4099:
        _, M_ref = oracle.block_scores(b["q_idx"], b["k_idx"], q_start=q_start, q_count=qc)
        I_ref = oracle.select_blocks(M_ref, N, k, q_start=q_start)
        assert np.array_equal(fused.cpu().numpy(), I_ref)


@pytest.mark.parametrize("trend,k", [("rising", 32), ("rising", 2), ("falling", 16), ("flat", 16)])
def test_index_select_score_trends(trend, k):
    """Block scores that rise with the block index make every block a candidate (the most
    compactions); falling scores fill the buffer once; flat scores tie everywhere, where the
    closed form is I = {0, ..., k-2} U {l}."""
    N, H_kv, d_idx = 8192, 4, 64
    j = torch.arange(N, device="cuda")
    val = {"rising": (j // 64) % 200, "falling": 199 - (j // 64) % 200, "flat": 0 * j}[trend]
    k_idx = (val.float()[:, None] / 8).expand(N, d_idx).to(torch.bfloat16).contiguous()
    q_idx = torch.ones((N, H_kv, d_idx), dtype=torch.bfloat16, device="cuda")
    fused = msa.msa_index_select(q_idx, k_idx, k)
    M = msa.msa_index_block_scores(q_idx, k_idx)
    ref = msa.msa_select_blocks(M, N, k)
    sync_ok()
    assert torch.equal(fused, ref)
    if trend == "flat":
        I = fused.cpu().numpy()
        for i in (0, 63, 64, 1000, N - 1):
            l = i // 64
            want = list(range(min(l, k - 1))) + [l]
            want += [-1] * (k - len(want))
            assert I[:, i].tolist() == [want] * H_kv


# ------------------------------------------------------------------- end to end --

@pytest.mark.parametrize("name,N,variant,seed", [("tiny", 1024, "gauss", 0), ("tiny", 1024, "gauss", 1),
                                                 ("tiny", 1024, "gauss", 2), ("tiny", 1024, "int", 0),
                                                 ("p32k", 3000, "gauss", 0), ("p32k", 3000, "int", 0),
                                                 ("p128k", 4500, "gauss", 0)])
def test_prefill_chain(name, N, variant, seed):
    cfg = cfg_of(name)
    x, b = fresh(cfg, N, seed, variant)
    M = msa.msa_index_block_scores(x["q_idx"], x["k_idx"])
    idx = msa.msa_select_blocks(M, N, cfg.k)
    o, lse = msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], idx)
    sync_ok()
    _, M_ref = oracle.block_scores(b["q_idx"], b["k_idx"])
    I_ref = oracle.select_blocks(M_ref, N, cfg.k)
    I_gpu = idx.cpu().numpy()
    if variant == "int":
        assert np.array_equal(I_gpu, I_ref)
    else:
        differ, bad = selection_mismatches(I_gpu, I_ref, M_ref, cfg.k)
        assert not bad, bad[:5]
        assert differ <= max(2, I_ref.shape[0] * N // 200)
    O64, _, L = oracle.sparse_attn(b["q"], b["k"], b["v"], I_gpu)
    assert max_abs(o.float().cpu().numpy(), O64) <= O_TOL
    assert max_abs(lse.cpu().numpy().T, L) <= LSE_TOL


# ---------------------------------------------------------------- KL alignment loss --
# The GPU loss (teacher normalised by the GPU forward's LSE) against the oracle evaluated on the
# GPU's own selection.  Tolerance: fp32 dot products of bf16 inputs and the forward's fp32 LSE
# leave ~1e-5 in each exponent; ex2/lg2 approximations ~2^-22 relative; fp32 sums of <= 1024
# terms of magnitude <= ~30 in C = sum P (ln P - S^idx) and in LSE^idx * sum P, which cancel
# down to the KL: a few 1e-5 typical, so 5e-4 + 1e-3 |KL| leaves a wide margin.
KL_ATOL, KL_RTOL = 5e-4, 1e-3

KL_CASES = [
    ("tiny", {}, 1024, 4), ("tiny", {}, 1000, 4), ("tiny", {}, 1024, 1), ("tiny", {}, 1024, 64),
    ("p32k", {}, 1, 16), ("p32k", {}, 65, 16), ("p32k", {}, 3000, 16), ("p32k", {}, 2500, 64),
    ("p32k", dict(H_q=4, H_kv=4), 700, 8), ("p32k", dict(H_q=8, H_kv=4), 700, 8),
    ("p32k", dict(H_q=16, H_kv=4), 700, 8), ("p32k", dict(H_q=8, H_kv=1), 700, 5),
    ("p32k", dict(d_h=64), 900, 16), ("tiny", dict(d_h=128), 900, 4),
    ("p32k", dict(d_idx=32), 900, 16),
]


def gpu_index(x, cfg, N):
    if cfg.k <= 32:
        return msa.msa_index_select(x["q_idx"], x["k_idx"], cfg.k)
    return msa.msa_select_blocks(msa.msa_index_block_scores(x["q_idx"], x["k_idx"]), N, cfg.k)


def check_kl(kl, ref):
    got = kl.cpu().numpy().T                                   # [N, H_kv]
    err = np.abs(got.astype(np.float64) - ref)
    assert np.isfinite(got).all()
    assert (err <= KL_ATOL + KL_RTOL * np.abs(ref)).all(), float(err.max())


@pytest.mark.parametrize("name,over,N,k", KL_CASES)
def test_kl_loss(name, over, N, k):
    cfg = cfg_of(name, k=k, **over)
    x, b = fresh(cfg, N, seed=21)
    idx = gpu_index(x, cfg, N)
    _, lse = msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], idx)
    kl = msa.msa_kl_loss_fwd(x["q"], x["k"], x["q_idx"], x["k_idx"], idx, lse)
    sync_ok()
    ref = oracle.kl_loss(b["q"], b["k"], b["q_idx"], b["k_idx"], idx.cpu().numpy())
    check_kl(kl, ref)
    assert ref.max() > 0.05 or N == 1                            # a loss that is not trivially 0


def test_kl_loss_zero_when_student_equals_teacher():
    """One head per group, d_idx = d_h = 64, q_idx = q and k_idx = k: the student's scores are
    the teacher's, so the loss is 0 up to the forward LSE's rounding."""
    cfg = cfg_of("p32k", H_q=1, H_kv=1, d_h=64, d_idx=64, k=8)
    x, _ = fresh(cfg, 2000, seed=22)
    x["q_idx"] = x["q"].clone()
    x["k_idx"] = x["k"][:, 0].contiguous()
    idx = msa.msa_index_select(x["q_idx"], x["k_idx"], 8)
    _, lse = msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], idx)
    kl = msa.msa_kl_loss_fwd(x["q"], x["k"], x["q_idx"], x["k_idx"], idx, lse)
    sync_ok()
    assert float(kl.abs().max()) <= 1e-4


def test_kl_loss_uniform_teacher():
    """Q = 0: the teacher is uniform over T, the oracle's closed-form case, on the GPU."""
    cfg = cfg_of("p32k")
    x, b = fresh(cfg, 1500, seed=23, variant="zero_q")
    idx = msa.msa_index_select(x["q_idx"], x["k_idx"], 16)
    _, lse = msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], idx)
    kl = msa.msa_kl_loss_fwd(x["q"], x["k"], x["q_idx"], x["k_idx"], idx, lse)
    sync_ok()
    check_kl(kl, oracle.kl_loss(b["q"], b["k"], b["q_idx"], b["k_idx"], idx.cpu().numpy()))


# ---------------------------------------- KL gradient (index branch, teacher fixed) --

KLB_CASES = [("p32k", {}, 1000, 16), ("p32k", {}, 65, 16), ("p32k", {}, 3000, 16),
             ("p32k", {}, 2500, 64), ("p32k", dict(d_idx=32), 900, 16),
             ("p32k", dict(d_h=64), 900, 16), ("p32k", dict(H_q=8, H_kv=1), 700, 5),
             # G = 1, 2, 4 (more entries per work tile), at both head sizes
             ("p32k", dict(H_q=4, H_kv=4), 700, 8), ("p32k", dict(H_q=8, H_kv=4), 1500, 16),
             ("p32k", dict(H_q=16, H_kv=4), 2000, 16), ("tiny", {}, 1024, 4),
             ("p32k", dict(H_q=4, H_kv=4, d_h=64), 900, 16),
             ("p32k", dict(H_q=8, H_kv=4, d_h=64, d_idx=32), 700, 8),
             ("p32k", dict(H_q=8, H_kv=4, d_h=64), 1200, 16), ("p32k", dict(H_q=16, H_kv=2), 1100, 64),
             ("tiny", dict(d_h=128), 1000, 64)]


@pytest.mark.parametrize("name,over,N,k", KLB_CASES)
def test_kl_loss_grad(name, over, N, k):
    """dQ_idx and dK_idx of sum(g * KL) against the oracle's fp64 gradient on the GPU's own
    selection.  Bound: the same fp32 error sources as the loss (about 1e-5 relative in each
    probability), plus the fp32 sums over every selecting row in dK_idx: 1e-3 of the largest
    magnitude.  Both are combined in a fixed order (no atomics), so a second call gives the
    same bits."""
    cfg = cfg_of(name, k=k, **over)
    x, b = fresh(cfg, N, seed=41)
    idx = gpu_index(x, cfg, N)
    _, lse = msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], idx)
    lse_idx = torch.empty((cfg.H_kv, N), dtype=torch.float32, device="cuda")
    psum = torch.empty_like(lse_idx)
    msa.msa_kl_loss_fwd(x["q"], x["k"], x["q_idx"], x["k_idx"], idx, lse, lse_idx=lse_idx,
                        p_sum=psum)
    g = torch.rand((cfg.H_kv, N), generator=torch.Generator(device="cuda").manual_seed(3),
                   device="cuda") * 1.5 + 0.5
    dq, dk = msa.msa_kl_loss_bwd(x["q"], x["k"], x["q_idx"], x["k_idx"], idx, lse, lse_idx, psum, g)
    sync_ok()
    ref = oracle.kl_loss_grad(b["q"], b["k"], b["q_idx"], b["k_idx"], idx.cpu().numpy(),
                              g.cpu().numpy().astype(np.float64))
    for got, want in ((dq, ref["dq_idx"]), (dk, ref["dk_idx"])):
        got = got.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert np.abs(got - want).max() <= 1e-3 * np.abs(want).max() + 1e-6, \
            float(np.abs(got - want).max())
    assert np.abs(lse_idx.cpu().numpy() - ref["lse_idx"]).max() <= 1e-3
    assert np.abs(psum.cpu().numpy() - ref["psum"]).max() <= 1e-4
    dq2, dk2 = msa.msa_kl_loss_bwd(x["q"], x["k"], x["q_idx"], x["k_idx"], idx, lse, lse_idx, psum,
                                   g)
    sync_ok()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2)


# ------------------------------------------------------- main-branch backward --
# dQ, dK, dV of the main branch against the oracle's fp64 gradient (which recomputes P and
# D = sum_j P_j dP_j itself) on the GPU's own selection.  Bound: P and dS enter the tensor-core
# products rounded to bf16 (2^-9 relative each), D comes from the bf16-rounded forward output,
# and the sums run in fp32 over at most 1024 tokens (dQ) or every selecting row (dK, dV): errors
# of a few 1e-3 of each tensor's largest magnitude, so 1e-2 of it leaves a wide margin.  Where a
# gradient vanishes exactly (a row with one visible token has dS = dP - D = 0), what remains is
# the fp32 rounding of the d_h-term dot products dP and D that cancel (|dP| ~ sqrt(d_h)): a floor
# of 1e-4 covers it with margin.
BWD_RTOL = 1e-2
BWD_ATOL = 1e-4

BWD_CASES = [
    ("tiny", {}, 1024, 4), ("tiny", {}, 4500, 4), ("tiny", {}, 1024, 64),
    ("p32k", {}, 1, 16), ("p32k", {}, 65, 16), ("p32k", {}, 1000, 16), ("p32k", {}, 2500, 16),
    ("p32k", dict(H_q=4, H_kv=4), 700, 8), ("p32k", dict(H_q=8, H_kv=4), 700, 8),
    ("p32k", dict(H_q=16, H_kv=4), 700, 8), ("p32k", dict(H_q=8, H_kv=1), 700, 5),
    ("p32k", dict(d_h=64), 900, 16), ("tiny", dict(d_h=128), 900, 4),
]


@pytest.mark.parametrize("name,over,N,k", BWD_CASES)
def test_sparse_attn_bwd(name, over, N, k):
    cfg = cfg_of(name, k=k, **over)
    x, b = fresh(cfg, N, seed=51)
    idx = gpu_index(x, cfg, N)
    o, lse = msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], idx)
    g = torch.Generator(device="cuda").manual_seed(5)
    d_o = torch.randn(x["q"].shape, generator=g, device="cuda").to(torch.bfloat16)
    dq, dk, dv = msa.msa_sparse_attn_bwd(x["q"], x["k"], x["v"], idx, o, lse, d_o)
    sync_ok()
    ref = oracle.sparse_attn_grad(b["q"], b["k"], b["v"], gen.to_bits(d_o), idx.cpu().numpy())
    for got, nm in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        got = got.cpu().numpy().astype(np.float64)
        want = ref[nm]
        assert np.isfinite(got).all(), nm
        err, scale = float(np.abs(got - want).max()), float(np.abs(want).max())
        assert err <= BWD_RTOL * scale + BWD_ATOL, (nm, err, scale)
    # deterministic: no atomic updates, so a second call gives the same bits
    dq2, dk2, dv2 = msa.msa_sparse_attn_bwd(x["q"], x["k"], x["v"], idx, o, lse, d_o)
    sync_ok()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


# -------------------------------------------------------------- varlen prefill --

@pytest.mark.parametrize("name,over,lens", [("p32k", {}, [1, 63, 64, 65, 1000, 3000, 4500]),
                                            ("tiny", {}, [700, 1, 1024, 129]),
                                            ("p32k", {}, [40000, 2000]),
                                            # lengths on the 128-row alignment: rows used in place
                                            ("p32k", {}, [2048, 128, 4096, 2048]),
                                            # H_kv = 1: 256-row alignment
                                            ("p32k", dict(H_q=8, H_kv=1), [300, 1500, 256]),
                                            ("tiny", dict(d_h=128, k=8), [5000, 77])])
def test_prefill_varlen_equals_single_sequences(name, over, lens):
    """A packed batch of independent sequences gives, per sequence, exactly the single-sequence
    results (positions restart at each sequence), whether the batch's rows are used in place or
    gathered into the aligned virtual rows."""
    cfg = cfg_of(name, **over)
    T = sum(lens)
    x, _ = fresh(cfg, T, seed=31)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lens), 0)
    o, lse, idx = msa.msa_prefill_varlen(x["q"], x["k"], x["v"], x["q_idx"], x["k_idx"], cu, cfg.k)
    sync_ok()
    for s_, n in enumerate(lens):
        t0 = int(cu[s_])
        sl = slice(t0, t0 + n)
        xs = {k_: x[k_][sl].contiguous() for k_ in ("q", "k", "v", "q_idx", "k_idx")}
        idx1 = msa.msa_index_select(xs["q_idx"], xs["k_idx"], cfg.k)
        o1, lse1 = msa.msa_sparse_attn_fwd(xs["q"], xs["k"], xs["v"], idx1)
        sync_ok()
        assert torch.equal(idx[t0 * cfg.H_kv * cfg.k:(t0 + n) * cfg.H_kv * cfg.k],
                           idx1.reshape(-1))
        assert torch.equal(o[sl], o1)
        assert torch.equal(lse[t0 * cfg.H_q:(t0 + n) * cfg.H_q], lse1.reshape(-1))
        # and against the oracle on the sequence alone (positions restart at 0)
        rows = np.unique(np.concatenate([np.arange(min(n, 70)), np.arange(max(0, n - 70), n),
                                         np.random.default_rng(s_).choice(n, min(n, 200),
                                                                          replace=False)]))
        check_prefill_rows(xs, cfg.k, idx1, o[sl], lse[t0 * cfg.H_q:(t0 + n) * cfg.H_q]
                           .view(cfg.H_q, n), rows, min_same=0.0 if n < 200 else 0.9)


# ------------------------------------------------------------------------ decode --

def decode_case(cfg, lens, seed, variant="gauss"):
    d = gen.decode_inputs(cfg, seed=seed, device="cuda", S=len(lens), len_lo=1, len_hi=1,
                          variant=variant)
    # replace the drawn lengths with the requested ones (same generator for the payload)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lens), 0)
    total = int(cu[-1])
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 17)
    draw = (lambda shape: torch.randint(-3, 4, shape, generator=g, device="cuda").float()) \
        if variant == "int" else (lambda shape: torch.randn(*shape, generator=g, device="cuda"))
    bf = torch.bfloat16
    d["k_cache"] = draw((total, cfg.H_kv, cfg.d_h)).to(bf)
    d["v_cache"] = draw((total, cfg.H_kv, cfg.d_h)).to(bf)
    d["k_idx_cache"] = draw((total, cfg.d_idx)).to(bf)
    d["cu_seqlens"] = cu.cuda()
    return d


def check_decode(cfg, d, max_len, exact_idx):
    o, lse, idx = msa.msa_sparse_decode(d["q"], d["q_idx"], d["k_cache"], d["v_cache"],
                                        d["k_idx_cache"], d["cu_seqlens"], max_len, cfg.k)
    sync_ok()
    b = bits(d)
    cu = d["cu_seqlens"].cpu().numpy()
    ref = oracle.decode(b["q"], b["q_idx"], b["k_cache"], b["v_cache"], b["k_idx_cache"], cu,
                        cfg.k, want_m=True)
    I_gpu = idx.cpu().numpy()                       # [S, H_kv, k]
    if exact_idx:
        assert np.array_equal(I_gpu, ref["I"])
    else:
        differ, bad = selection_mismatches(I_gpu.transpose(1, 0, 2), ref["I"].transpose(1, 0, 2),
                                           ref["M32"].transpose(1, 0, 2), cfg.k,
                                           rows=(cu[1:] - cu[:-1] - 1))
        assert not bad, bad
    # main branch on the GPU's own selection, one sequence at a time
    o_np, lse_np = o.float().cpu().numpy(), lse.cpu().numpy()
    for s in range(len(cu) - 1):
        L = int(cu[s + 1] - cu[s])
        sl = slice(int(cu[s]), int(cu[s + 1]))
        q = np.zeros((L, cfg.H_q, cfg.d_h), np.uint16)
        q[L - 1] = b["q"][s]
        I = np.full((cfg.H_kv, L, cfg.k), -1, np.int32)
        I[:, L - 1] = I_gpu[s]
        O64, _, Lr = oracle.sparse_attn(q, b["k_cache"][sl], b["v_cache"][sl], I, rows=[L - 1])
        assert max_abs(o_np[s], O64[0]) <= O_TOL
        assert max_abs(lse_np[s], Lr[0]) <= LSE_TOL


@pytest.mark.parametrize("name,lens,variant", [
    ("p32k", [1, 2, 63, 64, 65, 128, 1000, 1025, 5000, 4097], "gauss"),
    ("p32k", [70, 3000, 129, 64 * 17, 2049], "int"),
    ("tiny", [1, 100, 900, 1024, 333], "gauss"),
    ("tiny", [5, 700, 64, 2000], "int"),
])
def test_decode(name, lens, variant):
    cfg = cfg_of(name)
    dcfg = gen.DecodeConfig("t", len(lens), 1, 1, cfg.H_q, cfg.H_kv, cfg.d_h, cfg.d_idx, cfg.k)
    d = decode_case(dcfg, lens, seed=len(lens), variant=variant)
    check_decode(dcfg, d, max(lens) + 37, exact_idx=(variant == "int"))


@pytest.mark.parametrize("name,lens,variant", [
    ("p32k", [1, 2, 63, 64, 65, 128, 1000, 1025, 5000, 4097], "gauss"),
    ("p32k", [70, 3000, 129, 64 * 17, 2049], "int"),
    ("tiny", [1, 100, 900, 1024, 333], "gauss"),
])
def test_decode_paged_equals_packed(name, lens, variant):
    """The paged cache holds the same tokens in shuffled 64-token pages: the results equal the
    packed decode's bit for bit (same arithmetic in the same order), which the oracle pins."""
    cfg = cfg_of(name)
    dcfg = gen.DecodeConfig("t", len(lens), 1, 1, cfg.H_q, cfg.H_kv, cfg.d_h, cfg.d_idx, cfg.k)
    d = decode_case(dcfg, lens, seed=len(lens) + 7, variant=variant)
    max_len = max(lens) + 37
    o, lse, idx = msa.msa_sparse_decode(d["q"], d["q_idx"], d["k_cache"], d["v_cache"],
                                        d["k_idx_cache"], d["cu_seqlens"], max_len, dcfg.k)
    kp, vp, kip, pt, sl = to_pages(d, seed=len(lens))
    # max_len may exceed 64 * max_pages only up to the table's width
    max_len_p = min(max_len, 64 * pt.shape[1])
    o2, lse2, idx2 = msa.msa_sparse_decode_paged(d["q"], d["q_idx"], kp, vp, kip, pt, sl,
                                                 max_len_p, dcfg.k)
    sync_ok()
    assert torch.equal(idx2, idx)
    assert torch.equal(o2, o)
    assert torch.equal(lse2, lse)
    # and against the oracle on the tokens gathered back from the pages
    kc, vc, kic, cu = unpage((kp, vp, kip), pt, sl)
    dd = dict(q=d["q"], q_idx=d["q_idx"], k_cache=kc, v_cache=vc, k_idx_cache=kic, cu_seqlens=cu)
    check_decode_seqs(dd, dcfg.k, o2, lse2, idx2, exact_idx=(variant == "int"))


def test_decode_equals_prefill_last_row():
    cfg = cfg_of("p32k")
    x, _ = fresh(cfg, 2000, seed=4, variant="int")      # exact scores on both index paths
    lens = [2000, 1500, 64, 1]
    cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lens), 0)
    cat = lambda t: torch.cat([t[:L] for L in lens])
    last = torch.tensor([L - 1 for L in lens], device="cuda")
    o_d, lse_d, idx_d = msa.msa_sparse_decode(
        x["q"][last].contiguous(), x["q_idx"][last].contiguous(), cat(x["k"]), cat(x["v"]),
        cat(x["k_idx"]), cu.cuda(), 2000, cfg.k)
    M = msa.msa_index_block_scores(x["q_idx"], x["k_idx"])
    idx = msa.msa_select_blocks(M, 2000, cfg.k)
    o, lse = msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], idx)
    sync_ok()
    assert torch.equal(idx_d.cpu(), idx[:, last].permute(1, 0, 2).cpu())
    assert (o_d.float() - o[last].float()).abs().max().item() <= O_TOL   # 1 bf16 ulp at |O|~3
    assert (lse_d - lse[:, last].T).abs().max().item() <= 1e-4


# ---------------------------------------------------------------- error handling --

def test_errors_are_reported():
    cfg = cfg_of("tiny")
    x, _ = fresh(cfg, 128)
    with pytest.raises(msa.MSAError) as e:
        msa.msa_index_block_scores(x["q_idx"], x["k_idx"], q_start=100, q_count=100)
    assert e.value.code == 1
    with pytest.raises(msa.MSAError) as e:
        msa.msa_sparse_attn_fwd(x["q"][:, :, :48].contiguous(), x["k"][:, :, :48].contiguous(),
                                x["v"][:, :, :48].contiguous(),
                                torch.zeros((2, 128, 4), dtype=torch.int32, device="cuda"))
    assert e.value.code == 2
    d = gen.decode_inputs(gen.CONFIGS["decode"], S=2, len_lo=100, len_hi=200, device="cuda")
    with pytest.raises(msa.MSAError) as e:
        msa.msa_sparse_decode(d["q"], d["q_idx"], d["k_cache"], d["v_cache"], d["k_idx_cache"],
                              d["cu_seqlens"], 200, 16, ws=torch.empty(64, dtype=torch.uint8,
                                                                       device="cuda"))
    assert e.value.code == 3
    sync_ok()
