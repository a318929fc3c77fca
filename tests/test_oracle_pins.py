"""Pins of the CPU oracle against things other than itself (CPU only).

Each test ties one oracle function to an independent fact: a brute-force dense
computation written with numpy, a library routine (torch SDPA), a closed form, the
hand-worked golden case, or an invariant of the selection rule.  Together they are
chosen so that a dropped term, a wrong sign or index, a transposed operand, a lost
causal mask, a wrong tie-break or a misplaced local block fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import gen
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def bits(x):
    return {k: gen.to_bits(v) for k, v in x.items() if k != "meta"}


def small_cfg(N=300, H_q=8, H_kv=2, d_h=16, d_idx=8, k=3):
    return gen.PrefillConfig("pin", N, H_q, H_kv, d_h, d_idx, k)


def f64(a):
    return gen.bf16_bits_to_f64(a)


# ------------------------------------------------------------- brute force --

def dense_block_scores(q_idx, k_idx, B):
    """numpy fp64: S = Q_idx K_idx^T / sqrt(d_idx), causal -inf, per-block max."""
    Qi, Ki = f64(q_idx), f64(k_idx)
    N, H_kv, d = Qi.shape
    nblk = -(-N // B)
    S = np.einsum("nrd,md->rnm", Qi, Ki) / math.sqrt(d)
    S = np.where(np.tril(np.ones((N, N), bool))[None], S, -np.inf)
    pad = nblk * B - N
    S = np.concatenate([S, np.full((H_kv, N, pad), -np.inf)], axis=2)
    return S.reshape(H_kv, N, nblk, B).max(axis=3)


def brute_select(M32, k, B):
    H_kv, N, nblk = M32.shape
    I = np.full((H_kv, N, k), -1, np.int32)
    for r in range(H_kv):
        for i in range(N):
            l = i // B
            if l + 1 <= k:
                sel = list(range(l + 1))
            else:
                order = np.argsort(-M32[r, i, :l].astype(np.float64), kind="stable")
                sel = sorted(order[: k - 1].tolist()) + [l]
            I[r, i, : len(sel)] = sel
    return I


def dense_masked_attention(q, k, v, I, B):
    """numpy fp64: full score matrix, then a boolean mask built from I and causality."""
    Q, K, V = f64(q), f64(k), f64(v)
    N, H_q, d = Q.shape
    H_kv = K.shape[1]
    G = H_q // H_kv
    blk = np.arange(N) // B
    O = np.zeros((N, H_q, d))
    L = np.zeros((N, H_q))
    for h in range(H_q):
        r = h // G
        S = Q[:, h, :] @ K[:, r, :].T / math.sqrt(d)
        sel = np.zeros((N, N), bool)
        for i in range(N):
            chosen = set(int(b) for b in I[r, i] if b >= 0)
            sel[i] = np.isin(blk, list(chosen)) & (np.arange(N) <= i)
        S = np.where(sel, S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        P = np.exp(S - m)
        Z = P.sum(axis=1, keepdims=True)
        L[:, h] = (m + np.log(Z))[:, 0]
        O[:, h, :] = (P / Z) @ V[:, r, :]
    return O, L


# ------------------------------------------------------------------- tests --

@pytest.mark.parametrize("variant", ["int", "gauss"])
def test_block_scores_match_dense_bruteforce(variant):
    cfg = small_cfg(N=200)
    x = bits(gen.prefill_inputs(cfg, seed=1, variant=variant))
    B = 16
    M64, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    ref = dense_block_scores(x["q_idx"], x["k_idx"], B)
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(M64))            # same -inf pattern (causal)
    np.testing.assert_allclose(M64[fin], ref[fin], rtol=1e-14, atol=0)
    if variant == "int":
        # integer inputs: the block maxima of the raw dots are exact integers
        raw = dense_block_scores(x["q_idx"], x["k_idx"], B) * math.sqrt(8)
        assert np.array_equal(np.rint(M64[fin] * math.sqrt(8)), np.rint(raw[fin]))
        assert np.abs(raw[fin] - np.rint(raw[fin])).max() < 1e-9
    assert np.array_equal(M32, M64.astype(np.float32))


def test_block_scores_query_range():
    cfg = small_cfg(N=150)
    x = bits(gen.prefill_inputs(cfg, seed=2))
    full64, _ = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=16)
    part64, _ = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=16, q_start=37, q_count=50)
    assert np.array_equal(part64, full64[:, 37:87])


@pytest.mark.parametrize("variant,seed", [("int", 0), ("int", 3), ("gauss", 0), ("gauss", 5)])
def test_select_matches_stable_argsort(variant, seed):
    cfg = small_cfg(N=260, k=4)
    x = bits(gen.prefill_inputs(cfg, seed=seed, variant=variant))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 260, 4, block_size=B)
    assert np.array_equal(I, brute_select(M32, 4, B))


def test_select_constant_scores_closed_form():
    """Constant K_idx: all visible block scores of a row are equal, so ties decide
    everything: I = {0..k-2} U {l} once l >= k-1, else all visible blocks."""
    cfg = small_cfg(N=400, k=5)
    x = bits(gen.prefill_inputs(cfg, seed=4, variant="const_kidx"))
    B = 16
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 400, 5, block_size=B)
    for i in range(400):
        l = i // B
        want = list(range(l + 1)) if l + 1 <= 5 else list(range(4)) + [l]
        want += [-1] * (5 - len(want))
        for r in range(2):
            assert I[r, i].tolist() == want


def test_select_invariants_and_query_range():
    cfg = small_cfg(N=333, k=6)
    x = bits(gen.prefill_inputs(cfg, seed=6))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B, q_start=100, q_count=200)
    I = oracle.select_blocks(M32, 333, 6, block_size=B, q_start=100)
    assert (I[:, :100] == -2).all() and (I[:, 300:] == -2).all()   # untouched rows
    for r in range(2):
        for i in range(100, 300):
            l = i // B
            row = I[r, i]
            sel = row[row >= 0]
            assert l in sel                                    # forced local block
            assert len(sel) == min(6, l + 1)                   # count
            assert (np.diff(sel) > 0).all()                    # distinct, ascending
            assert sel.max() == l                              # nothing in the future
            assert (row[len(sel):] == -1).all()                # -1 padding last
            others = sel[:-1]                                  # the k-1 best of b < l
            if l + 1 > 6:
                worst_in = M32[r, i - 100, others].min()
                rest = np.setdiff1d(np.arange(l), others)
                assert (M32[r, i - 100, rest] <= worst_in).all()


@pytest.mark.parametrize("variant", ["gauss", "int"])
def test_attention_matches_dense_masked(variant):
    cfg = small_cfg(N=120, d_h=16, k=3)
    x = bits(gen.prefill_inputs(cfg, seed=7, variant=variant))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 120, 3, block_size=B)
    O64, O16, L = oracle.sparse_attn(x["q"], x["k"], x["v"], I, block_size=B)
    Oref, Lref = dense_masked_attention(x["q"], x["k"], x["v"], I, B)
    np.testing.assert_allclose(O64, Oref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lref, rtol=0, atol=1e-12)
    # the stored bf16 output is the RNE rounding of the fp64 result
    torch_round = gen.to_bits(torch.from_numpy(O64).to(torch.float32).to(torch.bfloat16))
    assert (O16 == torch_round).mean() > 0.999   # fp64->fp32->bf16 double rounding differs rarely
    # the compact form (only some rows' queries and selections passed) on the same rows
    rows = np.array([0, 7, 8, 63, 64, 119, 33])
    Oc, _, Lc = oracle.sparse_attn(x["q"][rows], x["k"], x["v"], I[:, rows], block_size=B,
                                   rows=rows, compact=True)
    np.testing.assert_allclose(Oc, Oref[rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lc, Lref[rows], rtol=0, atol=1e-12)


def test_full_k_equals_causal_sdpa():
    """k >= number of blocks: every visible token is attended -> plain causal GQA
    attention, checked against torch's scaled_dot_product_attention in fp64."""
    cfg = small_cfg(N=96, H_q=8, H_kv=2, d_h=16, k=12)
    x = bits(gen.prefill_inputs(cfg, seed=8))
    B = 8
    out = oracle.prefill(x["q"], x["k"], x["v"], x["q_idx"], x["k_idx"], 12, block_size=B)
    Q = torch.from_numpy(f64(x["q"])).permute(1, 0, 2)[None]          # [1,H_q,N,d]
    K = torch.from_numpy(f64(x["k"])).permute(1, 0, 2)[None].repeat_interleave(4, dim=1)
    V = torch.from_numpy(f64(x["v"])).permute(1, 0, 2)[None].repeat_interleave(4, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True)[0]
    np.testing.assert_allclose(out["O64"], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    S = (Q @ K.transpose(-1, -2)) / math.sqrt(16)
    S = S.masked_fill(~torch.tril(torch.ones(96, 96, dtype=torch.bool)), float("-inf"))
    lse = torch.logsumexp(S, dim=-1)[0].T
    np.testing.assert_allclose(out["LSE"], lse.numpy(), rtol=0, atol=1e-12)


def test_zero_query_closed_form():
    """Q = 0: every visible selected token has score 0, so LSE = ln|T| and O is the
    plain mean of V over T, with |T| = min(i+1, (k-1)B + (i mod B) + 1)."""
    cfg = small_cfg(N=140, k=3)
    x = bits(gen.prefill_inputs(cfg, seed=9, variant="zero_q"))
    B = 8
    out = oracle.prefill(x["q"], x["k"], x["v"], x["q_idx"], x["k_idx"], 3, block_size=B)
    V = f64(x["v"])
    for i in range(140):
        T = min(i + 1, 2 * B + (i % B) + 1)
        np.testing.assert_allclose(out["LSE"][i], math.log(T), rtol=0, atol=1e-13)
        for r in range(2):
            toks = [j for b in out["I"][i, r] if b >= 0 for j in range(b * B, min(b * B + B, i + 1))]
            assert len(toks) == T
            for h in range(r * 4, r * 4 + 4):
                np.testing.assert_allclose(out["O64"][i, h], V[toks, r].mean(axis=0), atol=1e-13)


def test_handworked_golden():
    g = json.load(open(os.path.join(HERE, "golden", "handworked_tiny.json")))
    B, kk = g["block_size"], g["k_blocks"]

    def bf(a):
        return gen.to_bits(torch.tensor(a, dtype=torch.float32).to(torch.bfloat16))

    q, k, v = bf(g["q"]), bf(g["k"]), bf(g["v"])
    q_idx, k_idx = bf(g["q_idx"]), bf(g["k_idx"])
    M64, M32 = oracle.block_scores(q_idx, k_idx, block_size=B)
    for i, row in g["expected_M_raw_dots"].items():
        for b, val in enumerate(row):
            want = -math.inf if val is None else val / math.sqrt(2)
            assert M64[0, int(i), b] == pytest.approx(want, abs=1e-15)
    I = oracle.select_blocks(M32, 6, kk, block_size=B)
    for i, sel in g["expected_I"].items():
        assert I[0, int(i)].tolist() == sel
    O64, _, L = oracle.sparse_attn(q, k, v, I, block_size=B)
    env = {"a": 1 / math.sqrt(2), "exp": math.exp, "log": math.log}
    for i, e in g["expected_attn"].items():
        for h in range(2):
            assert L[int(i), h] == pytest.approx(eval(e["lse"][h], env), abs=1e-14)
            for d in range(2):
                assert O64[int(i), h, d] == pytest.approx(eval(e["o"][h][d], env), abs=1e-14)


def test_decode_equals_prefill_last_row():
    cfg = small_cfg(N=500, k=4)
    x = bits(gen.prefill_inputs(cfg, seed=10))
    B = 16
    lens = [1, 17, 64, 65, 333, 500]
    cu = np.zeros(len(lens) + 1, np.int64)
    cu[1:] = np.cumsum(lens)
    cat = lambda a: np.concatenate([a[:L] for L in lens])
    last = np.array([L - 1 for L in lens])
    dec = oracle.decode(x["q"][last], x["q_idx"][last], cat(x["k"]), cat(x["v"]), cat(x["k_idx"]),
                        cu, 4, block_size=B)
    pre = oracle.prefill(x["q"], x["k"], x["v"], x["q_idx"], x["k_idx"], 4, block_size=B, rows=last)
    assert np.array_equal(dec["I"], pre["I"])
    assert np.array_equal(dec["O64"], pre["O64"])
    assert np.array_equal(dec["LSE"], pre["LSE"])


def test_bf16_rounding_pins():
    """Direct fp64 -> bf16 round-to-nearest-even: equals torch's fp32 -> bf16 on values
    that are exact in fp32, and rounds ties to even without double rounding."""
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                           (rng.standard_normal(2000) * 1e-38).astype(np.float32),
                           np.float32([0.0, -0.0, 1.0, -1.0, 3.0e38])])
    want = gen.to_bits(torch.from_numpy(vals).to(torch.bfloat16))
    got = np.array([oracle.f64_to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, want)
    one = 0x3F80
    assert oracle.f64_to_bf16(1.0 + 2 ** -8) == one                        # tie -> even (down)
    assert oracle.f64_to_bf16(1.0 + 3 * 2 ** -8) == one + 2                # tie -> even (up)
    assert oracle.f64_to_bf16(1.0 + 2 ** -8 + 2 ** -40) == one + 1         # above the tie
    assert oracle.f64_to_bf16(-(1.0 + 2 ** -8 + 2 ** -40)) == 0x8000 | (one + 1)


def test_flop_ratio_closed_form():
    """The digest's 28.4x fewer attention FLOPs per token at 1M context (section 实验数字)
    is reproduced by counting visible-token work: full causal attention vs 2048 attended
    tokens plus the index branch's 4 heads x 64 dims over the causal prefix."""
    N, hq_dh, hidx_didx = 2 ** 20, 32 * 128, 4 * 64
    ratio = lambda T: (4 * hq_dh * N / 2) / (4 * hq_dh * T + 2 * hidx_didx * N / 2)
    assert round(ratio(2048), 1) == 28.4
    assert round(ratio(1024), 1) == 30.1


# ------------------------------------------------------ KL alignment loss --

def selected_token_mask(I, N, B):
    """Brute force: mask[r, i, j] = token j is visible from i and its block is in I[r, i]."""
    H_kv = I.shape[0]
    blk = np.arange(N) // B
    mask = np.zeros((H_kv, N, N), bool)
    for r in range(H_kv):
        for i in range(N):
            chosen = [int(b) for b in I[r, i] if b >= 0]
            mask[r, i] = np.isin(blk, chosen) & (np.arange(N) <= i)
    return mask


def library_kl(x, mask):
    """Teacher and student from torch.softmax over the masked fp64 scores; the KL from
    scipy.stats.entropy (sum p log(p/q)) row by row -> [N, H_kv]."""
    from scipy.stats import entropy
    Q, K = torch.from_numpy(f64(x["q"])), torch.from_numpy(f64(x["k"]))
    Qi, Ki = torch.from_numpy(f64(x["q_idx"])), torch.from_numpy(f64(x["k_idx"]))
    N, H_q, d_h = Q.shape
    H_kv, d_idx = K.shape[1], Qi.shape[2]
    G = H_q // H_kv
    m = torch.from_numpy(np.array(mask))
    out = np.zeros((N, H_kv))
    for r in range(H_kv):
        S = torch.einsum("nhd,md->hnm", Q[:, r * G:(r + 1) * G], K[:, r]) / math.sqrt(d_h)
        teacher = torch.softmax(S.masked_fill(~m[r], float("-inf")), dim=-1).mean(dim=0)
        Si = (Qi[:, r] @ Ki.T) / math.sqrt(d_idx)
        student = torch.softmax(Si.masked_fill(~m[r], float("-inf")), dim=-1)
        for i in range(N):
            sel = m[r, i]
            out[i, r] = entropy(teacher[i, sel].numpy(), student[i, sel].numpy())
    return out


def test_kl_full_k_equals_library_entropy():
    """k >= number of blocks: T is the whole causal prefix, so the loss is the KL of two
    plain causal softmaxes (torch.softmax), computed by scipy.stats.entropy."""
    cfg = small_cfg(N=96, H_q=8, H_kv=2, d_h=16, d_idx=8, k=12)
    x = bits(gen.prefill_inputs(cfg, seed=11))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 96, 12, block_size=B)
    KL = oracle.kl_loss(x["q"], x["k"], x["q_idx"], x["k_idx"], I, block_size=B)
    causal = np.broadcast_to(np.tril(np.ones((96, 96), bool)), (2, 96, 96))
    np.testing.assert_allclose(KL, library_kl(x, causal), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("variant,seed", [("gauss", 12), ("int", 13)])
def test_kl_sparse_matches_library_on_bruteforce_mask(variant, seed):
    cfg = small_cfg(N=120, H_q=8, H_kv=2, d_h=16, d_idx=8, k=3)
    x = bits(gen.prefill_inputs(cfg, seed=seed, variant=variant))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 120, 3, block_size=B)
    KL = oracle.kl_loss(x["q"], x["k"], x["q_idx"], x["k_idx"], I, block_size=B)
    np.testing.assert_allclose(KL, library_kl(x, selected_token_mask(I, 120, B)), rtol=1e-10,
                               atol=1e-12)
    rows = np.array([0, 7, 8, 63, 119])
    sub = oracle.kl_loss(x["q"], x["k"], x["q_idx"], x["k_idx"], I, block_size=B, rows=rows)
    assert np.array_equal(sub, KL[rows])


def test_kl_uniform_teacher_closed_form():
    """Q = 0: every head's softmax over T is uniform, so the teacher is 1/|T| and
    KL(U || softmax(x)) = logsumexp_T(x) - mean_T(x) - ln|T|, x the index scores over T,
    with |T| = min(i+1, (k-1)B + (i mod B) + 1)."""
    from scipy.special import logsumexp
    cfg = small_cfg(N=140, k=3)
    x = bits(gen.prefill_inputs(cfg, seed=14, variant="zero_q"))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 140, 3, block_size=B)
    KL = oracle.kl_loss(x["q"], x["k"], x["q_idx"], x["k_idx"], I, block_size=B)
    Qi, Ki = f64(x["q_idx"]), f64(x["k_idx"])
    for r in range(2):
        for i in range(140):
            toks = [j for b in I[r, i] if b >= 0 for j in range(b * B, min(b * B + B, i + 1))]
            assert len(toks) == min(i + 1, 2 * B + (i % B) + 1)
            s = Ki[toks] @ Qi[i, r] / math.sqrt(8)
            want = logsumexp(s) - s.mean() - math.log(len(toks))
            assert KL[i, r] == pytest.approx(want, abs=1e-12)


def test_kl_uniform_student_closed_form():
    """Q_idx = 0: the student is 1/|T|, so KL(P || U) = ln|T| - H(P), H the entropy of the
    teacher (the mean of the group's per-head causal softmaxes over T)."""
    from scipy.stats import entropy
    cfg = small_cfg(N=100, H_q=8, H_kv=2, d_h=16, d_idx=8, k=4)
    x = bits(gen.prefill_inputs(cfg, seed=15))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 100, 4, block_size=B)
    x["q_idx"] = np.zeros_like(x["q_idx"])
    KL = oracle.kl_loss(x["q"], x["k"], x["q_idx"], x["k_idx"], I, block_size=B)
    Q, K = f64(x["q"]), f64(x["k"])
    for r in range(2):
        for i in range(100):
            toks = [j for b in I[r, i] if b >= 0 for j in range(b * B, min(b * B + B, i + 1))]
            P = np.zeros(len(toks))
            for h in range(4 * r, 4 * r + 4):
                s = K[toks, r] @ Q[i, h] / 4.0
                e = np.exp(s - s.max())
                P += e / e.sum() / 4
            want = math.log(len(toks)) - entropy(P)
            assert KL[i, r] == pytest.approx(want, abs=1e-12)


def test_kl_zero_when_student_scores_equal_teacher():
    """d_idx = d_h, one KV head, both query heads equal to the index query and K_idx = K:
    the student's scores are the teacher's, so the loss is 0 on every row; a perturbed
    index query gives a strictly positive loss (Gibbs' inequality)."""
    cfg = small_cfg(N=130, H_q=2, H_kv=1, d_h=16, d_idx=16, k=3)
    x = bits(gen.prefill_inputs(cfg, seed=16))
    B = 8
    x["q"][:, 1] = x["q"][:, 0]
    x["q_idx"] = np.ascontiguousarray(x["q"][:, :1])
    x["k_idx"] = np.ascontiguousarray(x["k"][:, 0])
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 130, 3, block_size=B)
    KL = oracle.kl_loss(x["q"], x["k"], x["q_idx"], x["k_idx"], I, block_size=B)
    assert np.abs(KL).max() < 1e-13
    x["q_idx"] = gen.to_bits(gen.from_bits(x["q_idx"]) * 2)
    KL2 = oracle.kl_loss(x["q"], x["k"], x["q_idx"], x["k_idx"], I, block_size=B)
    assert (KL2[1:] > 0).all() and KL2[0, 0] == pytest.approx(0, abs=1e-15)   # |T| = 1 at i = 0


def test_kl_nonnegative_and_group_specific():
    """KL >= 0 on every row; swapping the two groups' query heads changes the loss (the
    teacher of group r averages heads r*G .. r*G+G-1 only)."""
    cfg = small_cfg(N=90, H_q=8, H_kv=2, d_h=16, d_idx=8, k=3)
    x = bits(gen.prefill_inputs(cfg, seed=17))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 90, 3, block_size=B)
    KL = oracle.kl_loss(x["q"], x["k"], x["q_idx"], x["k_idx"], I, block_size=B)
    assert (KL >= -1e-15).all() and KL.max() > 0.01
    y = dict(x)
    y["q"] = np.ascontiguousarray(x["q"][:, [4, 5, 6, 7, 0, 1, 2, 3]])
    KL_sw = oracle.kl_loss(y["q"], y["k"], y["q_idx"], y["k_idx"], I, block_size=B)
    assert np.abs(KL_sw - KL).max() > 1e-3
    y["q"] = np.ascontiguousarray(x["q"][:, [3, 2, 1, 0, 7, 6, 5, 4]])  # within-group order
    KL_perm = oracle.kl_loss(y["q"], y["k"], y["q_idx"], y["k_idx"], I, block_size=B)
    np.testing.assert_allclose(KL_perm, KL, rtol=1e-12, atol=1e-14)


# ------------------------------------------ KL gradient (index branch, teacher fixed) --

def autograd_kl_grad(x, I, g, B):
    """torch.autograd in fp64 through a dense masked restatement of the loss: teacher from
    torch.softmax (no gradient), student log-probabilities from torch.log_softmax over T."""
    N = x["q"].shape[0]
    Q, K = torch.from_numpy(f64(x["q"])), torch.from_numpy(f64(x["k"]))
    Qi = torch.from_numpy(f64(x["q_idx"])).requires_grad_(True)
    Ki = torch.from_numpy(f64(x["k_idx"])).requires_grad_(True)
    H_q, d_h = Q.shape[1], Q.shape[2]
    H_kv, d_idx = K.shape[1], Qi.shape[2]
    G = H_q // H_kv
    mask = torch.from_numpy(np.array(selected_token_mask(I, N, B)))
    loss = 0.0
    for r in range(H_kv):
        S = torch.einsum("nhd,md->hnm", Q[:, r * G:(r + 1) * G], K[:, r]) / math.sqrt(d_h)
        teacher = torch.softmax(S.masked_fill(~mask[r], float("-inf")), dim=-1).mean(dim=0)
        Si = (Qi[:, r] @ Ki.T) / math.sqrt(d_idx)
        logp = torch.log_softmax(Si.masked_fill(~mask[r], float("-inf")), dim=-1)
        term = torch.where(mask[r], teacher * (torch.log(teacher.clamp_min(1e-300)) - logp),
                           torch.zeros((), dtype=torch.float64))
        loss = loss + (torch.from_numpy(g[r]) * term.sum(dim=-1)).sum()
    loss.backward()
    return Qi.grad.numpy(), Ki.grad.numpy()


@pytest.mark.parametrize("variant,seed", [("gauss", 21), ("int", 22)])
def test_kl_grad_matches_autograd(variant, seed):
    cfg = small_cfg(N=100, H_q=8, H_kv=2, d_h=16, d_idx=8, k=3)
    x = bits(gen.prefill_inputs(cfg, seed=seed, variant=variant))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 100, 3, block_size=B)
    g = np.random.default_rng(seed).uniform(0.5, 2.0, (2, 100))
    out = oracle.kl_loss_grad(x["q"], x["k"], x["q_idx"], x["k_idx"], I, g, block_size=B)
    dq_ref, dk_ref = autograd_kl_grad(x, I, g, B)
    np.testing.assert_allclose(out["dq_idx"], dq_ref, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(out["dk_idx"], dk_ref, rtol=1e-9, atol=1e-12)
    # by-products: the student's LSE over T and the teacher's mass (1 up to rounding)
    assert np.abs(out["psum"] - 1).max() < 1e-12
    Qi, Ki = f64(x["q_idx"]), f64(x["k_idx"])
    from scipy.special import logsumexp
    for r, i in [(0, 0), (1, 57), (0, 99)]:
        toks = [j for b in I[r, i] if b >= 0 for j in range(b * B, min(b * B + B, i + 1))]
        assert out["lse_idx"][r, i] == pytest.approx(logsumexp(Ki[toks] @ Qi[i, r] / math.sqrt(8)),
                                                     abs=1e-12)


def test_kl_grad_invariants():
    """sum_j dK_idx[j].K_idx[j] = sum_{i,r} dQ_idx[i,r].Q_idx[i,r] (both are sum g dS S^idx), and
    the gradient vanishes when the student's scores equal the teacher's."""
    cfg = small_cfg(N=120, H_q=8, H_kv=2, d_h=16, d_idx=8, k=4)
    x = bits(gen.prefill_inputs(cfg, seed=23))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 120, 4, block_size=B)
    g = np.random.default_rng(5).uniform(0.5, 2.0, (2, 120))
    out = oracle.kl_loss_grad(x["q"], x["k"], x["q_idx"], x["k_idx"], I, g, block_size=B)
    lhs = (out["dk_idx"] * f64(x["k_idx"])).sum()
    rhs = (out["dq_idx"] * f64(x["q_idx"])).sum()
    assert lhs == pytest.approx(rhs, rel=1e-10, abs=1e-12) and abs(lhs) > 1e-3
    # student == teacher
    cfg = small_cfg(N=130, H_q=1, H_kv=1, d_h=16, d_idx=16, k=3)
    y = bits(gen.prefill_inputs(cfg, seed=24))
    y["q_idx"] = np.ascontiguousarray(y["q"])
    y["k_idx"] = np.ascontiguousarray(y["k"][:, 0])
    _, M32 = oracle.block_scores(y["q_idx"], y["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 130, 3, block_size=B)
    out = oracle.kl_loss_grad(y["q"], y["k"], y["q_idx"], y["k_idx"], I, np.ones((1, 130)),
                              block_size=B)
    assert np.abs(out["dq_idx"]).max() < 1e-12 and np.abs(out["dk_idx"]).max() < 1e-12


# --------------------------------------------------------- main-branch gradient --

def autograd_attn_grad(x, dO, mask_fn):
    """torch.autograd in fp64 through attention whose score mask mask_fn(r) gives -> (dQ, dK, dV)."""
    Q = torch.from_numpy(f64(x["q"])).requires_grad_(True)
    K = torch.from_numpy(f64(x["k"])).requires_grad_(True)
    V = torch.from_numpy(f64(x["v"])).requires_grad_(True)
    N, H_q, d = Q.shape
    H_kv = K.shape[1]
    G = H_q // H_kv
    out = []
    for h in range(H_q):
        r = h // G
        S = (Q[:, h] @ K[:, r].T) / math.sqrt(d)
        P = torch.softmax(S.masked_fill(~mask_fn(r), float("-inf")), dim=-1)
        out.append(P @ V[:, r])
    O = torch.stack(out, dim=1)
    (O * torch.from_numpy(f64(dO))).sum().backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


@pytest.mark.parametrize("variant,seed", [("gauss", 31), ("int", 32)])
def test_attn_grad_matches_autograd(variant, seed):
    cfg = small_cfg(N=96, H_q=8, H_kv=2, d_h=16, d_idx=8, k=3)
    x = bits(gen.prefill_inputs(cfg, seed=seed, variant=variant))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 96, 3, block_size=B)
    dO = gen.to_bits(torch.randn(96, 8, 16, generator=torch.Generator().manual_seed(seed)).to(
        torch.bfloat16))
    out = oracle.sparse_attn_grad(x["q"], x["k"], x["v"], dO, I, block_size=B)
    mask = torch.from_numpy(np.array(selected_token_mask(I, 96, B)))
    dq, dk, dv = autograd_attn_grad(x, dO, lambda r: mask[r])
    np.testing.assert_allclose(out["dq"], dq, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(out["dk"], dk, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(out["dv"], dv, rtol=1e-9, atol=1e-12)


def test_attn_grad_full_k_equals_sdpa_autograd():
    """k >= number of blocks: plain causal GQA attention, so the gradient equals torch.autograd
    through scaled_dot_product_attention(is_causal=True) in fp64 (a library routine)."""
    cfg = small_cfg(N=64, H_q=8, H_kv=2, d_h=16, k=8)
    x = bits(gen.prefill_inputs(cfg, seed=33))
    B = 8
    _, M32 = oracle.block_scores(x["q_idx"], x["k_idx"], block_size=B)
    I = oracle.select_blocks(M32, 64, 8, block_size=B)
    dO = gen.to_bits(torch.randn(64, 8, 16, generator=torch.Generator().manual_seed(4)).to(
        torch.bfloat16))
    out = oracle.sparse_attn_grad(x["q"], x["k"], x["v"], dO, I, block_size=B)
    Q = torch.from_numpy(f64(x["q"])).permute(1, 0, 2)[None].requires_grad_(True)
    K = torch.from_numpy(f64(x["k"])).permute(1, 0, 2)[None].requires_grad_(True)
    V = torch.from_numpy(f64(x["v"])).permute(1, 0, 2)[None].requires_grad_(True)
    O = torch.nn.functional.scaled_dot_product_attention(
        Q, K.repeat_interleave(4, dim=1), V.repeat_interleave(4, dim=1), is_causal=True)
    (O * torch.from_numpy(f64(dO)).permute(1, 0, 2)[None]).sum().backward()
    np.testing.assert_allclose(out["dq"], Q.grad[0].permute(1, 0, 2).numpy(), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(out["dk"], K.grad[0].permute(1, 0, 2).numpy(), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(out["dv"], V.grad[0].permute(1, 0, 2).numpy(), rtol=1e-9, atol=1e-12)
