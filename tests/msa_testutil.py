"""Helpers shared by the parity tests: device copies of generator outputs, selection
comparison with the near-tie allowance, and tolerances."""
import numpy as np
import torch

import gen

# Tolerances for bf16 inputs with fp32 accumulation (O max-abs, LSE abs).
O_TOL = 2e-2
LSE_TOL = 1e-3
# Near-tie band for index selections on Gaussian inputs: 1e-3 relative to the (k-1)-th best
# non-local block score, plus an absolute floor for thresholds near 0.  The floor is the size
# of the fp32 accumulation-order difference of a d_idx <= 64 dot product of bf16 N(0,1) inputs
# (well under 1e-6 after the 1/sqrt(d_idx) scale), so it only matters where the relative band
# would shrink below what rounding alone can move a score.
TIE_REL = 1e-3
TIE_ABS = 1e-6


def bits(x):
    return {k: gen.to_bits(v) for k, v in x.items() if k not in ("meta",) and v.dtype == torch.bfloat16}


def cuda(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def selection_mismatches(I_gpu, I_ref, M_ref, k, rows=None, block=64):
    """Rows whose GPU selection differs from the oracle's by more than near-ties.

    I_gpu, I_ref: [H_kv, n, k] (n rows, row t is query rows[t] or t); M_ref: fp32/fp64 oracle
    block scores [H_kv, n, nblk].  A difference is accepted when every block in the symmetric
    difference scores within TIE_REL (relative) of the oracle's (k-1)-th best non-local score.
    Returns (n_differing_rows, list_of_bad_rows)."""
    H_kv, n, _ = I_ref.shape
    differ, bad = 0, []
    for r in range(H_kv):
        for t in range(n):
            a, b = I_gpu[r, t], I_ref[r, t]
            if np.array_equal(a, b):
                continue
            differ += 1
            i = t if rows is None else int(rows[t])
            l = i // block
            sa = set(int(x) for x in a if x >= 0)
            sb = set(int(x) for x in b if x >= 0)
            if l not in sa or len(sa) != len(sb):
                bad.append((r, i))
                continue
            cand = np.sort(np.asarray(M_ref[r, t, :l], np.float64))[::-1]
            thr = cand[k - 2]
            tol = TIE_REL * abs(thr) + TIE_ABS
            if any(abs(float(M_ref[r, t, x]) - thr) > tol for x in sa ^ sb):
                bad.append((r, i))
    return differ, bad


def max_abs(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.abs(a - b).max()) if a.size else 0.0


def bf16_dev_to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


from gen import to_pages  # noqa: E402,F401  (layout helper shared with the bench)


def check_prefill_rows(x, k, idx, o, lse, rows, min_same=0.9, rows_dev=None):
    """Prefill parity on sampled query rows of one sequence, against the oracle:
      - the GPU's selection equals the oracle's except at near-ties (selection_mismatches);
      - O and LSE of EVERY sampled row equal the oracle's main branch evaluated on the GPU's
        own selection (O max-abs <= O_TOL, LSE <= LSE_TOL).
    x: the sequence's bf16 tensors q, k, v, q_idx, k_idx (device); idx [H_kv, N, k] int32,
    o [N, H_q, d_h] bf16 and lse [H_q, N] fp32 are the GPU's results for that sequence.
    Returns (rows whose selection differs, max O error, max LSE error)."""
    import oracle
    b = {n: gen.to_bits(x[n]) for n in ("k", "v", "k_idx")}
    rows = np.asarray(rows, np.int64)
    rows_t = torch.from_numpy(rows).to(idx.device) if rows_dev is None else rows_dev
    qr = gen.to_bits(x["q"][rows_t])
    qir = gen.to_bits(x["q_idx"][rows_t])
    ref = oracle.prefill(qr, b["k"], b["v"], qir, b["k_idx"], k, rows=rows, want_m=True,
                         compact=True)
    I_gpu = idx[:, rows_t].cpu().numpy()                       # [H_kv, n, k]
    I_ref = ref["I"].transpose(1, 0, 2)
    differ, bad = selection_mismatches(I_gpu, I_ref, ref["M32"].transpose(1, 0, 2), k, rows=rows)
    assert not bad, bad[:5]
    same = (I_gpu == I_ref).all(axis=(0, 2))                   # rows with all groups identical
    assert same.mean() >= min_same, same.mean()
    O64, _, L = oracle.sparse_attn(qr, b["k"], b["v"], I_gpu, rows=rows, compact=True)
    err_o = max_abs(o[rows_t].float().cpu().numpy(), O64)
    err_l = max_abs(lse[:, rows_t].cpu().numpy().T, L)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)
    return differ, err_o, err_l


def check_decode_seqs(d, k, o, lse, idx, exact_idx=False, seqs=None):
    """Decode parity per sequence against the oracle: the selection equals the oracle's (bit for
    bit when exact_idx, else up to near-ties) and O / LSE equal the oracle's main branch on the
    GPU's own selection.  d: packed decode inputs (device tensors + cu_seqlens); o [S,H_q,d_h],
    lse [S,H_q], idx [S,H_kv,k] are the GPU's results."""
    import oracle
    cu = d["cu_seqlens"].cpu().numpy()
    S = len(cu) - 1
    seqs = range(S) if seqs is None else seqs
    I_all = idx.cpu().numpy()
    o_all, l_all = o.float().cpu().numpy(), lse.cpu().numpy()
    worst_o = worst_l = 0.0
    for s in seqs:
        sl = slice(int(cu[s]), int(cu[s + 1]))
        L = int(cu[s + 1] - cu[s])
        kb, vb = gen.to_bits(d["k_cache"][sl]), gen.to_bits(d["v_cache"][sl])
        kib = gen.to_bits(d["k_idx_cache"][sl])
        qb, qib = gen.to_bits(d["q"][s:s + 1]), gen.to_bits(d["q_idx"][s:s + 1])
        ref = oracle.decode(qb, qib, kb, vb, kib, np.array([0, L], np.int64), k, want_m=True)
        I_gpu = I_all[s:s + 1]                                 # [1, H_kv, k]
        if exact_idx:
            assert np.array_equal(I_gpu, ref["I"]), s
        else:
            _, bad = selection_mismatches(I_gpu.transpose(1, 0, 2), ref["I"].transpose(1, 0, 2),
                                          ref["M32"].transpose(1, 0, 2), k, rows=[L - 1])
            assert not bad, (s, bad)
        O64, _, Lr = oracle.sparse_attn(qb, kb, vb, I_gpu.transpose(1, 0, 2), rows=[L - 1],
                                        compact=True)
        eo, el = max_abs(o_all[s], O64[0]), max_abs(l_all[s], Lr[0])
        assert eo <= O_TOL and el <= LSE_TOL, (s, eo, el)
        worst_o, worst_l = max(worst_o, eo), max(worst_l, el)
    return worst_o, worst_l


def unpage(d_pages, page_table, seq_lens):
    """The tokens of a paged decode cache gathered back into the packed layout (layout only):
    returns k_cache, v_cache, k_idx_cache and cu_seqlens as device tensors."""
    kp, vp, kip = d_pages
    lens = seq_lens.cpu().numpy()
    pt = page_table.cpu().numpy()
    rows = []
    for s, L in enumerate(lens):
        toks = np.arange(int(L))
        rows.append(pt[s, toks // 64].astype(np.int64) * 64 + toks % 64)
    rows = torch.from_numpy(np.concatenate(rows)).to(kp.device)
    flat = lambda t: t.reshape((-1,) + tuple(t.shape[2:]))
    cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.from_numpy(lens.astype(np.int64)), 0)
    return flat(kp)[rows], flat(vp)[rows], flat(kip)[rows], cu.to(kp.device)
