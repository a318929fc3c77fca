"""Helpers shared by the parity tests: device copies of generator outputs, selection
comparison with the near-tie allowance, and tolerances."""
import numpy as np
import torch

import gen

# Tolerances for bf16 inputs with fp32 accumulation (O max-abs, LSE abs).
O_TOL = 2e-2
LSE_TOL = 1e-3
TIE_REL = 1e-3          # near-tie band for index selections on Gaussian inputs


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
            tol = TIE_REL * max(1.0, abs(thr))
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
