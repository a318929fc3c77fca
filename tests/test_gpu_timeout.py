"""The bounded-wait path on the GPU, driven without any fault: the index-branch kernel's pipeline
waits get a limit of 0 ns, so a wait that is not already satisfied gives up at once.  The kernel
must then stop, drain its copies and MMAs in flight, free its tensor memory and report
MSA_ERR_TIMEOUT through msa_device_status(); and the process must stay usable: the next call,
with the limit back at its default, gives the oracle's block scores."""
import numpy as np
import pytest
import torch

import gen
import oracle

pytestmark = pytest.mark.gpu

msa = pytest.importorskip("block_sparse_gqa_scores_gb300")

DEFAULT_NS = 2_000_000_000


def test_pipeline_wait_limit_reports_timeout_and_recovers():
    cfg = gen.CONFIGS["tiny"]
    x = gen.prefill_inputs(cfg, seed=0, device="cuda", variant="int")
    torch.cuda.synchronize()
    msa.msa_device_status()                                # start from a clear status word
    try:
        msa.msa_set_wait_limit_ns(0)
        msa.msa_index_block_scores(x["q_idx"], x["k_idx"])
        torch.cuda.synchronize()
        with pytest.raises(msa.MSAError) as e:
            msa.msa_device_status()
        assert e.value.code == 5                           # MSA_ERR_TIMEOUT
    finally:
        msa.msa_set_wait_limit_ns(DEFAULT_NS)
    # the status word was read and cleared; a normal call now runs to completion and is exact
    M = msa.msa_index_block_scores(x["q_idx"], x["k_idx"])
    torch.cuda.synchronize()
    msa.msa_device_status()
    b = {n: gen.to_bits(x[n]) for n in ("q_idx", "k_idx")}
    _, ref = oracle.block_scores(b["q_idx"], b["k_idx"])
    M = M.cpu().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(M), np.isneginf(ref))
    ulp = np.abs(M[fin].view(np.int32).astype(np.int64) - ref[fin].view(np.int32))
    assert ulp.max() <= 1                                  # d_idx = 32: scale rounded once
