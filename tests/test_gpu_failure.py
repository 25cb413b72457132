"""Failure detection without a GPU fault: the library's bounded waits give
up, report MSA_DEV_TIMEOUT and leave the context usable ("Attention sinks
for ROCm AITER sparse MLA" (vLLM PR 54404), "Key source snippets": a missing
result must raise, not hang).

msa_check_bounded_wait runs the same bounded wait the streaming kernels use
on an mbarrier armed for bytes that nothing delivers (a flag nothing sets),
with a 1 ms limit, optionally holding tensor memory or with a real bulk copy
in flight, exactly the states the kernels' expiry paths clean up."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.helpers import assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import block_sparse_paged_02_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_bounded_wait_gives_up_and_the_context_stays_usable(msa, orc, flags):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    src = torch.arange(4, dtype=torch.int32, device="cuda")  # 16 bytes for the copy
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    msa.msa_check_bounded_wait(status, 1000, flags,
                               src if flags & msa.MSA_CHECK_WAIT_COPY else None)
    end.record()
    torch.cuda.synchronize()
    # the wait ran out (and nothing else did: a drain that gave up would add a bit)
    assert int(status.item()) == msa.MSA_DEV_TIMEOUT
    ms = start.elapsed_time(end)
    assert 0.9 <= ms < 1000.0, ms
    # the context still answers: a decode on the same stream matches the oracle
    w = W.custom(90 + flags, q_lens=[1, 3], seq_lens=[5000, 900], hq=16, di=128, topk=8,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_SCALAR, with_sink=True)
    c = msa.DeviceCase(w)
    c.decode()
    got = c.fetch()
    ref = orc.decode(w)
    assert got["status"] == 0
    for key in ("topk_idx", "tbl", "sparse_len"):
        assert np.array_equal(got[key], ref[key])
    assert_attn_close(got["out"], got["lse"], ref["out"], ref["lse"])


def test_bounded_wait_argument_errors(msa):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(msa.MsaError):
        msa.msa_check_bounded_wait(status, 0)            # limit out of range
    with pytest.raises(msa.MsaError):
        msa.msa_check_bounded_wait(status, 1000, 4)      # unknown flag
    with pytest.raises(msa.MsaError):
        msa.msa_check_bounded_wait(status, 1000, msa.MSA_CHECK_WAIT_COPY)  # copy without source
    torch.cuda.synchronize()
    assert int(status.item()) == 0                       # nothing ran
