"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies runs out, the device error word reports MSA_ERR_DEVICE_TIMEOUT to
the host, the word is cleared by the poll, and the context keeps working."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import compare_rows, f32, head_qkv, scale_of

pytestmark = pytest.mark.gpu

MSA_ERR_DEVICE_TIMEOUT = 5


def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib):
    assert cuda_lib.poll_device_status() == 0
    cuda_lib.check_wait_timeout(20)
    assert cuda_lib.poll_device_status() == MSA_ERR_DEVICE_TIMEOUT
    assert cuda_lib.poll_device_status() == 0  # the poll cleared the word
    # the context still runs the library's kernels correctly
    q, k, v = synth.random_qkv(1, 2, 1, 300, 64, seed=3, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 300, device="cuda")
    cuda_lib.attn_ashape(q, k, v, [0, 1], 16, 64, o=o, lse=lse)
    assert cuda_lib.poll_device_status() == 0
    qn, kn, vn = head_qkv(q, k, v, 0, 1, 2, 1)
    ro, rl, _ = oracle.head_rows(dict(pattern=oracle.ASHAPE, sink=16, window=64), qn, kn, vn, np.arange(300),
                                 scale_of(64))
    compare_rows(f32(o[0, 1]), f32(lse[0, 1]), ro, rl, "after timeout")


def test_timeout_check_rejects_bad_limit(cuda_lib):
    with pytest.raises(cuda_lib.MsaError):
        cuda_lib.check_wait_timeout(0)


MSA_ERR_INDEX = 6


def test_bad_block_index_reports_index_error(cuda_lib):
    """Block-Sparse lists that break the index contract (an entry above its
    query block, a list out of ascending order) are caught by the kernel's own
    checks: the offending entries are skipped, the poll reports MSA_ERR_INDEX
    once, and the next call on the same context is correct."""
    n, d, topk = 1000, 128, 4
    q, k, v = synth.random_qkv(1, 2, 1, n, d, seed=21, device="cuda")
    qn, kn, vn = head_qkv(q, k, v, 0, 0, 2, 1)
    J, C = oracle.bs_index(qn, kn, 64, topk)
    bad = J.copy()
    bad[12, 0] = 40                       # block 40 lies above query block 12
    bad[10, :3] = bad[10, :3][::-1].copy()  # descending: out of order
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, n, device="cuda")
    cuda_lib.attn_block(q, k, v, [0], topk, torch.from_numpy(bad[None, None]).cuda(),
                        torch.from_numpy(C[None, None]).cuda(),
                        o=o, lse=lse)
    assert cuda_lib.poll_device_status() == MSA_ERR_INDEX
    assert cuda_lib.poll_device_status() == 0
    cuda_lib.attn_block(q, k, v, [0], topk, torch.from_numpy(J[None, None]).cuda(),
                        torch.from_numpy(C[None, None]).cuda(),
                        o=o, lse=lse)
    assert cuda_lib.poll_device_status() == 0
    cfg = dict(pattern=oracle.BLOCK, block=64, topk=topk)
    ro, rl, _ = oracle.head_rows(cfg, qn, kn, vn, np.arange(n), scale_of(d), J=J, cnt=C)
    compare_rows(f32(o[0, 0]), f32(lse[0, 0]), ro, rl, "after index error")
