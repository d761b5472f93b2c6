"""msa_build_block_index_static (built-in scratch, no workspace) against
msa_build_block_index with a caller workspace: the same kernels on the same
inputs, so the integer outputs must agree exactly, on two calls in a row."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,d,Hq,Hkv,heads,topk", [
    (4096, 128, 8, 2, [0, 1, 5, 7], 12),
    (1000, 64, 4, 1, [2], 5),
])
def test_static_scratch_matches_workspace_path(cuda_lib, n, d, Hq, Hkv, heads, topk):
    q, k, _ = synth.random_qkv(1, Hq, Hkv, n, d, seed=n + topk, device="cuda")
    J_ws, C_ws = cuda_lib.build_block_index(q, k, heads, topk)
    assert cuda_lib.poll_device_status() == 0
    for _ in range(2):
        J, C = cuda_lib.build_block_index_static(q, k, heads, topk)
        assert cuda_lib.poll_device_status() == 0
        assert torch.equal(C, C_ws)
        assert torch.equal(J, J_ws)


def test_static_scratch_counts_each_kv_head_once(cuda_lib):
    """16 query heads reading 4 KV heads at n = 32768, d_h = 128: pooled once
    per KV head the request needs about 15.5 MiB and fits, although the
    worst-case workspace query (one KV head per listed head, about 20 MiB)
    does not."""
    q, k, _ = synth.random_qkv(1, 16, 4, 32768, 128, seed=77, device="cuda")
    heads = list(range(16))
    J_ws, C_ws = cuda_lib.build_block_index(q, k, heads, 16)
    assert cuda_lib.poll_device_status() == 0
    for _ in range(2):
        J, C = cuda_lib.build_block_index_static(q, k, heads, 16)
        assert cuda_lib.poll_device_status() == 0
        assert torch.equal(C, C_ws)
        assert torch.equal(J, J_ws)


def test_static_scratch_rejects_oversize(cuda_lib):
    """A request whose scratch would exceed MSA_STATIC_SCRATCH_BYTES is refused
    on the host with MSA_ERR_WORKSPACE_TOO_SMALL (3) and launches nothing."""
    q = torch.zeros(1, 32, 65536, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 32, 65536, 128, dtype=torch.bfloat16, device="cuda")
    before = cuda_lib.kernel_launches()
    with pytest.raises(cuda_lib.MsaError, match=r"\(3\)"):
        cuda_lib.build_block_index_static(q, k, list(range(32)), 8)
    assert cuda_lib.kernel_launches() == before
