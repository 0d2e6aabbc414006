"""The binding's size and layout checks on CUDA tensors: each bad argument
raises before its pointer crosses the C ABI, so nothing is enqueued."""

from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bad_tensors_are_rejected(cuda_lib):
    dev = "cuda"
    B, k, L = 4, 16, 256
    scores = torch.zeros((B, L), dtype=torch.float32, device=dev)
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    table = torch.zeros((B, L // 64), dtype=torch.int32, device=dev)
    offs = torch.zeros(B, dtype=torch.int32, device=dev)
    ws = cuda_lib.new_workspace(B)
    out = torch.empty((B, k), dtype=torch.int32, device=dev)

    with pytest.raises(ValueError, match="out has 60 elements"):
        cuda_lib.topk_transform_ragged(scores, L, None, lens, offs, k, ws, out.view(-1)[:60])
    with pytest.raises(ValueError, match="seq_lens must be contiguous"):
        cuda_lib.topk_plan(torch.zeros(2 * B, dtype=torch.int32, device=dev)[::2], k, ws)
    with pytest.raises(ValueError, match="scores must have a unit innermost stride"):
        cuda_lib.topk_transform_paged(scores.t(), L, None, lens, table, L // 64, 64, k, ws, out)
    with pytest.raises(ValueError, match="page_table is required"):
        cuda_lib.topk_transform_paged(scores, L, None, lens, None, L // 64, 64, k, ws, out)
    with pytest.raises(TypeError, match="scores must be torch.float32"):
        cuda_lib.topk_transform_ragged(scores.double(), L, None, lens, offs, k, ws, out)
    with pytest.raises(ValueError, match="row_to_batch has 2 elements"):
        cuda_lib.topk_transform_paged_packed(scores, L, None, lens, table, L // 64, 64, None, offs[:2], k, ws, out)
    with pytest.raises(ValueError, match="out_raw must be contiguous"):
        cuda_lib.topk_transform_ragged(scores, L, None, lens, offs, k, ws, out,
                                       torch.empty((k, B), dtype=torch.int32, device=dev).t())
    # the same arguments, well formed, run
    cuda_lib.topk_plan(lens, k, ws)
    cuda_lib.topk_transform_ragged(scores, L, None, lens, offs, k, ws, out)
    torch.cuda.synchronize()
    assert cuda_lib.topk_read_device_errors(ws) == (0, 0)
