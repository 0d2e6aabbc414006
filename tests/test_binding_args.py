"""The Python binding checks every tensor before its pointer crosses the C
ABI: a wrong dtype raises TypeError and a host tensor raises ValueError, before
any CUDA call (so these run on CPU). The size and layout checks need CUDA
tensors and are covered by the GPU tests."""

from __future__ import annotations

import pytest
import torch

import sparse_attention_top_row_gb300 as topk


@pytest.fixture(scope="module", autouse=True)
def built():
    from sparse_attention_top_row_gb300 import build as b
    b.build()
    topk.load()


def i32(n):
    return torch.zeros(n, dtype=torch.int32)


def test_seq_lens_dtype_and_device():
    ws = torch.empty(256, dtype=torch.uint8)
    with pytest.raises(TypeError, match="seq_lens must be torch.int32"):
        topk.topk_plan(torch.zeros(4, dtype=torch.int64), 16, ws)
    with pytest.raises(ValueError, match="seq_lens must be a CUDA tensor"):
        topk.topk_plan(i32(4), 16, ws)


def test_transform_argument_types():
    f32 = torch.zeros(64, dtype=torch.float32)
    with pytest.raises(TypeError, match="seq_lens must be a torch.Tensor"):
        topk.topk_transform_ragged(f32, 0, None, [1, 2], i32(2), 16, None, i32(32))
    with pytest.raises(TypeError, match="seq_lens must be torch.int32"):
        topk.topk_transform_paged(f32, 64, None, torch.zeros(2), i32(2), 1, 64, 16, None, i32(32))
    with pytest.raises(ValueError, match="CUDA tensor"):
        topk.topk_transform_paged_packed(f32, 64, None, i32(2), i32(2), 1, 64, None, None, 16, None, i32(32))
    with pytest.raises(ValueError, match="CUDA tensor"):
        topk.topk_transform_ragged_noalloc(f32, 0, None, i32(2), i32(2), 16, i32(32))


def test_required_arguments():
    with pytest.raises(ValueError, match="workspace is required"):
        topk.topk_read_device_errors(None)
    with pytest.raises(ValueError, match="seq_lens is required"):
        topk.topk_plan(None, 16, torch.empty(256, dtype=torch.uint8))
