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


def test_short_strided_buffers_are_rejected(cuda_lib):
    """scores and page_table hold rows `stride` elements apart: a buffer that
    cannot even hold the last row's first element is rejected."""
    dev = "cuda"
    B, k, L = 4, 16, 256
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    ws = cuda_lib.new_workspace(B)
    out = torch.empty((B, k), dtype=torch.int32, device=dev)
    offs = torch.zeros(B, dtype=torch.int32, device=dev)
    short = torch.zeros((B - 1) * L, dtype=torch.float32, device=dev)   # (B-1)*L + 1 needed
    with pytest.raises(ValueError, match=f"scores has {(B - 1) * L} elements, fewer than the {(B - 1) * L + 1}"):
        cuda_lib.topk_transform_ragged(short, L, None, lens, offs, k, ws, out)
    scores = torch.zeros(B * L, dtype=torch.float32, device=dev)
    table = torch.zeros(3 * (L // 64), dtype=torch.int32, device=dev)   # 3 of the 4 rows
    with pytest.raises(ValueError, match="page_table has 12 elements, fewer than the 13"):
        cuda_lib.topk_transform_paged(scores, L, None, lens, table, L // 64, 64, k, ws, out)
    # packed rows name their table rows: any non-empty table passes this check
    cuda_lib.topk_plan(lens, k, ws)
    cuda_lib.topk_transform_paged_packed(scores, L, None, lens, table, L // 64, 64, None,
                                         torch.zeros(B, dtype=torch.int32, device=dev), k, ws, out)
    torch.cuda.synchronize()


def test_tensors_on_another_device_are_rejected(cuda_lib, monkeypatch):
    """Every tensor must live on the device the call launches on (the current
    one). With one GPU, another current device is simulated: the tensors on
    cuda:0 are then on the wrong device, and so is the stream."""
    dev = "cuda"
    B, k, L = 2, 16, 256
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    ws = cuda_lib.new_workspace(B)
    out = torch.empty((B, k), dtype=torch.int32, device=dev)
    scores = torch.zeros(B * L, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)
    with pytest.raises(ValueError, match="the stream belongs to cuda:0, but cuda:1 is current"):
        cuda_lib.topk_plan(lens, k, ws, stream=stream)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda *a: _FakeStream())
    with pytest.raises(ValueError, match="seq_lens is on cuda:0, but the call runs on cuda:1"):
        cuda_lib.topk_plan(lens, k, ws)
    with pytest.raises(ValueError, match="is on cuda:0, but the call runs on cuda:1"):
        cuda_lib.topk_transform_ragged(scores, L, None, lens, lens, k, ws, out)


class _FakeStream:
    """A stream handle that claims no device (the call's device is then the
    current one alone); it is never used to launch."""

    class device:  # noqa: N801
        index = None

    cuda_stream = 0
