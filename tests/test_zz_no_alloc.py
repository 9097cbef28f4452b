"""la_gemm_bf16_noalloc: the projection GEMM for callers that cannot allocate
device memory at call time (a plugin whose host framework owns every device
allocation, or a loop that must not call cudaMalloc), so they cannot hand
la_gemm_bf16 a split-K workspace.  It keeps the partial sums in a fixed
device array inside the library.  Its output must match la_gemm_bf16 (with a
caller workspace) on consecutive calls that reuse that array.

This file is collected last so that a run stopping at its first failure has
already run every other test."""
import numpy as np
import pytest

import synth
from helpers import ensure_built


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    import exact_decoding_gb300 as e
    return e


def _inputs(rows, out, k, seed):
    x = synth.normal((rows, k), seed, 1, 1.0, "bf16")
    w = synth.normal((out, k), seed, 2, 0.05, "bf16")
    return x, w


@pytest.mark.gpu
def test_noalloc_matches_workspace_gemm_on_consecutive_calls(lib):
    import torch
    cases = [(121, 1024, 4096, 3), (40, 600, 1024, 4), (121, 1024, 4096, 3), (17, 300, 200, 1)]
    for i, (rows, out, k, splits) in enumerate(cases):
        x, w = _inputs(rows, out, k, seed=10 + i)
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        wd = torch.from_numpy(w.view(np.int16)).cuda()
        ref = torch.empty((rows, out), dtype=torch.float32, device="cuda")
        ws = torch.empty(splits * rows * out, dtype=torch.float32, device="cuda")
        lib.la_gemm_bf16(xd.data_ptr(), wd.data_ptr(), ref.data_ptr(), rows, out, k, splits, ws.data_ptr(), None)
        got = torch.full((rows, out), float("nan"), dtype=torch.float32, device="cuda")
        lib.la_gemm_bf16_noalloc(xd.data_ptr(), wd.data_ptr(), got.data_ptr(), rows, out, k, splits, None)
        torch.cuda.synchronize()
        lib.la_gemm_status()
        # Same kernel, same split boundaries, same fixed-order reduction: the
        # two entry points must agree bit for bit (a stale plane left in the
        # shared array by the previous call would show here).
        assert torch.isfinite(got).all(), f"call {i}"
        assert torch.equal(got, ref), f"call {i}: max diff {(got - ref).abs().max().item()}"


@pytest.mark.gpu
def test_noalloc_at_exactly_its_capacity(lib):
    """splits * rows * out == LA_NOALLOC_SCRATCH_FLOATS: the largest accepted
    size fills the whole array and still matches the workspace GEMM."""
    import torch
    from exact_decoding_gb300.la import NOALLOC_SCRATCH_FLOATS
    rows, out, k, splits = 128, 8192, 1024, 4
    assert splits * rows * out == NOALLOC_SCRATCH_FLOATS
    x, w = _inputs(rows, out, k, seed=20)
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    wd = torch.from_numpy(w.view(np.int16)).cuda()
    ref = torch.empty((rows, out), dtype=torch.float32, device="cuda")
    ws = torch.empty(splits * rows * out, dtype=torch.float32, device="cuda")
    lib.la_gemm_bf16(xd.data_ptr(), wd.data_ptr(), ref.data_ptr(), rows, out, k, splits, ws.data_ptr(), None)
    for _ in range(2):
        got = torch.full((rows, out), float("nan"), dtype=torch.float32, device="cuda")
        lib.la_gemm_bf16_noalloc(xd.data_ptr(), wd.data_ptr(), got.data_ptr(), rows, out, k, splits, None)
        lib.la_gemm_status()
        assert torch.equal(got, ref)
    with pytest.raises(lib.LaError) as e:      # one more row of partials is one too many
        lib.la_gemm_bf16_noalloc(xd.data_ptr(), wd.data_ptr(), got.data_ptr(), rows, out + 1, k, splits, None)
    assert e.value.code == -3


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    from exact_decoding_gb300.la import NOALLOC_SCRATCH_FLOATS
    rows, out, splits = 256, 8192, 4
    assert splits * rows * out > NOALLOC_SCRATCH_FLOATS
    with pytest.raises(lib.LaError) as e:
        # pointers are never dereferenced: the size check comes first
        lib.la_gemm_bf16_noalloc(16, 16, 16, rows, out, 4096, splits, None)
    assert e.value.code == -3
    assert "LA_NOALLOC_SCRATCH_FLOATS" in str(e.value)
