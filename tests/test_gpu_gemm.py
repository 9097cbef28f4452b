"""tcgen05 GEMM through the C ABI vs the GEMM's definition (fp64 of the same
bf16 inputs)."""
import numpy as np
import pytest

import synth
from helpers import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    import exact_decoding_gb300 as e
    return e


@pytest.mark.parametrize("rows,out,k,splits", [
    (16, 128, 64, 1), (1, 128, 64, 1), (17, 300, 200, 1), (121, 1024, 4096, 1), (121, 1024, 4096, 3),
    (128, 384, 1024, 4), (200, 256, 512, 2), (41, 8192 + 64, 128, 1), (256, 128, 11008, 5),
])
def test_gemm_matches_definition(lib, rows, out, k, splits):
    import torch
    x = synth.normal((rows, k), 1, 1, 1.0, "bf16")
    w = synth.normal((out, k), 1, 2, 0.05, "bf16")
    ref = synth.bf16_to_f32(x).astype(np.float64) @ synth.bf16_to_f32(w).astype(np.float64).T
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    wd = torch.from_numpy(w.view(np.int16)).cuda()
    yd = torch.full((rows, out), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(splits * rows * out, dtype=torch.float32, device="cuda") if splits > 1 else None
    lib.la_gemm_bf16(xd.data_ptr(), wd.data_ptr(), yd.data_ptr(), rows, out, k, splits,
                     ws.data_ptr() if ws is not None else None, None)
    torch.cuda.synchronize()
    y = yd.cpu().numpy().astype(np.float64)
    scale = np.sqrt(k) * 0.05
    assert np.all(np.isfinite(y))
    np.testing.assert_allclose(y, ref, atol=2e-5 * scale * np.sqrt(k) / 8 + 1e-5, rtol=1e-5)


def test_gemm_is_deterministic(lib):
    import torch
    rows, out, k = 121, 512, 4096
    x = torch.from_numpy(synth.normal((rows, k), 3, 1, 1.0, "bf16").view(np.int16)).cuda()
    w = torch.from_numpy(synth.normal((out, k), 3, 2, 0.05, "bf16").view(np.int16)).cuda()
    ws = torch.empty(4 * rows * out, dtype=torch.float32, device="cuda")
    ys = []
    for _ in range(3):
        y = torch.empty((rows, out), dtype=torch.float32, device="cuda")
        lib.la_gemm_bf16(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, out, k, 4, ws.data_ptr(), None)
        ys.append(y)
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])
