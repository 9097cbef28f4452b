"""The failure path of the library's bounded in-kernel waits, exercised
without a GPU fault or a hang.

Every kernel here waits on TMA loads and tensor-core commits through one
bounded mbarrier wait; one that gives up sets a bit in an error word and
returns.  la_selftest_timeout launches one CTA that waits through that same
function on a barrier nothing arrives at, with a 1 ms limit, so the wait
gives up on purpose.  The tests check that the bit reaches the caller as
LA_ERR_DEVICE_TIMEOUT (-5): from la_gemm_status for the standalone GEMMs,
and from the next la_step / la_ar_step of a handle, which then needs a new
prefill and works again after it."""
import numpy as np
import pytest

import synth
from helpers import ensure_built

pytestmark = pytest.mark.gpu
TIMEOUT, STATE = -5, -6


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    import exact_decoding_gb300 as e
    return e


def _gemm_inputs(rows, out, k, seed):
    import torch
    x = torch.from_numpy(synth.normal((rows, k), seed, 1, 1.0, "bf16").view(np.int16)).cuda()
    w = torch.from_numpy(synth.normal((out, k), seed, 2, 0.05, "bf16").view(np.int16)).cuda()
    return x, w


def test_standalone_gemm_status_reports_a_timeout(lib):
    import torch
    x, w = _gemm_inputs(40, 256, 512, 21)
    y0 = torch.empty((40, 256), dtype=torch.float32, device="cuda")
    lib.la_gemm_bf16(x.data_ptr(), w.data_ptr(), y0.data_ptr(), 40, 256, 512, 1, None, None)
    lib.la_gemm_status()                       # a normal call leaves no bit
    lib.la_selftest_timeout(None, 1_000_000)
    with pytest.raises(lib.LaError) as e:
        lib.la_gemm_status()
    assert e.value.code == TIMEOUT
    assert "la_gemm_bf16" in str(e.value)
    lib.la_gemm_status()                       # read and cleared: clean again
    y1 = torch.empty_like(y0)
    lib.la_gemm_bf16(x.data_ptr(), w.data_ptr(), y1.data_ptr(), 40, 256, 512, 1, None, None)
    lib.la_gemm_status()
    assert torch.equal(y0, y1)                 # the context stayed usable


def test_noalloc_gemm_status_reports_a_timeout(lib):
    import torch
    x, w = _gemm_inputs(40, 256, 512, 22)
    y = torch.empty((40, 256), dtype=torch.float32, device="cuda")
    lib.la_gemm_bf16_noalloc(x.data_ptr(), w.data_ptr(), y.data_ptr(), 40, 256, 512, 2, None)
    lib.la_gemm_status()
    lib.la_selftest_timeout(None, 1_000_000)   # sets both standalone words
    with pytest.raises(lib.LaError) as e:
        lib.la_gemm_status()
    assert e.value.code == TIMEOUT
    assert "0x20 la_gemm_bf16_noalloc" in str(e.value)
    lib.la_gemm_status()


def test_selftest_rejects_a_bad_limit(lib):
    for bad in (0, 999, 3_000_000_000):
        with pytest.raises(lib.LaError) as e:
            lib.la_selftest_timeout(None, bad)
        assert e.value.code == -1


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_step_reports_a_timeout_and_recovers_after_prefill(lib, dtype):
    dims = synth.ModelDims(2, 256, 4, 4, 64, 688, 1024, dtype=dtype)
    w = synth.model_weights(dims, 31)
    p = synth.uniform_tokens(40, dims.vocab, 32)
    dec = lib.Decoder(w, 4, 5, 3, 256)
    dec.prefill(p)
    ref = [dec.step() for _ in range(3)]       # bf16: the later steps replay the captured graph
    lib.la_selftest_timeout(dec.h, 1_000_000)
    with pytest.raises(lib.LaError) as e:
        dec.step()
    assert e.value.code == TIMEOUT
    with pytest.raises(lib.LaError) as e:
        dec.step()
    assert e.value.code == STATE               # the step's results were void: prefill again
    dec.prefill(p)
    assert [dec.step() for _ in range(3)] == ref
    lib.la_selftest_timeout(dec.h, 1_000_000)
    with pytest.raises(lib.LaError) as e:
        dec.ar_step()
    assert e.value.code == TIMEOUT
    dec.close()
