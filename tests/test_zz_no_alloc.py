"""fos_quantize_noalloc against fos_quantize, through the C ABI.

fos_quantize_noalloc serves callers that cannot allocate device memory, such as
plugin hosts and inference runtimes that give an operator only its inputs and
outputs and forbid cudaMalloc after start-up.  It keeps the amax pass's scratch
in a fixed array owned by the library, shared by every call.  Its outputs must
equal fos_quantize's bit for bit (the tolerance every quantizer test here
uses), on consecutive calls that reuse the array with different tensors.

This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

from fos_testutil import mixed_bits, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fos():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300 as fos

    return fos


def _noalloc(fos, x, **opts):
    """Outputs of fos_quantize_noalloc; only the outputs are allocated here."""
    import torch

    rows, cols = x.shape
    opt = fos.options(**opts)
    R, C = (cols, rows) if opts.get("transpose") else (rows, cols)
    layout = opts.get("sf_layout", fos.FOS_SF_SWIZZLED_128x4)
    codes = torch.empty((R, max(8, ((C // 2 + 15) // 16) * 16)), dtype=torch.uint8, device=x.device)
    sf = torch.empty(max(1, fos.fos_sf_bytes(R, C, layout)), dtype=torch.uint8, device=x.device)
    ts = torch.empty(1, dtype=torch.float32, device=x.device)
    choice = torch.empty((R, C // 16), dtype=torch.uint8, device=x.device)
    st = fos.fos_quantize_noalloc(x.data_ptr(), rows, cols, x.stride(0), opt, codes.data_ptr(), codes.stride(0),
                                  sf.data_ptr(), ts.data_ptr(), choice.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert st == fos.FOS_OK, fos._lib.fos_status_string(st)
    return codes, sf, ts, choice


def test_noalloc_matches_quantize_on_consecutive_calls(fos):
    import torch

    cases = [
        (mixed_bits(1024, 4096, seed=101), dict()),  # many amax partials
        (mixed_bits(304, 1040, seed=103), dict(transpose=True, hadamard=True, hadamard_seed=9)),
        (mixed_bits(64, 256, seed=104), dict(block_2d=True, rounding=fos.FOS_ROUND_STOCHASTIC, sr_seed=5)),
        (mixed_bits(1024, 4096, seed=101), dict()),  # the first case again, after the array held other data
    ]
    for bits, opts in cases:
        x = to_device_bf16(bits)
        ref = fos.quantize(x, with_choice=True, **opts)
        codes, sf, ts, choice = _noalloc(fos, x, **opts)
        torch.cuda.synchronize()
        C = ref.cols
        assert np.array_equal(codes[:, : C // 2].cpu().numpy(), ref.codes[:, : C // 2].cpu().numpy()), opts
        assert np.array_equal(sf.cpu().numpy(), ref.sf.cpu().numpy()), opts
        assert ts.cpu().numpy().view(np.uint32)[0] == ref.tensor_scale.cpu().numpy().view(np.uint32)[0], opts
        assert np.array_equal(choice.cpu().numpy(), ref.choice.cpu().numpy()), opts


def test_noalloc_rejects_bad_arguments(fos):
    st = fos.fos_quantize_noalloc(1 << 20, 32, 40, 40, fos.options(), 1 << 20, 32, 1 << 20, 1 << 20, 0, 0)
    assert st == fos.FOS_ERR_INVALID_ARG  # cols % 16 != 0: rejected before any launch
