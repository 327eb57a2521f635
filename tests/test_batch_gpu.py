"""fos_quantize_batch against the oracle: every job of a batch must equal the
oracle's quantization of that matrix bit for bit (codes, scale bytes, tensor
scale, choices), whatever the shapes of its neighbours.  Both forms: the
chained row form, and the transposed / 2D form (one amax launch per group of
up to 32 jobs, then one quantize launch per job)."""
import numpy as np
import pytest

import workloads
from fos_testutil import assert_same, mixed_bits, oracle_quantize, to_device_bf16, QOut

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fos():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300 as fos

    return fos


def run_batch(fos, bits_list, lds=None, **opts):
    import torch

    xs = [to_device_bf16(b, None if lds is None else lds[i]) for i, b in enumerate(bits_list)]
    bq = fos.BatchQuantizer([b.shape for b in bits_list], with_choice=True, **opts)
    outs = bq(xs)
    torch.cuda.synchronize()
    res = []
    for o in outs:
        res.append(QOut(codes=o.codes[:, : o.cols // 2].cpu().numpy(),
                        sf=o.sf.cpu().numpy()[: fos.fos_sf_bytes(o.rows, o.cols, o.sf_layout)],
                        s_t=np.float32(o.tensor_scale.item()), choice=o.choice.cpu().numpy()))
    return res


SHAPES = [(64, 256), (300, 1040), (1, 16), (129, 512), (1024, 4096), (3, 48)]


@pytest.mark.parametrize("opts", [dict(), dict(scale_rule=1), dict(rounding=1, sr_seed=123),
                                  dict(hadamard=True, hadamard_seed=7), dict(sf_layout=1)])
def test_batch_matches_oracle(fos, opts):
    bits = [mixed_bits(r, c, seed=41 + i) for i, (r, c) in enumerate(SHAPES)]
    got = run_batch(fos, bits, **opts)
    oopts = dict(opts)
    for i, b in enumerate(bits):
        assert_same(got[i], oracle_quantize(b, **oopts), f"job {i} {b.shape} {opts}")


def test_batch_quantizer_reused_on_new_inputs(fos):
    """One BatchQuantizer called on the same inputs twice, then on other
    tensors of the same shapes (other addresses, one of them inside wider
    rows), then on the first ones again: every call must quantize the tensors
    it is given."""
    import torch

    shapes = [(64, 256), (300, 1040)]
    first = [mixed_bits(r, c, seed=51 + i) for i, (r, c) in enumerate(shapes)]
    second = [mixed_bits(r, c, seed=61 + i) for i, (r, c) in enumerate(shapes)]
    xa = [to_device_bf16(b) for b in first]
    xb = [to_device_bf16(second[0]), to_device_bf16(second[1], 1048)]
    bq = fos.BatchQuantizer(shapes, with_choice=True)

    def got():
        torch.cuda.synchronize()
        return [QOut(codes=o.codes[:, : o.cols // 2].cpu().numpy(),
                     sf=o.sf.cpu().numpy()[: fos.fos_sf_bytes(o.rows, o.cols, o.sf_layout)],
                     s_t=np.float32(o.tensor_scale.item()), choice=o.choice.cpu().numpy()) for o in bq.outs]

    for xs, bits in ((xa, first), (xa, first), (xb, second), (xa, first)):
        bq(xs)
        for i, (g, b) in enumerate(zip(got(), bits)):
            assert_same(g, oracle_quantize(b), f"job {i}")


def test_batch_padded_rows_and_weight_like_jobs(fos):
    bits = [workloads.student_t(512, 4096, seed=81), mixed_bits(256, 1024, seed=82),
            workloads.student_t(1024, 1536, seed=83)]
    got = run_batch(fos, bits, lds=[4104, 1040, 1536])
    for i, b in enumerate(bits):
        assert_same(got[i], oracle_quantize(b), f"job {i}")


def test_batch_with_empty_job_and_single_job(fos):
    bits = [mixed_bits(128, 512, seed=91), np.zeros((0, 64), np.uint16), mixed_bits(64, 64, seed=92)]
    got = run_batch(fos, bits)
    assert_same(got[0], oracle_quantize(bits[0]), "job 0")
    assert_same(got[2], oracle_quantize(bits[2]), "job 2")
    one = run_batch(fos, [bits[0]])
    assert_same(one[0], oracle_quantize(bits[0]), "single job")


# rows % 16 == 0 (transposed and 2D): 16-row groups; output rows of 16, 80,
# 1040, 4096 (transposed); tiles per 2D row band 1, 5, 65, 256
SHAPES_16 = [(64, 256), (304, 1040), (16, 16), (48, 80), (128, 4096), (32, 96)]


@pytest.mark.parametrize("opts", [dict(transpose=True), dict(transpose=True, scale_rule=2),
                                  dict(transpose=True, rounding=1, sr_seed=5, hadamard=True, hadamard_seed=9),
                                  dict(transpose=True, hadamard=True, hadamard_seed=4, sf_layout=1),
                                  dict(block_2d=True), dict(block_2d=True, rounding=1, sr_seed=3),
                                  dict(block_2d=True, hadamard=True, hadamard_seed=2),
                                  dict(block_2d=True, transpose=True, rounding=1, sr_seed=8, hadamard=True,
                                       hadamard_seed=6)])
def test_layout_batch_matches_oracle(fos, opts):
    bits = [mixed_bits(r, c, seed=141 + i) for i, (r, c) in enumerate(SHAPES_16)]
    got = run_batch(fos, bits, **opts)
    for i, b in enumerate(bits):
        assert_same(got[i], oracle_quantize(b, **opts), f"job {i} {b.shape} {opts}")


def test_layout_batch_padded_rows_and_empty_job(fos):
    """Transposed jobs read from wider rows, with an empty job between them."""
    bits = [workloads.student_t(256, 1024, seed=151), np.zeros((0, 64), np.uint16),
            mixed_bits(160, 528, seed=152)]
    opts = dict(transpose=True, hadamard=True, hadamard_seed=11)
    got = run_batch(fos, bits, lds=[1032, 64, 544], **opts)
    assert_same(got[0], oracle_quantize(bits[0], **opts), "job 0")
    assert_same(got[2], oracle_quantize(bits[2], **opts), "job 2")


def test_layout_batch_more_jobs_than_one_amax_launch(fos):
    """34 jobs: two groups (32 and 2) of one amax launch each."""
    bits = [mixed_bits(16 * (1 + i % 3), 16 * (2 + i % 5), seed=161 + i) for i in range(34)]
    opts = dict(block_2d=True, transpose=True)
    got = run_batch(fos, bits, **opts)
    for i, b in enumerate(bits):
        assert_same(got[i], oracle_quantize(b, **opts), f"job {i} {b.shape}")


def test_batch_rejects_unsupported_and_invalid(fos):
    import ctypes

    import torch

    x = to_device_bf16(mixed_bits(32, 64, seed=1))
    amax = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(fos.FosError):
        fos.BatchQuantizer([x.shape], tensor_amax=amax)([x])
    # a transposed job needs whole 16-row groups: refused before any launch
    y = to_device_bf16(mixed_bits(24, 64, seed=2))
    out = torch.empty(64 * 16, dtype=torch.uint8, device="cuda")
    ts = torch.empty(1, dtype=torch.float32, device="cuda")
    job = fos.fos_quant_job(y.data_ptr(), 24, 64, 64, out.data_ptr(), 16, out.data_ptr(), ts.data_ptr(), None)
    ws = torch.empty(fos.fos_quantize_batch_workspace_size(1), dtype=torch.uint8, device="cuda")
    st = fos.fos_quantize_batch((fos.fos_quant_job * 1)(job), fos.options(transpose=True), ws.data_ptr(),
                                ws.numel(), 0)
    assert st == fos.FOS_ERR_INVALID_ARG
    assert ctypes.sizeof(fos.fos_quant_job) > 0
    torch.cuda.synchronize()
