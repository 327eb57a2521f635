"""fos_quantize_batch against the oracle: every job of a chained batch must
equal the oracle's quantization of that matrix bit for bit (codes, scale
bytes, tensor scale, choices), whatever the shapes of its neighbours."""
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


def test_batch_rejects_unsupported_options(fos):
    import torch

    x = to_device_bf16(mixed_bits(32, 64, seed=1))
    for bad in (dict(transpose=True), dict(block_2d=True)):
        with pytest.raises(fos.FosError):
            fos.BatchQuantizer([x.shape], **bad)([x])
    torch.cuda.synchronize()
