"""Full-size parity of the quantizer on the measured workloads, every output
byte compared with the oracle (the oracle finishes each in seconds):

- the Qwen3-8B-shaped layer weight set, quantized as one chained batch in the
  order and launch configuration the benchmark times (smallest first), and as
  one batch of transposed jobs and of 2D jobs (one amax launch, then a
  quantize launch per matrix), as the benchmark also times them;
- the 16384 x 4096 activation with the RHT, row-major and transposed;
- the 8192 x 12288 gradient with stochastic rounding, 1D and 2D, and 2D RNE.
"""
import numpy as np
import pytest

import workloads
from fos_testutil import QOut, assert_same, gpu_quantize, oracle_quantize, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fos():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300 as fos

    return fos


def test_qwen3_weight_set_as_one_batch(fos):
    import torch

    mats = workloads.qwen3_8b_weights()
    order = sorted(mats, key=lambda k: mats[k].size)
    xs = [to_device_bf16(mats[k]) for k in order]
    bq = fos.BatchQuantizer([x.shape for x in xs], with_choice=True)
    outs = bq(xs)
    torch.cuda.synchronize()
    for k, o in zip(order, outs):
        got = QOut(codes=o.codes[:, : o.cols // 2].cpu().numpy(), sf=o.sf.cpu().numpy(),
                   s_t=np.float32(o.tensor_scale.item()), choice=o.choice.cpu().numpy())
        assert_same(got, oracle_quantize(mats[k]), k)


@pytest.mark.parametrize("opts", [dict(transpose=True), dict(block_2d=True)])
def test_qwen3_weight_set_layout_batch(fos, opts):
    import torch

    mats = workloads.qwen3_8b_weights()
    order = sorted(mats, key=lambda k: mats[k].size)
    xs = [to_device_bf16(mats[k]) for k in order]
    bq = fos.BatchQuantizer([x.shape for x in xs], with_choice=True, **opts)
    outs = bq(xs)
    torch.cuda.synchronize()
    for k, o in zip(order, outs):
        got = QOut(codes=o.codes[:, : o.cols // 2].cpu().numpy(), sf=o.sf.cpu().numpy(),
                   s_t=np.float32(o.tensor_scale.item()), choice=o.choice.cpu().numpy())
        assert_same(got, oracle_quantize(mats[k], **opts), f"{k} {opts}")


@pytest.mark.parametrize("transpose", [False, True])
def test_activation_rht(fos, transpose):
    x = workloads.activations(16384, 4096, seed=3001)
    opts = dict(hadamard=True, hadamard_seed=3002, transpose=transpose)
    assert_same(gpu_quantize(x, **opts), oracle_quantize(x, **opts), f"activation transpose={transpose}")


@pytest.mark.parametrize("opts", [dict(rounding=1, sr_seed=4002), dict(rounding=1, sr_seed=4002, block_2d=True),
                                  dict(block_2d=True)])
def test_gradient(fos, opts):
    g = workloads.gradients(8192, 12288, seed=4001)
    assert_same(gpu_quantize(g, **opts), oracle_quantize(g, **opts), f"gradient {opts}")
