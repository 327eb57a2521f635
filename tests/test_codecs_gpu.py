"""The device conversions and Philox stream against the oracle's codecs.

These pin the hardware E2M1/E4M3 conversions (rounding, ties, saturation, the
sign of zero) and the device Philox to the definitions the oracle follows."""
import numpy as np
import pytest

from conftest import read_golden

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaptive_quantization_fos_b300 as fos

    return fos, torch


def _enc(dev, fn, x):
    fos, torch = dev
    xt = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    out = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    st = getattr(fos, fn)(xt.data_ptr(), x.size, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _dense_floats(lo_exp: int, hi_exp: int, step: int) -> np.ndarray:
    """Every `step`-th float32 bit pattern between 2^lo_exp and 2^hi_exp, both signs."""
    lo = np.float32(2.0 ** lo_exp).view(np.uint32)
    hi = np.float32(2.0 ** hi_exp).view(np.uint32)
    u = np.arange(lo, hi, step, dtype=np.uint32).view(np.float32)
    return np.concatenate([u, -u])


def test_e2m1_encode_matches_oracle(dev, orc):
    x = np.concatenate([
        _dense_floats(-4, 4, 97),
        np.array([float(r[0]) for r in read_golden("e2m1_rne_cases.txt")], np.float32),
        np.array([0.0, -0.0, 1e-45, -1e-45, 1e-38, -1e-38, 3e38, -3e38, np.inf, -np.inf], np.float32),
    ]).astype(np.float32)
    # every tie point and its neighbours
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    x = np.concatenate([x, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 10)]).astype(np.float32)
    got = _enc(dev, "fos_e2m1_encode", x)
    want = orc.e2m1_rne(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(x[i]), int(got[i]), int(want[i])) for i in bad[:10]]


def test_e4m3_encode_matches_oracle(dev, orc):
    finite = orc.e4m3_decode(np.arange(0x7F)).astype(np.float64)
    mids = ((finite[:-1] + finite[1:]) / 2).astype(np.float32)
    x = np.concatenate([
        _dense_floats(-12, 9, 211), mids, np.nextafter(mids, 0), np.nextafter(mids, 1e3),
        np.array([0.0, 448.0, 449.0, 464.0, 480.0, 1e30, np.inf, 1e-45], np.float32),
    ]).astype(np.float32)
    x = x[x >= 0]  # the quantizer only converts non-negative scale candidates
    got = _enc(dev, "fos_e4m3_encode", x)
    want = orc.e4m3_rne_satfinite(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(want[i])) for i in bad[:10]]


def test_philox_matches_known_answers_and_oracle(dev, orc):
    fos, torch = dev
    rows = read_golden("philox4x32_10_kat.txt")
    for row in rows:
        w = [int(v, 16) for v in row]
        ctr = torch.tensor(np.array(w[0:4], np.uint32).view(np.int32), device="cuda")
        out = torch.empty(4, dtype=torch.int32, device="cuda")
        key = w[4] | (w[5] << 32)
        assert fos.fos_philox4x32_10(ctr.data_ptr(), 1, key, out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        assert out.cpu().numpy().view(np.uint32).tolist() == w[6:10]
    rng = np.random.default_rng(3)
    ctrs = rng.integers(0, 2**32, (1000, 4), dtype=np.uint64).astype(np.uint32)
    key = 0xDEADBEEF12345678
    ct = torch.from_numpy(ctrs.view(np.int32)).cuda()
    out = torch.empty((1000, 4), dtype=torch.int32, device="cuda")
    assert fos.fos_philox4x32_10(ct.data_ptr(), 1000, key, out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint32)
    for i in range(0, 1000, 37):
        assert got[i].tolist() == orc.philox4x32_10(ctrs[i], [key & 0xFFFFFFFF, key >> 32]).tolist()
