"""Helpers shared by the parity tests: run the CUDA path and the oracle on the
same seeded bf16 bits and compare their outputs in a common format."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class QOut:
    codes: np.ndarray  # uint8 [R, C/2] (only the meaningful bytes of each row)
    sf: np.ndarray  # uint8 flat scale buffer (including pad bytes)
    s_t: np.float32
    choice: np.ndarray | None  # uint8 [R, C/16], 1 = kept the 4 candidate


def to_device_bf16(bits: np.ndarray, ld: int | None = None):
    """uint16 bf16 bits [rows, cols] -> CUDA bf16 tensor, optionally inside wider rows."""
    import torch

    b = np.ascontiguousarray(bits, dtype=np.uint16)
    rows, cols = b.shape
    t = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
    if ld is not None and ld > cols:
        wide = torch.full((rows, ld), float("nan"), dtype=torch.bfloat16)
        wide[:, :cols] = t
        return wide.cuda()[:, :cols]
    return t.cuda()


def gpu_quantize(bits: np.ndarray, ld: int | None = None, with_choice=True, **opts) -> QOut:
    import torch

    import adaptive_quantization_fos_b300 as fos

    x = to_device_bf16(bits, ld)
    q = fos.quantize(x, with_choice=with_choice, **opts)
    torch.cuda.synchronize()
    C = q.cols
    return QOut(
        codes=q.codes[:, : C // 2].cpu().numpy(),
        sf=q.sf.cpu().numpy()[: fos.fos_sf_bytes(q.rows, q.cols, q.sf_layout)],
        s_t=np.float32(q.tensor_scale.item()),
        choice=q.choice.cpu().numpy() if with_choice else None,
    )


def choice_bits_to_bytes(bits: np.ndarray, nb: int) -> np.ndarray:
    R = bits.shape[0]
    return ((bits[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(R, -1)[:, :nb].astype(np.uint8)


def oracle_quantize(bits: np.ndarray, **opts) -> QOut:
    import oracle

    kw = dict(opts)
    layout = kw.pop("sf_layout", oracle.SF_SWIZZLED)
    r = oracle.quantize(bits, sf_layout=layout, **kw)
    C = r.cols
    return QOut(codes=np.ascontiguousarray(r.codes[:, : C // 2]), sf=r.sf, s_t=np.float32(r.tensor_scale),
                choice=choice_bits_to_bytes(r.choice, C // 16))


def assert_same(g: QOut, o: QOut, what: str = "") -> None:
    assert g.s_t.view(np.uint32) == o.s_t.view(np.uint32), f"{what}: s_t {g.s_t!r} vs oracle {o.s_t!r}"
    assert g.sf.shape == o.sf.shape, what
    bad_sf = np.nonzero(g.sf != o.sf)[0]
    assert bad_sf.size == 0, f"{what}: {bad_sf.size} scale bytes differ, first at {bad_sf[:8]}"
    assert g.codes.shape == o.codes.shape, what
    bad = np.argwhere(g.codes != o.codes)
    assert bad.size == 0, f"{what}: {len(bad)} code bytes differ, first {bad[:4].tolist()}"
    if g.choice is not None and o.choice is not None:
        assert np.array_equal(g.choice, o.choice), f"{what}: choice differs"


def mixed_bits(rows: int, cols: int, seed: int) -> np.ndarray:
    """bf16 bits with a mix of distributions, zero blocks, -0, outliers and tiny values."""
    import workloads

    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    q = max(rows // 5, 1)
    x[:q] = rng.standard_t(3, (q, cols)) * 0.02
    x[q: 2 * q] = rng.uniform(-1, 1, (min(q, rows - q), cols)) if rows > q else x[q: 2 * q]
    x[2 * q:, ::37] *= 40.0
    flat = x.reshape(-1)
    n = flat.size
    for k in range(0, n - 16, 997):
        flat[k: k + 16] = 0.0  # scattered all-zero blocks (not all aligned)
    flat[rng.integers(0, n, max(n // 200, 1))] = -0.0
    flat[rng.integers(0, n, max(n // 300, 1))] *= 1e-30  # tiny magnitudes
    return workloads.bf16_bits(x)


def e4m3_tie_blocks():
    """bf16 rows whose tensor amax is 1.1484375 (s_t = 7/16384 exactly) and
    whose block maxima a_b make a_b / (M s_t) land exactly on the midpoint of
    two neighbouring E4M3 values, for M = 4 and M = 6: the cases where a
    quotient must round to the even neighbour."""
    from fractions import Fraction

    import oracle
    import workloads

    finite = [Fraction(float(v)) for v in oracle.e4m3_decode(np.arange(0x7F))]
    s_t = Fraction(7, 16384)
    amax = Fraction(1.1484375)
    ties = []  # (a_b, M, the even neighbour's byte)
    for M in (4, 6):
        for k in range(1, len(finite) - 1):
            mid = (finite[k] + finite[k + 1]) / 2
            a = mid * M * s_t
            if a > amax or a <= 0:
                continue
            f = np.float32(float(a))
            if Fraction(float(f)) != a or (f.view(np.uint32) & 0xFFFF):
                continue  # not a bf16 value
            ties.append((a, M, k if k % 2 == 0 else k + 1))
    rows = []
    for a, _, _ in ties:
        row = np.zeros(64, np.float32)
        row[0] = 1.1484375  # the tensor amax (its own block)
        row[16] = float(a)  # a block whose maximum is the tie
        row[17:32] = float(a) * np.linspace(-0.9, 0.9, 15)
        rows.append(row)
    return workloads.bf16_bits(np.stack(rows)), ties
