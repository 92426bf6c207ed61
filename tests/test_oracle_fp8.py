"""Pins of the oracle's FP8 e4m3 dispatch arithmetic (CPU only).

The FP8 step ("Expert Parallelism (EP)" page, the FP8 dispatch of its next
steps) sends the dispatched activations as e4m3 values with scales.  The
format ("fn": bias 7, 3 mantissa bits, no infinities, largest finite 448) is
pinned against its closed forms and against torch's float8_e4m3fn type (a
library routine written independently of the oracle); the row quantisation
(one binary32 scale per row, amax / 448) against the same library cast of
numpy's binary32 quotients, and against the properties it must have.
"""
import numpy as np
import pytest
import torch

import oracle


def _torch_codes(v32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v32, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_decode_table_matches_library_and_closed_forms():
    tab = oracle.e4m3_table()
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    lib = lib.to(torch.float32).numpy().astype(np.float64)
    nan = np.isnan(tab)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(nan, np.isnan(lib))
    assert np.array_equal(tab[~nan], lib[~nan])
    assert tab[0x7E] == 448.0 and tab[0xFE] == -448.0            # largest finite
    assert tab[0x01] == 2.0 ** -9 and tab[0x08] == 2.0 ** -6     # smallest subnormal, normal
    assert tab[0x38] == 1.0 and tab[0x00] == 0.0
    assert np.signbit(tab[0x80]) and tab[0x80] == 0.0
    # every finite positive value is (1 + m/8) 2^(e-7) or m/8 2^-6
    pos = tab[:0x7F]
    assert np.all(np.diff(pos) > 0)                               # monotone codes


def test_encode_exact_values_midpoints_and_library():
    tab = oracle.e4m3_table()
    pos = tab[:0x7F]                                              # 0 .. 448
    # exact values encode to themselves
    for c, v in enumerate(pos):
        assert oracle.e4m3_encode(v) == c
        assert oracle.e4m3_encode(-v) == (c | 0x80)
    # midpoints go to the even code; one binary32 step either side goes to the near one
    for c in range(len(pos) - 1):
        mid = np.float32((pos[c] + pos[c + 1]) / 2)
        assert float(mid) == (pos[c] + pos[c + 1]) / 2            # exact in binary32
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even
        assert oracle.e4m3_encode(np.nextafter(mid, np.float32(0))) == c
        assert oracle.e4m3_encode(np.nextafter(mid, np.float32(1e9))) == c + 1
    # the library agrees on a wide in-range sample
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-12, 6, 20000))).astype(np.float32)
    v = v[np.abs(v) < 448]
    ours = np.array([oracle.e4m3_encode(x) for x in v], np.uint8)
    assert np.array_equal(ours, _torch_codes(v))


def test_encode_saturates_and_nan():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(460.0) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert oracle.e4m3_encode(2.0 ** -11) == 0x00                 # below half the smallest step
    assert oracle.e4m3_encode(3 * 2.0 ** -11) == 0x01             # above it


@pytest.mark.parametrize("rows,cols", [(7, 128), (33, 2048)])
def test_quantize_rows_matches_library_and_properties(rows, cols):
    rng = np.random.default_rng(rows)
    x = (rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-4, 4, (rows, 1))))
    x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()   # bf16 values
    x[3] = 0.0                                                              # an all-zero row
    q, s = oracle.quantize_rows_e4m3(x)
    # the same rule with numpy's binary32 arithmetic and the library cast
    amax = np.abs(x).max(axis=1).astype(np.float32)
    s_ref = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    assert np.array_equal(s, s_ref)
    q_ref = _torch_codes((x / s_ref[:, None]).astype(np.float32))
    assert np.array_equal(q, q_ref)
    # properties: zero row, the largest element lands on +-448, error within half a step
    assert s[3] == 1.0 and not q[3].any()
    tab = oracle.e4m3_table()
    deq = oracle.dequantize_rows_e4m3(q, s)
    for r in range(rows):
        if r == 3:
            continue
        c = int(np.argmax(np.abs(x[r])))
        assert abs(tab[q[r, c]]) == 448.0
        big = np.abs(x[r]) >= s[r] * 2.0 ** -6
        rel = np.abs(deq[r, big] - x[r, big]) / np.abs(x[r, big])
        assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)
        assert np.abs(deq[r, ~big] - x[r, ~big]).max(initial=0) <= s[r] * 2.0 ** -10 * (1 + 1e-6)


def test_quantize_accepts_bf16_bits():
    rng = np.random.default_rng(5)
    x = torch.from_numpy(rng.standard_normal((4, 256)).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q1, s1 = oracle.quantize_rows_e4m3(bits)
    q2, s2 = oracle.quantize_rows_e4m3(x.to(torch.float32).numpy())
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
