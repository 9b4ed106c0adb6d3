"""Pins of the oracle's number formats and group operators against library
routines, closed forms and format specifications (no GPU).

- bfloat16 round-to-nearest-even: torch's CPU float32 -> bfloat16 conversion.
- OCP FP8 E4M3: torch's float8_e4m3fn decode table (all 256 codes) and its
  encoder for in-range values; saturation to +-448 (torch does not saturate).
- INT8: numpy's rint (round half to even) and clip.
- scale/accumulate/zero: numpy float32 arithmetic, and fp64 closed forms where the
  result is exactly representable.
- norm: math.fsum; an all-ones tensor has norm sqrt(n) exactly.
- block quantisation: block amax via numpy, codes via torch's encoder, the
  dequantisation error bound, zero blocks.
"""
import math
import random

import numpy as np
import pytest
import torch

from workloads.configs import TensorSpec


def _torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_rne_matches_torch(oracle_lib):
    hi = np.arange(65536, dtype=np.uint32) << 16
    lows = [0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1234, 0xC000]
    bits = np.concatenate([hi | lo for lo in lows])
    rng = np.random.default_rng(0)
    bits = np.concatenate([bits, rng.integers(0, 2 ** 32, 1 << 20, dtype=np.uint64).astype(np.uint32)])
    x = bits.view(np.float32)
    got = oracle_lib.f32_to_bf16_bits(x)
    want = _torch_bf16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    # NaN stays NaN with the sign kept
    back = (got[nan].astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.isnan(back))
    assert np.array_equal(np.signbit(back), np.signbit(x[nan]))


def test_bf16_known_values(oracle_lib):
    L = oracle_lib.lib()
    assert L.orc_f32_to_bf16(1.0) == 0x3F80
    assert L.orc_f32_to_bf16(-2.0) == 0xC000
    assert L.orc_f32_to_bf16(float("inf")) == 0x7F80
    # 1 + 2^-8 is exactly half-way between 1 and 1 + 2^-7: ties to even -> 1.0
    assert L.orc_f32_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is half-way between 1+2^-7 (odd) and 1+2^-6 (even) -> up
    assert L.orc_f32_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # the largest finite float32 rounds to infinity in bfloat16
    assert L.orc_f32_to_bf16(np.finfo(np.float32).max) == 0x7F80


def test_e4m3_decode_table_matches_torch(oracle_lib):
    codes = torch.arange(256, dtype=torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([oracle_lib.e4m3_value(c) for c in range(256)])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan].astype(np.float64))
    # OCP E4M3 landmarks: 448 is the largest finite value, 2^-9 the smallest
    # subnormal, 2^-6 the smallest normal, 1.0 = 0x38.
    assert oracle_lib.e4m3_value(0x7E) == 448.0
    assert oracle_lib.e4m3_value(0x01) == 2.0 ** -9
    assert oracle_lib.e4m3_value(0x08) == 2.0 ** -6
    assert oracle_lib.e4m3_value(0x38) == 1.0


def _e4m3_probe_values():
    vals = []
    # a dense sweep of float32 patterns from 2^-12 up to past 448
    for e in range(-12, 9):
        mant = np.arange(0, 1 << 23, 1 << 9, dtype=np.uint32)
        vals.append(((np.uint32(e + 127) << 23) | mant).view(np.float32))
    # exact midpoints between consecutive finite codes and their neighbours
    mags = np.array([float(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float())
                     for c in range(127)])
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    vals += [mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))]
    v = np.concatenate(vals + [np.array([0.0, 2.0 ** -10, 2.0 ** -149], np.float32)])
    return np.concatenate([v, -v]).astype(np.float32)


def test_e4m3_encode_matches_torch_in_range(oracle_lib):
    x = _e4m3_probe_values()
    x = x[np.abs(x) < 464.0]      # torch's encoder does not saturate beyond this
    got = oracle_lib.f32_to_e4m3_bits(x)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_e4m3_saturates(oracle_lib):
    x = np.array([448.0, 464.0, 500.0, 1e30, np.inf, -448.0, -1e9, -np.inf], np.float32)
    got = oracle_lib.f32_to_e4m3_bits(x)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0xFE]


def test_int8_matches_numpy(oracle_lib):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-200, 200, 200000).astype(np.float32),
                        (np.arange(-300, 301) / 2).astype(np.float32),
                        np.array([126.5, 127.49, -126.5, -127.5, 0.5, -0.5, 1.5], np.float32)])
    got = oracle_lib.f32_to_int8(x)
    want = np.clip(np.rint(x), -127, 127).astype(np.int8)
    assert np.array_equal(got, want)


def _plan_vectors(oracle_lib, sizes, m=2, align=4):
    specs = [TensorSpec(f"t{i}", n, 1, 1) for i, n in enumerate(sizes)]
    return specs, oracle_lib.plan_specs(specs, m, None, align)


def test_sac_matches_numpy_float32(oracle_lib):
    rng = np.random.default_rng(2)
    specs, p = _plan_vectors(oracle_lib, [1000, 3, 517])
    for scale in [0.25, 1.0 / 64, 0.3, 1.7]:
        g = rng.standard_normal(p.total).astype(np.float32)
        acc = rng.standard_normal(p.total).astype(np.float32)
        g0, acc0 = g.copy(), acc.copy()
        oracle_lib.scale_accum_zero(p, g, acc, scale)
        s32 = np.float32(scale)
        for t, s in enumerate(specs):
            sl = slice(int(p.offsets[t]), int(p.offsets[t]) + s.numel)
            want = acc0[sl] + g0[sl] * s32      # numpy: each op rounded to float32
            assert np.array_equal(acc[sl].view(np.uint32), want.view(np.uint32))
            assert np.all(g[sl].view(np.uint32) == 0)       # +0.0, bitwise
        # padding untouched
        mask = np.ones(p.total, bool)
        for t, s in enumerate(specs):
            mask[int(p.offsets[t]):int(p.offsets[t]) + s.numel] = False
        assert np.array_equal(g[mask], g0[mask]) and np.array_equal(acc[mask], acc0[mask])


def test_sac_exact_closed_form(oracle_lib):
    """Small dyadic values with s = 2^-k: the fp32 result equals the exact sum."""
    specs, p = _plan_vectors(oracle_lib, [4096])
    k = np.arange(-2048, 2048)
    g = (k * 2.0 ** -10).astype(np.float32)
    acc = ((k % 97) * 2.0 ** -6).astype(np.float32)
    gb = np.zeros(p.total, np.float32); ab = np.zeros(p.total, np.float32)
    o = int(p.offsets[0])
    gb[o:o + 4096] = g; ab[o:o + 4096] = acc
    oracle_lib.scale_accum_zero(p, gb, ab, 1.0 / 8)
    exact = acc.astype(np.float64) + g.astype(np.float64) / 8
    assert np.array_equal(ab[o:o + 4096].astype(np.float64), exact)


def test_sac_bf16_grads(oracle_lib):
    rng = np.random.default_rng(3)
    specs, p = _plan_vectors(oracle_lib, [777, 64])
    gf = rng.standard_normal(p.total).astype(np.float32) * np.float32(1e-3)
    g = _torch_bf16_bits(gf)
    acc = rng.standard_normal(p.total).astype(np.float32)
    acc0, g0 = acc.copy(), g.copy()
    oracle_lib.scale_accum_zero(p, g, acc, 1.0 / 16)
    o = int(p.offsets[0])
    gv = (g0[o:o + 777].astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(acc[o:o + 777], acc0[o:o + 777] + gv * np.float32(1 / 16))
    assert np.all(g[o:o + 777] == 0)


def test_norm_matches_fsum(oracle_lib):
    rng = np.random.default_rng(4)
    sizes = [1, 1000, 4096, 33333]
    specs, p = _plan_vectors(oracle_lib, sizes, m=3)
    buf = (rng.standard_normal(p.total) * 1e-3).astype(np.float32)
    norms, total, flag = oracle_lib.norm_nonfinite(p, buf)
    assert flag == 0
    tot = []
    for t, n in enumerate(sizes):
        x = buf[int(p.offsets[t]):int(p.offsets[t]) + n].astype(np.float64)
        sq = math.fsum(x * x)           # x*x is exact in fp64
        tot.append(sq)
        assert abs(norms[t] - math.sqrt(sq)) <= 1e-13 * math.sqrt(sq)
    assert abs(total - math.sqrt(math.fsum(tot))) <= 1e-13 * total


def test_norm_all_ones_and_flag(oracle_lib):
    specs, p = _plan_vectors(oracle_lib, [4096, 10, 0, 25])
    buf = np.zeros(p.total, np.float32)
    for t, n in enumerate([4096, 10, 0, 25]):
        buf[int(p.offsets[t]):int(p.offsets[t]) + n] = 1.0
    norms, total, flag = oracle_lib.norm_nonfinite(p, buf)
    assert norms[0] == 64.0 and norms[2] == 0.0 and norms[3] == 5.0
    assert total == math.sqrt(4096 + 10 + 25) and flag == 0
    for bad in [np.inf, -np.inf, np.nan]:
        b2 = buf.copy()
        b2[int(p.offsets[3]) + 7] = bad
        assert oracle_lib.norm_nonfinite(p, b2)[2] == 1
    # a non-finite value in the padding is outside every tensor and is not seen
    b3 = buf.copy()
    pad = int(p.offsets[1]) + 10
    assert pad < int(p.offsets[3])
    b3[pad] = np.inf
    assert oracle_lib.norm_nonfinite(p, b3)[2] == 0


def _quant_case(oracle_lib, R, C, qb, kind, seed):
    specs = [TensorSpec("v", 5, 1, 1), TensorSpec("w", R, C, qb[0], qb, kind)]
    p = oracle_lib.plan_specs(specs, 2, None, 16)
    rng = np.random.default_rng(seed)
    buf = np.zeros(p.total, np.float32)
    o = int(p.offsets[1])
    x = (rng.standard_normal((R, C)) * 0.02).astype(np.float32)
    x[0, : min(C, 3)] = 0.0
    buf[o:o + R * C] = x.reshape(-1)
    codes = np.full(p.total, 0xAB, np.uint8)
    scales = oracle_lib.block_quant(p, specs, buf, codes)
    return specs, p, x, codes[o:o + R * C].reshape(R, C), scales, codes


@pytest.mark.parametrize("R,C,qb,kind", [
    (256, 384, (128, 128), "e4m3"), (200, 130, (128, 128), "e4m3"),
    (64, 300, (1, 128), "int8"), (9, 64, (1, 128), "int8")])
def test_block_quant_structure(oracle_lib, R, C, qb, kind):
    specs, p, x, code, scales, allcodes = _quant_case(oracle_lib, R, C, qb, kind, 5)
    qr, qc = qb
    nbr, nbc = -(-R // qr), -(-C // qc)
    assert scales.size == nbr * nbc
    qmax = np.float32(448.0 if kind == "e4m3" else 127.0)
    for bi in range(nbr):
        for bj in range(nbc):
            blk = x[bi * qr:(bi + 1) * qr, bj * qc:(bj + 1) * qc]
            cb = code[bi * qr:(bi + 1) * qr, bj * qc:(bj + 1) * qc]
            amax = np.float32(np.abs(blk).max())
            scale = np.float32(amax / qmax) if amax > 0 else np.float32(1.0)
            assert scales[bi * nbc + bj] == scale
            v = blk / scale                      # numpy float32 division (IEEE)
            if kind == "e4m3":
                want = torch.from_numpy(np.ascontiguousarray(v)).to(torch.float8_e4m3fn) \
                    .view(torch.uint8).numpy()
                assert np.array_equal(cb, want)
                dec = torch.from_numpy(cb.copy()).view(torch.float8_e4m3fn).float().numpy()
                # relative half-ulp of E4M3 (3 mantissa bits) or the subnormal step
                bound = np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10)
                assert np.all(np.abs(dec - v) <= bound)
            else:
                want = np.clip(np.rint(v), -127, 127).astype(np.int8).view(np.uint8)
                assert np.array_equal(cb, want)
                assert np.all(np.abs(cb.view(np.int8) - v) <= 0.5 + 1e-4)
    # bytes of the vector tensor (not quantised) and of the padding are untouched
    o0 = int(p.offsets[0])
    assert np.all(allcodes[o0:o0 + 5] == 0xAB)


def test_block_quant_zero_block(oracle_lib):
    specs = [TensorSpec("w", 128, 128, 128, (128, 128), "e4m3")]
    p = oracle_lib.plan_specs(specs, 1, None, 16)
    buf = np.zeros(p.total, np.float32)
    codes = np.full(p.total, 0x55, np.uint8)
    scales = oracle_lib.block_quant(p, specs, buf, codes)
    assert scales.tolist() == [1.0]
    assert np.all(codes[:128 * 128] == 0)
