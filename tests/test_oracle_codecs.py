"""Pins for the oracle's number-format codecs against library casts and closed forms."""
import numpy as np

import oracle
import pytest
import torch

from oracle import decode_bf16, decode_e4m3, encode_e4m3, unpack_int4, decode_int4_grouped
from synth.inputs import _pack_int4, _encode_expert


def test_bf16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = decode_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    # closed forms from the format definition
    assert decode_e4m3(np.array([0x7E]))[0] == 448.0
    assert decode_e4m3(np.array([0x01]))[0] == 2.0 ** -9
    assert decode_e4m3(np.array([0x08]))[0] == 2.0 ** -6
    assert decode_e4m3(np.array([0x38]))[0] == 1.0
    assert decode_e4m3(np.array([0xB8]))[0] == -1.0


def _e4m3_probe_values():
    finite = np.sort(np.unique(decode_e4m3(np.arange(256, dtype=np.uint8))))
    finite = finite[np.isfinite(finite)]
    mids = (finite[:-1] + finite[1:]) / 2.0
    f32 = np.float32
    vals = [finite, mids]
    for m in (mids, finite):
        m32 = m.astype(f32)
        vals.append(np.nextafter(m32, f32(np.inf)).astype(np.float64))
        vals.append(np.nextafter(m32, f32(-np.inf)).astype(np.float64))
    rng = np.random.default_rng(0)
    vals.append(rng.standard_normal(200_000) * 30.0)
    vals.append(np.exp2(rng.uniform(-12, 9, 200_000)) * rng.choice([-1, 1], 200_000))
    v = np.concatenate(vals).astype(np.float32)
    return v[np.abs(v) < 464.0]


def test_e4m3_encode_matches_torch_cast_in_range():
    v = _e4m3_probe_values()
    ours = encode_e4m3(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_saturates():
    big = np.array([448.0, 463.9, 464.0, 470.0, 1e6, 3e38], dtype=np.float32)
    assert np.all(decode_e4m3(encode_e4m3(big)) == 448.0)
    assert np.all(decode_e4m3(encode_e4m3(-big)) == -448.0)
    assert encode_e4m3(np.array([np.nan], dtype=np.float32))[0] & 0x7F == 0x7F


def test_int4_unpack_closed_form_all_bytes():
    b = np.arange(256, dtype=np.uint8)
    q = unpack_int4(b[:, None])
    lo = b & 0xF
    hi = b >> 4
    sext = lambda v: np.where(v >= 8, v.astype(np.int64) - 16, v.astype(np.int64))
    assert np.array_equal(q[:, 0], sext(lo))
    assert np.array_equal(q[:, 1], sext(hi))
    assert q.min() == -8 and q.max() == 7


def test_int4_pack_matches_unpack():
    g = torch.Generator().manual_seed(3)
    codes = torch.randint(-8, 8, (5, 64), generator=g, dtype=torch.int8)
    packed = _pack_int4(codes).numpy()
    assert np.array_equal(unpack_int4(packed), codes.numpy().astype(np.int64))


def test_int4_grouped_decode_brute_force():
    g = torch.Generator().manual_seed(4)
    w = torch.randn((3, 256), generator=g) * 0.02
    packed, s16 = _encode_expert(w, "int4", 128)
    deq = decode_int4_grouped(packed.numpy(), s16.numpy(), 128)
    q = unpack_int4(packed.numpy())
    for r in range(3):
        for k in range(256):
            assert deq[r, k] == q[r, k] * float(s16[r, k // 128])
    # symmetric quantisation error is at most half a step per element
    step = np.repeat(s16.float().numpy(), 128, axis=1)
    assert np.all(np.abs(deq - w.numpy()) <= step * 0.5 + 1e-12)


# ------------------------------------------------------ int4 with zero points

def test_unpack_uint4_all_bytes():
    b = np.arange(256, dtype=np.uint8).reshape(1, 256)
    q = oracle.unpack_uint4(b)
    assert q.shape == (1, 512)
    for v in range(256):
        assert q[0, 2 * v] == v & 0xF and q[0, 2 * v + 1] == v >> 4


def test_decode_zp_brute_force():
    rng = np.random.default_rng(5)
    rows, K, G = 3, 256, 128
    packed = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    scales = rng.uniform(1e-3, 2e-2, (rows, K // G)).astype(np.float16)
    zeros = rng.integers(0, 16, (rows, K // G), dtype=np.uint8)
    got = oracle.decode_int4_grouped_zp(packed, scales.view(np.uint16), zeros, G)
    for r in range(rows):
        for k in range(K):
            byte = int(packed[r, k // 2])
            q = (byte >> 4) if k % 2 else (byte & 0xF)
            want = (q - int(zeros[r, k // G])) * float(scales[r, k // G])
            assert got[r, k] == want


def test_zero_point_eight_on_flipped_nibbles_is_the_signed_format():
    # a two's-complement nibble n read as unsigned after flipping bit 3 is n + 8,
    # so (q - 8) * s with q = nibble ^ 8 reproduces the symmetric signed decode
    rng = np.random.default_rng(6)
    packed = rng.integers(0, 256, (4, 128), dtype=np.uint8)
    scales = rng.uniform(1e-3, 2e-2, (4, 2)).astype(np.float16).view(np.uint16)
    sym = oracle.decode_int4_grouped(packed, scales, 128)
    zp = oracle.decode_int4_grouped_zp(packed ^ np.uint8(0x88), scales, np.full((4, 2), 8, np.uint8), 128)
    assert np.array_equal(sym, zp)


def test_zero_point_zero_gives_nonnegative_multiples():
    packed = np.arange(64, dtype=np.uint8).reshape(1, 64)
    scales = np.array([[np.float16(0.5)]]).view(np.uint16)
    w = oracle.decode_int4_grouped_zp(packed, scales, np.zeros((1, 1), np.uint8), 128)
    assert (w >= 0).all() and w.max() == 7.5  # q = 15 at most, times 0.5


def test_zero_point_input_encoding_round_trips_within_half_a_step():
    from synth.inputs import _encode_expert_zp
    g = torch.Generator().manual_seed(2)
    w = torch.randn(6, 256, generator=g) * 0.02
    packed, s, z = _encode_expert_zp(w, 128)
    assert int(z.max()) <= 15
    dec = oracle.decode_int4_grouped_zp(packed.numpy(), s.numpy().view(np.uint16), z.numpy(), 128)
    step = np.repeat(s.float().numpy().astype(np.float64), 128, axis=-1)
    # rounding to the nearest level (edge groups may clamp by at most one step)
    assert (np.abs(dec - w.double().numpy()) <= step * 1.0 + 1e-12).all()


# ---------------------------------------------------------------- int8 group-128


def test_int8_codes_are_twos_complement_bytes():
    b = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(b.copy()).view(torch.int8).numpy().astype(np.int64)
    assert np.array_equal(oracle.int8_codes(b), want)


def test_int8_grouped_decode_brute_force():
    rng = np.random.default_rng(5)
    rows, K, G = 3, 384, 128
    codes = rng.integers(0, 256, size=(rows, K), dtype=np.uint8)
    s = rng.uniform(0.01, 2.0, size=(rows, K // G)).astype(np.float16)
    z = rng.integers(0, 256, size=(rows, K // G), dtype=np.uint8)
    sym = oracle.decode_int8_grouped(codes, s, G)
    asym = oracle.decode_int8_grouped_zp(codes, s, z, G)
    for r in range(rows):
        for k in range(K):
            b = int(codes[r, k])
            sc = float(s[r, k // G])
            assert sym[r, k] == (b - 256 if b >= 128 else b) * sc
            assert asym[r, k] == (b - int(z[r, k // G])) * sc


def test_int8_zero_point_128_on_flipped_sign_bits_is_the_signed_format():
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 256, size=(4, 256), dtype=np.uint8)
    s = rng.uniform(0.01, 1.0, size=(4, 2)).astype(np.float16)
    z = np.full((4, 2), 128, dtype=np.uint8)
    assert np.array_equal(oracle.decode_int8_grouped_zp(codes ^ 0x80, s, z, 128),
                          oracle.decode_int8_grouped(codes, s, 128))


def test_int8_agrees_with_int4_on_the_int4_range():
    # a code in [-8, 7] means the same in both formats; same scales, same groups
    rng = np.random.default_rng(7)
    c = rng.integers(-8, 8, size=(5, 512))
    s = rng.uniform(0.01, 1.0, size=(5, 4)).astype(np.float16)
    from synth.inputs import _pack_int4
    packed = _pack_int4(torch.from_numpy(c).to(torch.int8)).numpy()
    assert np.array_equal(oracle.decode_int8_grouped(c.astype(np.int8).view(np.uint8), s, 128),
                          oracle.decode_int4_grouped(packed, s, 128))


@pytest.mark.parametrize("zp", [False, True])
def test_int8_input_encoding_round_trips(zp):
    from synth.inputs import _encode_expert, _encode_expert_zp
    g = torch.Generator().manual_seed(3)
    w = torch.randn(6, 256, generator=g) * 0.02
    if zp:
        q, s, z = _encode_expert_zp(w, 128, bits=8)
        assert q.shape == w.shape
        dec = oracle.decode_int8_grouped_zp(q.numpy(), s.numpy(), z.numpy(), 128)
    else:
        q, s = _encode_expert(w, "int8", 128)
        dec = oracle.decode_int8_grouped(q.numpy(), s.numpy(), 128)
    step = np.repeat(s.float().numpy().astype(np.float64), 128, axis=-1)
    assert (np.abs(dec - w.double().numpy()) <= step + 1e-12).all()
    # nearest level: most errors within half a step
    assert np.mean(np.abs(dec - w.double().numpy()) <= 0.5 * step + 1e-9) > 0.99
