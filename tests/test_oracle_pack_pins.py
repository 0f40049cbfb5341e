"""Pins for the oracle's cache writer (latent rows -> bf16 or FP8 cache rows).

The pages name the step (their benchmark packs the KV with the same quantiser on both
sides: flashinfer PR "add topk=256 prefill-dsv4 dispatch", conversation, the GB10
benchmark's "Method" paragraph) but print no arithmetic. The reading under test: per
128 latent channels scale = fl32(amax / 448) (1 for an all-zero block), code = the E4M3FN
value nearest to fl32(x / scale) with ties to the even code and saturation at 448; rope
channels (and every channel of a bf16 row) are rounded to bf16, nearest with ties to even.

The expectations come from the E4M3FN and bfloat16 format definitions and from exact
arithmetic (every value written below is exactly representable), not from the oracle.
"""
import numpy as np

from sparse_top_mla_gb300 import synth

from . import npref

FP8, BF16 = 1, 0


def _row(latent, rope=None):
    x = np.zeros((1, 576), dtype=np.float32)
    x[0, :512] = latent
    if rope is not None:
        x[0, 512:] = rope
    return x


def _codes(oracle_mod, x):
    r = oracle_mod.pack_rows(x, FP8)
    return r[:, :512], r[:, 512:528].view(np.float32), r[:, 528:].view(np.uint16)


def _e4m3_positive_values():
    t = npref.e4m3_table()
    return np.array([t[c] for c in range(0x7F)], dtype=np.float64)  # codes 0x00..0x7E


def test_every_finite_code_round_trips(oracle_mod):
    vals = _e4m3_positive_values()  # 127 values, the largest is 448
    lat = np.zeros(512, dtype=np.float32)
    lat[:127] = vals                # block 0: all positive codes (amax 448 -> scale exactly 1)
    lat[128:255] = -vals            # block 1: all negative codes
    lat[256:383] = vals / 4         # block 2: amax 112 -> scale 1/4 exactly, codes unchanged
    codes, scale, _ = _codes(oracle_mod, _row(lat))
    assert scale[0, 0] == 1.0 and scale[0, 1] == 1.0 and scale[0, 2] == 0.25
    assert np.array_equal(codes[0, :127], np.arange(127, dtype=np.uint8))
    neg = (np.arange(127, dtype=np.uint8) | 0x80)
    neg[0] = 0x80  # -0.0 keeps its sign bit
    assert np.array_equal(codes[0, 128:255], neg)
    assert np.array_equal(codes[0, 256:383], np.arange(127, dtype=np.uint8))


def test_halfway_values_round_to_the_even_code(oracle_mod):
    vals = _e4m3_positive_values()
    mids = (vals[:-1] + vals[1:]) / 2          # 126 midpoints, each exact in fp32
    lat = np.zeros(512, dtype=np.float32)
    lat[0] = 448.0                              # scale 1
    lat[1:127] = mids
    lat[128] = 448.0
    lat[129:255] = -mids
    codes, scale, _ = _codes(oracle_mod, _row(lat))
    assert scale[0, 0] == 1.0
    for c in range(126):
        even = c if c % 2 == 0 else c + 1
        assert codes[0, 1 + c] == even, (c, mids[c], codes[0, 1 + c])
        assert codes[0, 129 + c] == (even | 0x80)
    # just off the midpoint the nearer code wins
    lat2 = np.zeros(512, dtype=np.float32)
    lat2[0] = 448.0
    lat2[1] = np.nextafter(np.float32(mids[8]), np.float32(0))  # between codes 8 and 9, below the tie
    lat2[2] = np.nextafter(np.float32(mids[8]), np.float32(1e9))
    codes2, _, _ = _codes(oracle_mod, _row(lat2))
    assert codes2[0, 1] == 8 and codes2[0, 2] == 9


def test_subnormal_codes(oracle_mod):
    lat = np.zeros(512, dtype=np.float32)
    lat[0] = 448.0
    q = 2.0 ** -9                               # subnormal quantum of E4M3FN
    lat[1:8] = np.arange(1, 8) * q              # codes 1..7
    lat[8] = 0.5 * q                            # tie between 0 and 1 -> 0
    lat[9] = 1.5 * q                            # tie between 1 and 2 -> 2
    lat[10] = 0.25 * q                          # -> 0
    lat[11] = 7.5 * q                           # tie between 7 (odd) and 8 (2^-6, code 8) -> 8
    codes, _, _ = _codes(oracle_mod, _row(lat))
    assert list(codes[0, 1:8]) == [1, 2, 3, 4, 5, 6, 7]
    assert list(codes[0, 8:12]) == [0, 2, 0, 8]


def test_saturation_never_gives_nan(oracle_mod):
    # amax / fl32(amax / 448) can exceed 448 by rounding; such values saturate to 448 (0x7E)
    rng = np.random.default_rng(11)
    amax = rng.uniform(1e-3, 1e3, size=4000).astype(np.float32)
    over = [a for a in amax if np.float32(a) / np.float32(np.float32(a) / np.float32(448.0)) > 448.0]
    assert len(over) > 10  # the case really occurs
    for a in over[:32]:
        lat = np.zeros(512, dtype=np.float32)
        lat[5] = a
        lat[6] = -a
        codes, _, _ = _codes(oracle_mod, _row(lat))
        assert codes[0, 5] == 0x7E and codes[0, 6] == 0xFE


def test_zero_block(oracle_mod):
    lat = np.zeros(512, dtype=np.float32)
    lat[128:256] = -0.0
    lat[300] = 3.0
    codes, scale, _ = _codes(oracle_mod, _row(lat))
    assert scale[0, 0] == 1.0 and scale[0, 1] == 1.0
    assert np.all(codes[0, :128] == 0) and np.all(codes[0, 128:256] == 0x80)
    assert scale[0, 2] == np.float32(3.0) / np.float32(448.0) and codes[0, 300] == 0x7E


def test_bf16_rounding(oracle_mod):
    vals = np.array([1 + 2 ** -8,         # tie between 1 and 1 + 2^-7 -> 1 (even)
                     1 + 3 * 2 ** -8,     # tie between 1 + 2^-7 and 1 + 2^-6 -> 1 + 2^-6 (even)
                     1 + 2 ** -8 + 2 ** -20,  # above the tie -> 1 + 2^-7
                     -2.5, 0.0, 3e38], dtype=np.float32)
    rope = np.zeros(64, dtype=np.float32)
    rope[:6] = vals
    _, _, bits = _codes(oracle_mod, _row(np.zeros(512, dtype=np.float32), rope))
    assert list(bits[0, :6]) == [0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000, 0x7F62]
    # a bf16 row is the same rounding on all 576 channels
    x = np.zeros((1, 576), dtype=np.float32)
    x[0, 10:16] = vals
    r = oracle_mod.pack_rows(x, BF16).view(np.uint16)
    assert list(r[0, 10:16]) == [0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000, 0x7F62]


def test_bf16_input_is_exact(oracle_mod):
    rng = np.random.default_rng(12)
    bits = synth.f32_to_bf16_bits(rng.standard_normal((7, 576)).astype(np.float32))
    as_f32 = (bits.astype(np.uint32) << 16).view(np.float32)
    for fmt in (BF16, FP8):
        assert np.array_equal(oracle_mod.pack_rows(bits, fmt), oracle_mod.pack_rows(as_f32, fmt))
    assert np.array_equal(oracle_mod.pack_rows(bits, BF16).view(np.uint16), bits)


def test_dequantised_error_is_within_half_a_step(oracle_mod):
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((64, 576)) * rng.uniform(1e-3, 1e3, size=(64, 1))).astype(np.float32)
    r = oracle_mod.pack_rows(x, FP8)
    table = npref.e4m3_table()
    vals = _e4m3_positive_values()
    for i in range(x.shape[0]):
        scale = r[i, 512:528].view(np.float32).astype(np.float64)
        for b in range(4):
            y = x[i, 128 * b:128 * (b + 1)].astype(np.float64) / scale[b]
            got = table[r[i, 128 * b:128 * (b + 1)]]
            # local spacing of E4M3 around |y|
            k = np.clip(np.searchsorted(vals, np.abs(y), side="right") - 1, 0, 125)
            step = vals[k + 1] - vals[k]
            assert np.all(np.abs(got - y) <= step / 2 + 1e-6 * np.abs(y))


def test_agrees_with_the_workload_generators_encoder(oracle_mod):
    # synth.encode_rows is a second, separately written encoder of the same definition
    # (bit manipulation rather than a search over codes)
    rng = np.random.default_rng(14)
    x = rng.standard_normal((300, 576)).astype(np.float32)
    x[::7] *= 1e-4
    x[::11] *= 1e4
    x[5, :128] = 0.0
    for fmt in (BF16, FP8):
        assert np.array_equal(oracle_mod.pack_rows(x, fmt), synth.encode_rows(x, fmt))
