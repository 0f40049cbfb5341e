"""Host tests of the seeded input generator (formats, determinism, index sets)."""
import numpy as np

from sparse_top_mla_gb300 import synth

from . import npref


def test_e4m3_encoder_roundtrips_every_finite_code():
    table = npref.e4m3_table()
    codes = np.arange(256, dtype=np.uint8)
    finite = ~np.isnan(table)
    enc = synth.e4m3_encode(table[finite].astype(np.float32))
    # +0 and -0 both encode to their own sign
    assert np.array_equal(enc, codes[finite])


def test_e4m3_encoder_rounds_half_to_even_and_saturates():
    table = npref.e4m3_table()
    pos = table[:127]
    mids = (pos[:-1] + pos[1:]) / 2
    enc = synth.e4m3_encode(mids.astype(np.float32))
    # a midpoint goes to the neighbour with an even code
    lo = np.arange(126)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(enc, expect.astype(np.uint8))
    assert synth.e4m3_encode(np.array([1e9, -1e9, 449.0, 500.0], dtype=np.float32)).tolist() == [0x7E, 0xFE, 0x7E, 0x7E]


def test_e4m3_encoder_is_nearest():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(4000) * 30, rng.standard_normal(4000) * 0.02]).astype(np.float32)
    table = npref.e4m3_table()
    dec = table[synth.e4m3_encode(x)]
    pos = table[:127]
    best = np.min(np.abs(np.abs(x.astype(np.float64))[:, None] - pos[None, :]), axis=1)
    assert np.allclose(np.abs(np.abs(dec) - np.abs(x)), best, rtol=0, atol=0)


def test_bf16_rounding():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 1.0 + 2 ** -7 + 2 ** -8], dtype=np.float32)
    got = npref.bf16_to_f64(synth.f32_to_bf16_bits(x))
    assert got.tolist() == [1.0, 1.0, 1.0 + 2 ** -7, -2.5, 1.0 + 2 ** -6]


def test_fp8_rows_dequantise_close_to_source():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((16, 576)).astype(np.float32)
    raw = synth.encode_rows(x, synth.FMT_FP8)
    s = synth._kvset(raw.reshape(-1), synth.FMT_FP8, 656, 656 * 64, 1, np.zeros((1, 1)), [16], np.zeros((1, 1)), 1)
    for r in range(16):
        k = npref.decode_row(s, 0, r)
        assert np.max(np.abs(k[:512] - x[r, :512])) <= np.max(np.abs(x[r, :512])) * 2 ** -4
        assert np.max(np.abs(k[512:] - x[r, 512:])) <= np.max(np.abs(x[r, 512:])) * 2 ** -8


def test_generator_is_deterministic():
    a = synth.small_case(5, T=3, H=2, topk=64, ctx=256, fmt=synth.FMT_FP8, sink=True, mask_p=0.1)
    b = synth.small_case(5, T=3, H=2, topk=64, ctx=256, fmt=synth.FMT_FP8, sink=True, mask_p=0.1)
    assert np.array_equal(a.main.cache, b.main.cache)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.main.indices, b.main.indices)
    assert np.array_equal(a.sink, b.sink)


def test_distinct_indices():
    rng = np.random.default_rng(2)
    hi = np.array([10, 63, 5000, 100000, 300])
    idx = synth.distinct_indices(rng, hi, 128)
    for t, h in enumerate(hi):
        row = idx[t]
        valid = row[row >= 0]
        assert len(valid) == min(128, h + 1)
        assert len(np.unique(valid)) == len(valid)
        assert valid.min() >= 0 and valid.max() <= h
        assert np.all(row[len(valid):] == -1)


def test_config1_shape():
    w = synth.config(1)
    assert (w.T, w.H, w.main.topk) == (4, 16, 128)
    assert w.main.cache.nbytes == 256 * 1152
    assert w.flops() == 2 * 4 * 16 * 128 * 1088
    assert w.sink is None


def test_padded_cache_rows_are_written():
    w = synth.small_case(3, T=1, H=1, topk=64, ctx=128, row_pad=32, page_pad=128)
    s = w.main
    pages = s.cache.reshape(s.num_pages, s.page_stride)
    rows = pages[:, :64 * s.row_stride].reshape(s.num_pages, 64, s.row_stride)
    assert not np.all(rows[:, :, :1152] == 0xFF)
    assert np.all(rows[:, :, 1152:] == 0xFF) and np.all(pages[:, 64 * s.row_stride:] == 0xFF)
