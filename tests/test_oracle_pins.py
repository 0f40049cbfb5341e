"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics, not by the oracle itself.

Each test would fail under a plausible mistake in the oracle: a dropped sink term, the
sink counted in the LSE, a wrong scale, a transposed operand, V taken from the wrong
channels, masked entries leaking, a wrong page translation, a wrong E4M3 decode.
"""
import json
import math
import os
import struct

import numpy as np
import pytest

from sparse_top_mla_gb300 import synth
from sparse_top_mla_gb300.synth import D_QK, D_V, FMT_BF16, FMT_FP8, PAGE

from . import npref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _run(oracle_mod, w, tokens=None):
    return oracle_mod.attention(w, tokens=tokens, nthreads=4)


def _q64(w):
    return npref.bf16_to_f64(w.q)


# --------------------------------------------------------------------------- formats
def test_e4m3_table_matches_spec_formula(oracle_mod):
    table = npref.e4m3_table()
    for code in range(256):
        v = oracle_mod.e4m3_value(code)
        if np.isnan(table[code]):
            assert np.isnan(v), code
        else:
            assert v == table[code], (code, v, table[code])
    # spot values from the format definition
    assert oracle_mod.e4m3_value(0x7E) == 448.0
    assert oracle_mod.e4m3_value(0x01) == 2.0 ** -9
    assert oracle_mod.e4m3_value(0x08) == 2.0 ** -6
    assert oracle_mod.e4m3_value(0xB8) == -1.0


def test_bf16_decode(oracle_mod):
    for bits, val in [(0x3F80, 1.0), (0xC000, -2.0), (0x0000, 0.0), (0x3E80, 0.25), (0x4040, 3.0),
                      (0x0001, 2.0 ** -133)]:
        assert oracle_mod.bf16_value(bits) == val


# --------------------------------------------------------------------------- golden
def _golden_workload(ex):
    fmt = FMT_BF16 if ex["fmt"] == "bf16" else FMT_FP8
    ctx, H = ex["ctx"], ex["H"]
    row_bytes = synth.ROW_BYTES_BF16 if fmt == FMT_BF16 else synth.ROW_BYTES_FP8
    cache = np.full(ctx * row_bytes, 0xFF, dtype=np.uint8)  # NaN everywhere
    rows = cache.reshape(ctx, row_bytes)
    if fmt == FMT_BF16:
        for r, chans in ex["rows"].items():
            vals = np.zeros(D_QK, dtype=np.float32)
            for c, v in chans.items():
                vals[int(c)] = v
            rows[int(r)] = synth.f32_to_bf16_bits(vals).view(np.uint8)
    else:
        for r, spec in ex["fp8_rows"].items():
            raw = np.zeros(row_bytes, dtype=np.uint8)
            for c, code in spec["codes"].items():
                raw[int(c)] = code
            raw[512:528] = np.array(spec["scales"], dtype=np.float32).view(np.uint8)
            rope = np.zeros(64, dtype=np.float32)
            for c, v in spec["rope"].items():
                rope[int(c)] = v
            raw[528:] = synth.f32_to_bf16_bits(rope).view(np.uint8)
            rows[int(r)] = raw
    qv = np.zeros((1, H, D_QK), dtype=np.float32)
    for c, v in ex["q"].items():
        qv[0, :, int(c)] = v
    q = synth.f32_to_bf16_bits(qv)
    idx = np.array([ex["indices"]], dtype=np.int32)
    main = synth._kvset(cache, fmt, row_bytes, ctx * row_bytes, 1, np.array([[0]]), [ctx], idx, idx.shape[1])
    sink = None if ex["sink"] is None else np.array(ex["sink"], dtype=np.float32)
    return synth.Workload(ex["name"], 1, H, q, np.zeros(1, np.int32), main, None, sink, ex["sm_scale"])


@pytest.mark.parametrize("k", range(3))
def test_golden_worked_examples(oracle_mod, k):
    ex = json.load(open(GOLDEN))["examples"][k]
    O, lse = _run(oracle_mod, _golden_workload(ex))
    for c, v in ex["expect_O"].items():
        assert O[0, 0, int(c)] == pytest.approx(v, rel=1e-14, abs=1e-15)
    rest = np.delete(O[0, 0], [int(c) for c in ex["expect_O"]])
    assert np.all(rest == 0.0)
    assert lse[0, 0] == pytest.approx(ex["expect_lse"], rel=1e-14)


# --------------------------------------------------------------------------- reductions
@pytest.mark.parametrize("fmt", [FMT_BF16, FMT_FP8])
@pytest.mark.parametrize("with_sink", [False, True])
def test_full_coverage_equals_dense_mqa(oracle_mod, fmt, with_sink):
    """topk covering every cached token = dense multi-query attention."""
    ctx, T, H = 192, 3, 4
    w = synth.small_case(11 + fmt, T=T, H=H, topk=ctx, ctx=ctx, fmt=fmt, sink=with_sink)
    O, lse = _run(oracle_mod, w)
    q = _q64(w)
    K = np.stack([npref.decode_logical(w.main, 0, i) for i in range(ctx)])
    for t in range(T):
        Or, Lr = npref.dense_mqa(q[t], K, float(np.float32(w.sm_scale)), w.sink)
        np.testing.assert_allclose(O[t], Or, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse[t], Lr, rtol=1e-12)


def test_sink_minus_inf_is_no_sink(oracle_mod):
    w = synth.small_case(3, T=3, H=5, topk=128, ctx=256, sink=False, mask_p=0.2)
    O0, L0 = _run(oracle_mod, w)
    w2 = synth.replace(w, sink=np.full(w.H, -np.inf, dtype=np.float32))
    O1, L1 = _run(oracle_mod, w2)
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)


def test_sink_renormalisation_relation(oracle_mod):
    """With a sink, O_sink = O * e^LSE / (e^LSE + e^sigma) and LSE is unchanged."""
    w = synth.small_case(4, T=3, H=6, topk=128, ctx=300, sink=True, mask_p=0.1)
    Os, Ls = _run(oracle_mod, w)
    On, Ln = _run(oracle_mod, synth.replace(w, sink=None))
    sig = w.sink.astype(np.float64)[None, :]
    factor = np.exp(Ln) / (np.exp(Ln) + np.exp(sig))
    np.testing.assert_allclose(Os, On * factor[:, :, None], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(Ls, Ln, rtol=1e-13)


# --------------------------------------------------------------------------- invariances
def test_permuting_indices_leaves_output(oracle_mod):
    w = synth.small_case(5, T=4, H=3, topk=192, ctx=512, fmt=FMT_FP8, sink=True, mask_p=0.1)
    O0, L0 = _run(oracle_mod, w)
    rng = np.random.default_rng(0)
    idx = w.main.indices.copy()
    for t in range(w.T):
        idx[t] = idx[t, rng.permutation(idx.shape[1])]
    O1, L1 = _run(oracle_mod, synth.with_indices(w, idx))
    np.testing.assert_allclose(O1, O0, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(L1, L0, rtol=1e-13)


def test_masked_entries_contribute_nothing(oracle_mod):
    w = synth.small_case(6, T=4, H=3, topk=128, ctx=256, mask_p=0.3, sink=True)
    O0, L0 = _run(oracle_mod, w)
    idx = w.main.indices.copy()
    neg = idx < 0
    variants = []
    a = idx.copy(); a[neg] = -7; variants.append(a)
    b = idx.copy(); b[neg] = 256; variants.append(b)            # == seq_len
    c = idx.copy(); c[neg] = 10 ** 6; variants.append(c)        # far beyond seq_len
    for v in variants:
        O1, L1 = _run(oracle_mod, synth.with_indices(w, v))
        assert np.array_equal(O0, O1) and np.array_equal(L0, L1)


def test_unreferenced_rows_are_never_read(oracle_mod):
    """NaN-poison every cache row that no valid entry references: output bit-identical."""
    w = synth.small_case(7, T=3, H=2, topk=64, ctx=512, mask_p=0.2, spare_pages=2)
    O0, L0 = _run(oracle_mod, w)
    s = w.main
    used = set()
    for t in range(w.T):
        for i in s.indices[t, :s.topk]:
            if 0 <= i < 512:
                used.add((int(s.block_table[0, i // PAGE]), int(i % PAGE)))
    cache = s.cache.copy()
    for p in range(s.num_pages):
        for r in range(PAGE):
            if (p, r) not in used:
                off = p * s.page_stride + r * s.row_stride
                cache[off:off + s.row_stride] = 0xFF
    O1, L1 = _run(oracle_mod, synth.replace(w, main=synth.replace(s, cache=cache)))
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)
    assert np.isfinite(O0).all()


def test_page_outside_cache_is_masked(oracle_mod):
    w = synth.small_case(8, T=2, H=2, topk=64, ctx=256, shuffle_pages=False)
    bt = w.main.block_table.copy()
    bt[0, 1] = w.main.num_pages + 3      # logical page 1 -> nonexistent physical page
    O1, L1 = _run(oracle_mod, synth.replace(w, main=synth.replace(w.main, block_table=bt)))
    idx = w.main.indices.copy()
    idx[(idx >= 64) & (idx < 128)] = -1
    O2, L2 = _run(oracle_mod, synth.with_indices(w, idx))
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_head_independence_bitwise(oracle_mod):
    """A head's output is identical whether the call has H or 2H heads."""
    w = synth.small_case(9, T=3, H=4, topk=128, ctx=256, sink=True, mask_p=0.1)
    O0, L0 = _run(oracle_mod, w)
    rng = np.random.default_rng(1)
    extra_q = synth.make_q(rng, w.T, w.H)
    q2 = np.concatenate([w.q, extra_q], axis=1)
    sink2 = np.concatenate([w.sink, rng.standard_normal(w.H).astype(np.float32)])
    O1, L1 = _run(oracle_mod, synth.replace(w, H=2 * w.H, q=q2, sink=sink2))
    assert np.array_equal(O1[:, :w.H], O0) and np.array_equal(L1[:, :w.H], L0)


def test_physical_page_shuffle_invariance(oracle_mod):
    w = synth.small_case(10, T=3, H=2, topk=128, ctx=512, fmt=FMT_FP8, shuffle_pages=False)
    O0, L0 = _run(oracle_mod, w)
    s = w.main
    perm = np.random.default_rng(2).permutation(s.num_pages)  # new physical slot of old page p
    pages = s.cache.reshape(s.num_pages, s.page_stride)
    moved = np.empty_like(pages)
    moved[perm] = pages
    bt = perm[s.block_table].astype(np.int32)
    s2 = synth.replace(s, cache=moved.reshape(-1), block_table=bt)
    O1, L1 = _run(oracle_mod, synth.replace(w, main=s2))
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)


def test_strided_views_equal_contiguous(oracle_mod):
    w = synth.small_case(12, T=3, H=3, topk=128, ctx=256, idx_pad=40, row_pad=64, page_pad=256)
    O0, L0 = _run(oracle_mod, w)
    wide = np.zeros((w.T, w.H + 2, D_QK + 32), dtype=np.uint16)
    wide[:, :w.H, :D_QK] = w.q
    w2 = synth.replace(w, q=wide[:, :w.H, :D_QK])
    O1, L1 = _run(oracle_mod, w2)
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)
    contig = synth.with_indices(w, np.ascontiguousarray(w.main.indices[:, :w.main.topk]))
    O2, L2 = _run(oracle_mod, contig)
    assert np.array_equal(O0, O2) and np.array_equal(L0, L2)


def test_topk_length_equals_truncation(oracle_mod):
    w = synth.small_case(13, T=5, H=2, topk=128, ctx=256, topk_length=True)
    O0, L0 = _run(oracle_mod, w)
    idx = w.main.indices.copy()
    for t in range(w.T):
        idx[t, w.main.topk_length[t]:] = -1
    O1, L1 = _run(oracle_mod, synth.replace(w, main=synth.replace(w.main, indices=idx, topk_length=None)))
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)


def test_extra_set_merges_into_one_softmax(oracle_mod):
    """Main + extra over the same cache == one set holding both index lists."""
    w = synth.small_case(14, T=3, H=3, topk=128, ctx=512, sink=True, mask_p=0.05)
    rng = np.random.default_rng(3)
    xidx = synth.distinct_indices(rng, np.full(w.T, 511), 64)
    extra = synth.replace(w.main, indices=xidx, topk=64)
    O0, L0 = _run(oracle_mod, synth.replace(w, extra=extra))
    both = np.concatenate([w.main.indices[:, :w.main.topk], xidx], axis=1)
    O1, L1 = _run(oracle_mod, synth.with_indices(w, both))
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)


# --------------------------------------------------------------------------- closed forms
def test_single_valid_index(oracle_mod):
    w = synth.small_case(15, T=2, H=3, topk=64, ctx=256, fmt=FMT_FP8)
    idx = np.full((w.T, 64), -1, dtype=np.int32)
    idx[0, 17] = 100
    idx[1, 0] = 3
    O, L = _run(oracle_mod, synth.with_indices(w, idx))
    q = _q64(w)
    for t, pos in [(0, 100), (1, 3)]:
        K = npref.decode_logical(w.main, 0, pos)
        np.testing.assert_allclose(O[t], np.broadcast_to(K[:D_V], (w.H, D_V)), rtol=1e-15, atol=0)
        np.testing.assert_allclose(L[t], (q[t] @ K) * float(np.float32(w.sm_scale)), rtol=1e-13)


def test_identical_rows(oracle_mod):
    """n identical valid rows: O = V, LSE = x + log n."""
    w = synth.small_case(16, T=1, H=2, topk=64, ctx=128, shuffle_pages=False)
    s = w.main
    cache = s.cache.copy()
    row0 = cache[:s.row_stride].copy()
    n = 40
    idx = np.full((1, 64), -1, dtype=np.int32)
    idx[0, :n] = np.arange(n) + 10
    for i in range(10, 10 + n):
        cache[i * s.row_stride:(i + 1) * s.row_stride] = row0
    w2 = synth.replace(w, main=synth.replace(s, cache=cache, indices=idx))
    O, L = _run(oracle_mod, w2)
    K = npref.decode_row(s, 0, 0)
    x = (_q64(w)[0] @ K) * float(np.float32(w.sm_scale))
    np.testing.assert_allclose(O[0], np.broadcast_to(K[:D_V], (2, D_V)), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(L[0], x + math.log(n), rtol=1e-13)


def test_zero_query_gives_mean_of_values(oracle_mod):
    w = synth.small_case(17, T=2, H=2, topk=128, ctx=256, mask_p=0.25, fmt=FMT_FP8)
    w0 = synth.replace(w, q=np.zeros_like(w.q))
    O, L = _run(oracle_mod, w0)
    for t in range(w.T):
        pos = [int(i) for i in w.main.indices[t] if i >= 0]
        V = np.stack([npref.decode_logical(w.main, 0, p)[:D_V] for p in pos])
        np.testing.assert_allclose(O[t], np.broadcast_to(V.mean(axis=0), (2, D_V)), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(L[t], math.log(len(pos)), rtol=1e-14)


@pytest.mark.parametrize("with_sink", [False, True])
def test_empty_row(oracle_mod, with_sink):
    w = synth.small_case(18, T=2, H=2, topk=64, ctx=128, sink=with_sink)
    idx = w.main.indices.copy()
    idx[1] = -1
    O, L = _run(oracle_mod, synth.with_indices(w, idx))
    assert np.all(O[1] == 0.0) and np.all(np.isneginf(L[1]))
    assert np.isfinite(L[0]).all()
    bad_seq = synth.replace(w, token_seq=np.array([0, 5], dtype=np.int32))
    O2, L2 = _run(oracle_mod, bad_seq)
    assert np.all(O2[1] == 0.0) and np.all(np.isneginf(L2[1]))


# --------------------------------------------------------------------------- brute force
def test_brute_force_tiny(oracle_mod):
    """A straight-line scalar loop, written separately, agrees to 1e-12."""
    w = synth.small_case(19, T=2, H=2, topk=64, ctx=128, sink=True, mask_p=0.2, fmt=FMT_FP8)
    O, L = _run(oracle_mod, w)
    s = w.main
    e4 = npref.e4m3_table()

    def bf(b):
        return struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]

    def row(pos):
        page = int(s.block_table[0, pos // 64])
        off = page * s.page_stride + (pos % 64) * s.row_stride
        raw = bytes(s.cache[off:off + 656])
        sc = struct.unpack("<4f", raw[512:528])
        k = [e4[raw[c]] * sc[c // 128] for c in range(512)]
        k += [bf(struct.unpack("<H", raw[528 + 2 * c:530 + 2 * c])[0]) for c in range(64)]
        return k

    scale = float(np.float32(w.sm_scale))
    for t in range(w.T):
        rows = [row(int(i)) for i in s.indices[t] if 0 <= i < 128]
        for h in range(w.H):
            qv = [bf(b) for b in w.q[t, h]]
            xs = [scale * sum(a * b for a, b in zip(qv, k)) for k in rows]
            sig = float(w.sink[h])
            m = max(xs + [sig])
            ws = [math.exp(x - m) for x in xs]
            D = sum(ws) + math.exp(sig - m)
            for c in range(0, 512, 37):
                ref = sum(wj * k[c] for wj, k in zip(ws, rows)) / D
                assert O[t, h, c] == pytest.approx(ref, rel=1e-12, abs=1e-14)
            assert L[t, h] == pytest.approx(m + math.log(sum(ws)), rel=1e-12)


def test_token_subset_matches_full(oracle_mod):
    w = synth.small_case(20, T=6, H=2, topk=64, ctx=128)
    O, L = _run(oracle_mod, w)
    sel = np.array([4, 1, 5])
    O2, L2 = _run(oracle_mod, w, tokens=sel)
    assert np.array_equal(O2, O[sel]) and np.array_equal(L2, L[sel])
