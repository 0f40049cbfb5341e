"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle.

Tolerances (stated with the method): max|O - O_ref| <= 2e-2 * max|O_ref| when every cache
is bf16, <= 4e-2 when any cache is FP8; |LSE - LSE_ref| <= 1e-2 where LSE_ref is finite.
Where the oracle has an empty set the GPU must give exactly O = 0 and LSE = -inf. Index
and mask handling is checked bit-exactly through invariances of the GPU output itself.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from sparse_top_mla_gb300 import binding, synth  # noqa: E402
from sparse_top_mla_gb300 import build as smla_build  # noqa: E402
from sparse_top_mla_gb300.synth import FMT_BF16, FMT_FP8  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smla_build.build()
    binding.load()
    yield
    assert binding.device_error() == 0


def tol_for(w):
    fp8 = w.main.fmt == FMT_FP8 or (w.extra is not None and w.extra.fmt == FMT_FP8)
    return 4e-2 if fp8 else 2e-2


def run_gpu(w, mode, **kw):
    dp = binding.DeviceProblem(w, **kw)
    dp.run(mode)
    O, L = dp.results()
    assert binding.device_error() == 0
    return O, L, dp


def check_against(w, O, L, O_ref, L_ref, what="", lse_rel=0.0):
    tol = tol_for(w)
    empty = np.isneginf(L_ref)
    assert np.all(np.isneginf(L[empty])), f"{what}: empty rows must give LSE=-inf"
    assert np.all(O[empty] == 0.0), f"{what}: empty rows must give O=0"
    fin = ~empty
    assert np.all(np.isfinite(L[fin])), what
    assert np.all(np.isfinite(O)), what
    scale = max(np.max(np.abs(O_ref)), 1e-30)
    err = np.max(np.abs(O - O_ref)) / scale
    lerr = np.max(np.abs(L[fin] - L_ref[fin]) - lse_rel * np.abs(L_ref[fin])) if fin.any() else 0.0
    assert err <= tol, f"{what}: O rel err {err:.3e} > {tol}"
    assert lerr <= 1e-2, f"{what}: LSE err {lerr:.3e} (beyond {lse_rel:g} * |LSE_ref|)"
    return err, lerr


def parity(w, mode, oracle_mod, tokens=None, lse_rel=0.0, **kw):
    O, L, _ = run_gpu(w, mode, **kw)
    O_ref, L_ref = oracle_mod.attention(w, tokens=tokens)
    if tokens is not None:
        O, L = O[tokens], L[tokens]
    return check_against(w, O, L, O_ref, L_ref, f"{w.name} mode={mode}", lse_rel)


MODES = ["prefill", "decode", "forward"]


# --------------------------------------------------------------------------- small cases
@pytest.mark.parametrize("mode", MODES)
def test_config1_tiny(oracle_mod, mode):
    parity(synth.config(1), mode, oracle_mod)


@pytest.mark.parametrize("H", [1, 8, 16, 17, 32, 48, 64, 65, 100, 128])
@pytest.mark.parametrize("fmt", [FMT_BF16, FMT_FP8])
def test_heads_envelope(oracle_mod, H, fmt):
    w = synth.small_case(100 + H, T=3, H=H, topk=256, ctx=1024, fmt=fmt, sink=(H % 2 == 0), mask_p=0.05)
    for mode in ("prefill", "decode"):
        parity(w, mode, oracle_mod)


@pytest.mark.parametrize("topk", [1, 63, 64, 100, 128, 130, 320, 500])
def test_ragged_topk(oracle_mod, topk):
    w = synth.small_case(200 + topk, T=5, H=32, topk=topk, ctx=2048, fmt=FMT_FP8, sink=True, mask_p=0.05)
    for mode in ("prefill", "decode"):
        parity(w, mode, oracle_mod)


def growing_scores_case(fmt, T=64, H=40, topk=1024, ctx=2048, seed=410):
    """Scores that climb along each token's ascending index list: the cache row at position i
    is i * u (+ noise) for one unit direction u, and head h's query is alpha_h * u with alpha_h
    from -0.5 to 1.2. Per 128-entry tile (~256 positions) a head's maximum then rises by
    alpha_h * 256 / 24 * log2(e) ~ 15 alpha_h in base 2: past the 2^8 lazy-rescale threshold on
    every tile for alpha_h > 0.52, every other tile for smaller positive alpha_h, never after the
    first tile for negative alpha_h. So the running maxima move mid-item at rates that differ
    by head, in whole items (prefill) and in split ranges that start mid-item (decode)."""
    w = synth.small_case(seed, T=T, H=H, topk=topk, ctx=ctx, fmt=fmt, sink=True)
    s = w.main
    assert s.page_stride == 64 * s.row_stride and w.num_seqs == 1
    rng = np.random.default_rng(seed + 1)
    u = rng.standard_normal(576)
    u /= np.linalg.norm(u)
    pos = np.arange(ctx)
    x = pos[:, None] * u[None, :] + 0.05 * rng.standard_normal((ctx, 576))
    rows = synth.encode_rows(x.astype(np.float32), fmt)
    cache = s.cache.copy().reshape(s.num_pages, 64, s.row_stride)
    cache[s.block_table[0, pos // 64], pos % 64, :rows.shape[1]] = rows
    idx = np.sort(synth.distinct_indices(rng, np.full(T, ctx - 1), topk), axis=1)
    idx = synth.mask_random(rng, idx, 0.05)
    alpha = np.linspace(-0.5, 1.2, H)
    q = alpha[None, :, None] * u[None, None, :] + 0.02 * rng.standard_normal((T, H, 576))
    main = synth.replace(s, cache=cache.reshape(-1), indices=np.ascontiguousarray(idx, dtype=np.int32))
    return synth.replace(w, q=synth.f32_to_bf16_bits(q.astype(np.float32)), main=main,
                         name=f"growing scores fmt={fmt} T={T} H={H} topk={topk}")


@pytest.mark.parametrize("fmt", [FMT_BF16, FMT_FP8])
def test_running_max_moves_mid_item(oracle_mod, fmt):
    # Scores reach ~100 here. With an FP8 cache the kernels multiply the dequantised K rounded
    # to bf16 (2^-9 relative per element) while the oracle keeps it exact. The products are
    # coherent (q and K share one direction), so a score moves by about
    # 2^-9/sqrt(3) * sqrt(sum u^4)/sum u^2 ~ 6e-5 of itself (RMS), and the LSE with it. This case
    # allows 1e-2 + 2^-12 * |LSE_ref| (4x that RMS); a bf16 cache has no such rounding.
    w = growing_scores_case(fmt)
    for mode in ("prefill", "decode"):
        parity(w, mode, oracle_mod, lse_rel=2.0**-12 if fmt == FMT_FP8 else 0.0)


def test_topk_length(oracle_mod):
    w = synth.small_case(300, T=9, H=16, topk=384, ctx=1024, topk_length=True, sink=True)
    for mode in ("prefill", "decode"):
        parity(w, mode, oracle_mod)


@pytest.mark.parametrize("xfmt", [FMT_BF16, FMT_FP8])
def test_dual_cache(oracle_mod, xfmt):
    w = synth.small_case(310 + xfmt, T=4, H=64, topk=512, ctx=4096, fmt=FMT_FP8, sink=True, mask_p=0.05,
                         extra_topk=128, extra_fmt=xfmt)
    for mode in MODES:
        parity(w, mode, oracle_mod)


def test_many_sequences_causal(oracle_mod):
    w = synth.small_case(320, T=12, H=24, topk=192, ctx=700, num_seqs=4, causal=True, sink=True)
    for mode in ("prefill", "decode"):
        parity(w, mode, oracle_mod)


def test_strided_views(oracle_mod):
    w = synth.small_case(330, T=4, H=20, topk=256, ctx=1024, fmt=FMT_FP8, row_pad=48, page_pad=512, idx_pad=13,
                         sink=True)
    for mode in ("prefill", "decode"):
        parity(w, mode, oracle_mod, out_pad=64, lse_pad=5, q_pad=(3, 64))


def test_empty_and_out_of_range(oracle_mod):
    w = synth.small_case(340, T=6, H=16, topk=192, ctx=512, sink=True)
    idx = w.main.indices.copy()
    idx[1] = -1                      # fully masked row
    idx[2, :100] = 10 ** 6           # beyond seq_len
    idx[3, ::2] = -3
    w = synth.with_indices(w, idx)
    w = synth.replace(w, token_seq=np.array([0, 0, 0, 0, 7, -1], dtype=np.int32))  # tokens 4, 5: bad sequence
    for mode in MODES:
        O, L, _ = run_gpu(w, mode)
        O_ref, L_ref = oracle_mod.attention(w)
        check_against(w, O, L, O_ref, L_ref, mode)
        assert np.all(O[[1, 4, 5]] == 0) and np.all(np.isneginf(L[[1, 4, 5]]))


def test_zero_tokens_launches_nothing(oracle_mod):
    w = synth.small_case(350, T=1, H=4, topk=64, ctx=128)
    dp = binding.DeviceProblem(w)
    dp.call.p.T = 0
    for mode in MODES:
        assert dp.run(mode) == binding.SMLA_OK
    torch.cuda.synchronize()
    assert torch.isnan(dp.out.float()).all()  # untouched


def test_workspace_too_small_is_rejected():
    w = synth.small_case(351, T=2, H=64, topk=1024, ctx=2048, fmt=FMT_FP8)
    dp = binding.DeviceProblem(w)
    need = binding.workspace_size(dp.call)
    assert need > 0
    small = torch.empty(need // 2, dtype=torch.uint8, device="cuda")
    dp.call.set_workspace(small)
    assert binding.decode(dp.call, check=False) == binding.SMLA_ERR_WORKSPACE


# --------------------------------------------------------------------------- exact mask handling
def test_mask_variants_bit_identical_on_gpu():
    w = synth.small_case(360, T=5, H=32, topk=320, ctx=1024, fmt=FMT_FP8, mask_p=0.3, sink=True)
    base = run_gpu(w, "prefill")
    idx = w.main.indices.copy()
    neg = idx < 0
    for fill in (-7, 1024, 10 ** 7):
        v = idx.copy()
        v[neg] = fill
        O, L, _ = run_gpu(synth.with_indices(w, v), "prefill")
        assert np.array_equal(O, base[0]) and np.array_equal(L, base[1]), fill


def test_unreferenced_rows_never_read_on_gpu():
    w = synth.small_case(361, T=4, H=16, topk=256, ctx=2048, fmt=FMT_BF16, mask_p=0.2, spare_pages=3)
    O0, L0, _ = run_gpu(w, "decode")
    s = w.main
    keep = np.zeros(s.num_pages * 64, dtype=bool)
    for t in range(w.T):
        for i in s.indices[t, :s.topk]:
            if 0 <= i < 2048:
                keep[int(s.block_table[0, i // 64]) * 64 + int(i % 64)] = True
    cache = s.cache.copy().reshape(s.num_pages, s.page_stride)
    rows = cache[:, :64 * s.row_stride].reshape(s.num_pages * 64, s.row_stride)
    rows[~keep] = 0xFF  # NaN in bf16
    w2 = synth.replace(w, main=synth.replace(s, cache=cache.reshape(-1)))
    O1, L1, _ = run_gpu(w2, "decode")
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)
    assert np.isfinite(O1).all()


def test_decode_and_prefill_agree(oracle_mod):
    w = synth.small_case(370, T=2, H=64, topk=2048, ctx=8192, fmt=FMT_FP8, sink=True, mask_p=0.05)
    Op, Lp, _ = run_gpu(w, "prefill")
    Od, Ld, _ = run_gpu(w, "decode")
    assert np.max(np.abs(Op - Od)) <= 2e-2 * np.max(np.abs(Op))
    assert np.max(np.abs(Lp - Ld)) <= 1e-3


def test_head_independence_on_gpu():
    w = synth.small_case(380, T=3, H=32, topk=256, ctx=1024, sink=True)
    O1, L1, _ = run_gpu(w, "prefill")
    rng = np.random.default_rng(5)
    q2 = np.concatenate([w.q, synth.make_q(rng, w.T, w.H)], axis=1)
    s2 = np.concatenate([w.sink, rng.standard_normal(w.H).astype(np.float32)])
    O2, L2, _ = run_gpu(synth.replace(w, H=64, q=q2, sink=s2), "prefill")
    assert np.max(np.abs(O2[:, :32] - O1)) <= 1e-2 * np.max(np.abs(O1))
    assert np.max(np.abs(L2[:, :32] - L1)) <= 1e-4


# --------------------------------------------------------------------------- full-size configs
def _sample(T, n, seed):
    """n distinct tokens of T (seeded), always including the first and the last."""
    rng = np.random.default_rng(seed)
    if n >= T:
        return np.arange(T)
    mid = rng.choice(np.arange(1, T - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, T - 1], mid]))


@pytest.fixture(scope="module")
def config2():
    return synth.config(2)


@pytest.mark.parametrize("mode", MODES)
def test_config2_decode_full(oracle_mod, config2, mode):
    # every token of the batch
    parity(config2, mode, oracle_mod, tokens=_sample(config2.T, config2.T, 2))


def test_config3_prefill_full(oracle_mod):
    # every token (the threaded oracle takes a few seconds for the 146 GFLOP)
    w = synth.config(3)
    parity(w, "forward", oracle_mod, tokens=_sample(w.T, w.T, 3))


def test_config4_large_prefill_full(oracle_mod):
    # 1024 of 8192 tokens (the whole workload is ~5 TFLOP for the fp64 oracle), first and last
    # included
    w = synth.config(4)
    parity(w, "forward", oracle_mod, tokens=_sample(w.T, 1024, 4))


def test_sweep_points(oracle_mod):
    pool = synth.SweepPool()
    for (H, topk, T, sink) in [(1, 64, 1, False), (8, 1024, 16, True), (16, 128, 65, True), (32, 512, 64, False),
                               (64, 2048, 1, True), (128, 256, 16, True), (128, 2048, 65, False)]:
        w = pool.point(H, topk, T, sink)
        tokens = _sample(T, 6, H + topk)
        for mode in ("prefill", "decode", "forward"):
            parity(w, mode, oracle_mod, tokens=tokens)
