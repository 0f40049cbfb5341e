"""GPU cache writer (smla_quantize_kv) against the oracle's cache writer: bit-exact.

Both sides take every rounding decision in fp32 (scale = amax / 448, quotient x / scale)
and round to E4M3FN / bf16 to nearest even, so the cache bytes must be identical. Rows are
written at physical slots of a paged cache with padded rows and pages; slots that are
negative or past the cache are skipped and every byte the writer must not touch keeps its
sentinel value.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from sparse_top_mla_gb300 import binding, synth  # noqa: E402
from sparse_top_mla_gb300 import build as smla_build  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smla_build.build()
    binding.load()
    yield
    assert binding.device_error() == 0


def _inputs(seed, n, in_f32):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 576)).astype(np.float32)
    x *= rng.uniform(1e-3, 1e3, size=(n, 1)).astype(np.float32)  # scales over six decades
    x[::97, :128] = 0.0                                          # all-zero blocks
    if in_f32:
        return x, x
    bits = synth.f32_to_bf16_bits(x)
    return bits, bits


def _edge_inputs(seed, n, in_f32):
    """Rows built to stress the quotient x / scale: negative zeros inside live blocks, values
    at the block maximum and at exact multiples of the block scale (ties after scaling), tiny
    values down to the bf16 subnormals beside large ones, and exponents over 60 decades."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 576)).astype(np.float32)
    x *= (10.0 ** rng.uniform(-30, 30, size=(n, 1))).astype(np.float32)
    x[::3, 5:40] = -0.0
    x[1::3, :128] *= np.float32(1e-36)
    x[1::3, 7] = np.float32(9.2e-41)                          # a bf16 subnormal
    x[2::3, 130:250] = np.float32(-0.0)
    amax = np.abs(x[:, 256:384]).max(axis=1, keepdims=True)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    k = rng.integers(-448, 449, size=(n, 128)).astype(np.float32)
    x[:, 256:384] = (k * scale).astype(np.float32)            # multiples of the block scale
    x[:, 384] = amax[:, 0]                                    # the maximum itself
    x[:, 385] = -amax[:, 0]
    if in_f32:
        return x, x
    bits = synth.f32_to_bf16_bits(x)
    return bits, bits


def _write(oracle_mod, seed, n, fmt, in_f32, num_pages, row_pad=0, page_pad=0, kv_pad=0, edge=False):
    host, oracle_in = (_edge_inputs if edge else _inputs)(seed, n, in_f32)
    row_bytes = 1152 if fmt == 0 else 656
    row_stride = row_bytes + row_pad
    page_stride = 64 * row_stride + page_pad
    rng = np.random.default_rng(seed + 1)
    slots = rng.choice(num_pages * 64, size=n, replace=False).astype(np.int64)
    slots[::13] = -1                          # skipped
    slots[5::17] = num_pages * 64 + 3         # past the cache: skipped
    dev = torch.device("cuda")
    width = 576 + kv_pad
    if in_f32:
        kv_full = torch.zeros((n, width), dtype=torch.float32, device=dev)
        kv_full[:, :576] = torch.from_numpy(host).to(dev)
    else:
        kv_full = torch.zeros((n, width), dtype=torch.int16, device=dev)
        kv_full[:, :576] = torch.from_numpy(host.view(np.int16)).to(dev)
        kv_full = kv_full.view(torch.bfloat16)
    kv = kv_full[:, :576]
    cache = torch.full((num_pages * page_stride,), 0xA5, dtype=torch.uint8, device=dev)
    binding.quantize_kv(kv, torch.from_numpy(slots).to(dev), cache, fmt, row_stride, page_stride, num_pages)
    torch.cuda.synchronize()
    got = cache.cpu().numpy()
    ref_rows = oracle_mod.pack_rows(oracle_in, fmt)
    expect = np.full_like(got, 0xA5)
    for i, s in enumerate(slots):
        if 0 <= s < num_pages * 64:
            off = (s // 64) * page_stride + (s % 64) * row_stride
            expect[off:off + row_bytes] = ref_rows[i]
    return got, expect


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("in_f32", [False, True])
def test_quantize_kv_bit_exact_small(oracle_mod, fmt, in_f32):
    got, expect = _write(oracle_mod, 700 + 2 * fmt + in_f32, 1000, fmt, in_f32, num_pages=40, row_pad=32,
                         page_pad=48, kv_pad=8 if in_f32 else 16)
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("in_f32", [False, True])
def test_quantize_kv_bit_exact_edge_values(oracle_mod, in_f32):
    got, expect = _write(oracle_mod, 800 + in_f32, 3000, 1, in_f32, num_pages=60, edge=True)
    assert np.array_equal(got, expect)


def test_quantize_kv_large_prefill_cache_size(oracle_mod):
    # the large-prefill main cache: 65536 tokens in 1024 pages of FP8 rows, written in full
    got, expect = _write(oracle_mod, 710, 65536, 1, False, num_pages=1024)
    assert np.array_equal(got, expect)


def test_quantize_kv_decode_cache_size(oracle_mod):
    # the decode cache: 16384 pages (1,048,576 slots); 65536 rows scattered over all of it
    got, expect = _write(oracle_mod, 711, 65536, 1, True, num_pages=16384)
    assert np.array_equal(got, expect)


def test_quantize_kv_rejects_bad_arguments():
    dev = torch.device("cuda")
    kv = torch.zeros((4, 576), dtype=torch.bfloat16, device=dev)
    slots = torch.arange(4, dtype=torch.int64, device=dev)
    cache = torch.zeros(64 * 656, dtype=torch.uint8, device=dev)
    assert binding.quantize_kv(kv, slots, cache, 2, 656, 64 * 656, 1, check=False) == binding.SMLA_ERR_UNSUPPORTED
    assert binding.quantize_kv(kv, slots, cache, 1, 650, 64 * 656, 1, check=False) == binding.SMLA_ERR_INVALID
    assert binding.quantize_kv(kv, slots, cache, 1, 656, 64 * 656, 0, check=False) == binding.SMLA_ERR_INVALID
    assert binding.quantize_kv(kv[:0], slots, cache, 1, 656, 64 * 656, 1, check=False) == binding.SMLA_OK


def test_written_cache_feeds_attention(oracle_mod):
    # rows written by the device writer, read back by the attention kernel, against the oracle
    w = synth.small_case(720, T=3, H=16, topk=256, ctx=1024, fmt=synth.FMT_FP8, sink=True)
    rng = np.random.default_rng(721)
    x = rng.standard_normal((w.main.num_pages * 64, 576)).astype(np.float32)
    rows = oracle_mod.pack_rows(x, 1)
    host_cache = w.main.cache.copy().reshape(w.main.num_pages, w.main.page_stride)
    for s in range(w.main.num_pages * 64):
        host_cache[s // 64, (s % 64) * w.main.row_stride:(s % 64) * w.main.row_stride + 656] = rows[s]
    w2 = synth.replace(w, main=synth.replace(w.main, cache=host_cache.reshape(-1)))
    dp = binding.DeviceProblem(w2)
    dp.main.cache.fill_(0)
    kv = torch.from_numpy(x).cuda()
    slots = torch.arange(x.shape[0], dtype=torch.int64, device="cuda")
    binding.quantize_kv(kv, slots, dp.main.cache, 1, w.main.row_stride, w.main.page_stride, w.main.num_pages)
    dp.run("prefill")
    O, L = dp.results()
    O_ref, L_ref = oracle_mod.attention(w2)
    assert np.max(np.abs(O - O_ref)) <= 4e-2 * np.max(np.abs(O_ref))
    assert np.max(np.abs(L - L_ref)) <= 1e-2
