"""Host-only tests of the C-ABI boundary: the library builds, loads, exports every symbol the
header declares, and validates arguments before any launch (fake device pointers are fine
here because every case returns before touching device memory)."""
import ctypes
import json
import os
import re

import pytest

from sparse_top_mla_gb300 import binding
from sparse_top_mla_gb300 import build as smla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "smla.h")


@pytest.fixture(scope="module")
def lib():
    smla_build.build()
    return binding.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(smla_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    declared = header_functions()
    assert declared, "no declarations parsed"
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(binding.EXPORTS)


def test_struct_sizes_match_binding(lib):
    assert lib.smla_struct_size(0) == ctypes.sizeof(binding.Params)
    assert lib.smla_struct_size(1) == ctypes.sizeof(binding.KvSet)
    assert lib.smla_version() >> 16 == 1


FAKE = 1 << 40  # 16-byte aligned fake device address; never dereferenced in these tests


def fake_params(T=4, H=16, topk=128, fmt=0, page_size=64):
    rs = 1152 if fmt == 0 else 656
    main = binding.KvSet(FAKE, fmt, rs, 64 * rs, page_size, 4, FAKE, 4, FAKE, FAKE, topk, topk, None)
    return binding.Params(T, H, 576, 512, 1, FAKE, H * 576, 576, FAKE, main, None, None, 0.04, FAKE, H * 512,
                          512, FAKE, H, None, 0)


def why(lib, p):
    buf = ctypes.create_string_buffer(512)
    ok = lib.smla_supported(ctypes.byref(p), buf, 512)
    return ok, buf.value.decode()


def test_supported_accepts_the_envelope(lib):
    for H in (1, 7, 16, 33, 64, 80, 128):
        for topk in (1, 64, 100, 2048):
            for fmt in (0, 1):
                ok, msg = why(lib, fake_params(H=H, topk=topk, fmt=fmt))
                assert ok == 1, (H, topk, fmt, msg)


@pytest.mark.parametrize("mutate,field,status", [
    (lambda p: setattr(p, "H", 0), "H=0", binding.SMLA_ERR_UNSUPPORTED),
    (lambda p: setattr(p, "H", 129), "H=129", binding.SMLA_ERR_UNSUPPORTED),
    (lambda p: setattr(p, "d_qk", 1088), "d_qk=1088", binding.SMLA_ERR_UNSUPPORTED),
    (lambda p: setattr(p.main, "page_size", 32), "page_size=32", binding.SMLA_ERR_UNSUPPORTED),
    (lambda p: setattr(p.main, "format", 7), "format=7", binding.SMLA_ERR_UNSUPPORTED),
    (lambda p: setattr(p.main, "topk", 0), "topk=0", binding.SMLA_ERR_UNSUPPORTED),
    (lambda p: setattr(p.main, "idx_stride", 64), "idx_stride=64", binding.SMLA_ERR_INVALID),
    (lambda p: setattr(p.main, "row_stride_bytes", 1000), "row_stride_bytes=1000", binding.SMLA_ERR_INVALID),
    (lambda p: setattr(p.main, "page_stride_bytes", 1152 * 63), "page_stride_bytes", binding.SMLA_ERR_INVALID),
    (lambda p: setattr(p.main, "cache", FAKE + 8), "16-byte aligned", binding.SMLA_ERR_INVALID),
    (lambda p: setattr(p, "q_stride_h", 577), "q must be", binding.SMLA_ERR_INVALID),
    (lambda p: setattr(p, "out", None), "non-NULL", binding.SMLA_ERR_INVALID),
    (lambda p: setattr(p, "lse_stride_t", 3), "lse_stride_t=3", binding.SMLA_ERR_INVALID),
    (lambda p: setattr(p, "sm_scale", float("nan")), "sm_scale", binding.SMLA_ERR_INVALID),
])
def test_rejections_name_the_field(lib, mutate, field, status):
    p = fake_params()
    mutate(p)
    ok, msg = why(lib, p)
    assert ok == 0 and field in msg, msg
    # every entry point returns the same status before launching anything
    for fn in (lib.smla_prefill, lib.smla_decode, lib.smla_forward):
        assert fn(ctypes.byref(p), None) == status


def test_extra_set_is_validated(lib):
    p = fake_params()
    extra = binding.KvSet(FAKE, 0, 1152, 64 * 1152, 16, 4, FAKE, 4, FAKE, FAKE, 128, 128, None)
    p.extra = ctypes.addressof(extra)
    ok, msg = why(lib, p)
    assert ok == 0 and "extra.page_size=16" in msg


def test_zero_tokens_is_a_no_op(lib):
    p = fake_params(T=0)
    for fn in (lib.smla_prefill, lib.smla_decode, lib.smla_forward):
        assert fn(ctypes.byref(p), None) == binding.SMLA_OK
    assert lib.smla_workspace_size(ctypes.byref(p)) == 0


def test_null_params(lib):
    assert lib.smla_supported(None, None, 0) == 0
    assert lib.smla_prefill(None, None) == binding.SMLA_ERR_INVALID


def test_status_strings(lib):
    for s in range(6):
        assert lib.smla_status_string(s).decode().startswith("SMLA_")
    assert lib.smla_status_string(99) == b"unknown smla_status"


def test_crossover_table(lib, tmp_path):
    binding.set_crossover([(64, 2048, 1, 24), (128, 2048, 1, 8), (8, 1024, 1, 64)])
    assert binding.decode_max_tokens(64, 2048, 1) == 24
    assert binding.decode_max_tokens(100, 2048, 1) == 8     # nearest in log2 H
    assert binding.decode_max_tokens(8, 900, 1) == 64
    path = tmp_path / "crossover.json"
    path.write_text(json.dumps({"version": 1, "entries": [[32, 512, 0, 17], [32, 512, 1, 9]]}))
    assert binding.load_crossover(str(path)) == binding.SMLA_OK
    assert binding.decode_max_tokens(32, 512, 0) == 17
    assert binding.decode_max_tokens(32, 512, 1) == 9
    path.write_text(json.dumps({"version": 2, "entries": [[32, 512, 0, 5]]}))
    assert binding.load_crossover(str(path)) == binding.SMLA_ERR_UNSUPPORTED
    assert binding.decode_max_tokens(32, 512, 0) >= 1  # table cleared -> built-in default
    with pytest.raises(binding.SmlaError):
        binding.set_crossover([(0, 512, 0, 5)])
    binding.set_crossover([])
    if os.path.exists(binding.CROSSOVER_TABLE):  # put the packaged calibration back
        assert binding.load_crossover(binding.CROSSOVER_TABLE) == binding.SMLA_OK


def test_timing_hook_pairs(lib):
    assert lib.smla_set_timing_events(ctypes.c_void_p(FAKE), None) == binding.SMLA_ERR_INVALID
    assert lib.smla_set_timing_events(None, None) == binding.SMLA_OK


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        binding.load(str(tmp_path / "nope.so"))


@pytest.mark.parametrize("kw", [dict(T=1, H=1, topk=64, ctx=128), dict(T=3, H=20, topk=256, ctx=1024, row_pad=48,
                                page_pad=512, idx_pad=13, sink=True), dict(T=4, H=64, topk=512, ctx=4096, fmt=1,
                                extra_topk=128), dict(T=9, H=16, topk=384, ctx=1024, topk_length=True)])
def test_binding_marshals_supported_calls(lib, kw):
    """The binding's structs (built from CPU tensors here) pass the library's validation."""
    from sparse_top_mla_gb300 import synth
    w = synth.small_case(1, **kw)
    dp = binding.DeviceProblem(w, device="cpu", out_pad=64, lse_pad=3, q_pad=(2, 8))
    ok, msg = binding.supported(dp.call)
    assert ok, msg
    assert dp.call.p.main.idx_stride == w.main.indices.shape[1]
    if w.H > 1:
        assert dp.call.p.q_stride_h == 576 + 8 and dp.call.p.out_stride_h == 512 + 64


def test_binding_config1_supported(lib):
    from sparse_top_mla_gb300 import synth
    dp = binding.DeviceProblem(synth.config(1), device="cpu")
    assert binding.supported(dp.call) == (True, "")
    assert dp.call.p.main.bt_stride == 4
