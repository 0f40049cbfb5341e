"""smla_decode_static: split-K decode for callers that cannot allocate device memory.

Such callers (a plugin behind a fixed C interface that hands over only the problem tensors,
or a runtime whose device memory all belongs to its own pool) cannot pass a workspace. The
entry point keeps its split-K scratch in a fixed 32 MiB array inside the library instead.
These tests call it through the C ABI and compare it with smla_decode, which uses a
caller-provided workspace, on two calls in a row (the second call reuses the array the
first one left behind). The file is named so that pytest collects it last.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from sparse_top_mla_gb300 import binding, synth  # noqa: E402
from sparse_top_mla_gb300 import build as smla_build  # noqa: E402

pytestmark = pytest.mark.gpu

TOL_FP8 = 4e-2  # the parity tolerance for FP8 caches, relative to max|O|
SCRATCH_LIMIT = 32 << 20


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smla_build.build()
    binding.load()


def _outputs(dp):
    torch.cuda.synchronize()
    return dp.out.float().cpu().numpy().copy(), dp.lse.cpu().numpy().copy()


@pytest.mark.parametrize("seed,T,H,topk", [(901, 4, 64, 2048), (902, 7, 24, 1024)])
def test_static_scratch_matches_workspace_decode(seed, T, H, topk):
    w = synth.small_case(seed, T=T, H=H, topk=topk, ctx=8192, fmt=synth.FMT_FP8, sink=True, mask_p=0.05,
                         extra_topk=128)
    ref = binding.DeviceProblem(w)
    need = binding.workspace_size(ref.call)
    assert 0 < need <= SCRATCH_LIMIT  # the case really uses split-K scratch
    ref.run("decode")
    O_ref, L_ref = _outputs(ref)
    assert binding.device_error() == 0

    dp = binding.DeviceProblem(w)
    assert dp.workspace is None and dp.call.p.workspace is None
    scale = np.max(np.abs(O_ref))
    for call in range(2):
        dp.out.fill_(float("nan"))
        dp.lse.fill_(float("nan"))
        assert binding.decode_static(dp.call) == binding.SMLA_OK
        O, L = _outputs(dp)
        assert binding.device_error() == 0
        assert np.isfinite(O).all(), call
        assert np.max(np.abs(O - O_ref)) <= TOL_FP8 * scale, call
        fin = np.isfinite(L_ref)
        assert np.array_equal(fin, np.isfinite(L)), call
        assert np.max(np.abs(L[fin] - L_ref[fin])) <= 1e-2, call
        # the same plan and kernels run in both entry points: the bytes are identical
        assert np.array_equal(O, O_ref) and np.array_equal(L, L_ref), call


def test_static_scratch_against_the_oracle(oracle_mod):
    w = synth.small_case(903, T=5, H=32, topk=1536, ctx=8192, fmt=synth.FMT_FP8, sink=True, mask_p=0.05)
    dp = binding.DeviceProblem(w)
    assert 0 < binding.workspace_size(dp.call) <= SCRATCH_LIMIT
    for call in range(2):
        assert binding.decode_static(dp.call) == binding.SMLA_OK
        O, L = _outputs(dp)
        O_ref, L_ref = oracle_mod.attention(w)
        assert np.max(np.abs(O - O_ref)) <= TOL_FP8 * np.max(np.abs(O_ref)), call
        assert np.max(np.abs(L - L_ref)) <= 1e-2, call


def test_static_scratch_rejects_problems_beyond_its_size():
    # T=1024 tokens of 128 heads on the split-K schedule need far more than 32 MiB of partials;
    # the tensors are real and full-sized, so nothing could be read out of bounds in any case
    w = synth.small_case(905, T=1024, H=128, topk=2048, ctx=4096, fmt=synth.FMT_FP8)
    dp = binding.DeviceProblem(w)
    assert binding.workspace_size(dp.call) > SCRATCH_LIMIT
    dp.out.fill_(float("nan"))
    assert binding.decode_static(dp.call, check=False) == binding.SMLA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(dp.out.float()).all()  # nothing was launched


def test_static_scratch_validates_like_decode():
    w = synth.small_case(904, T=2, H=8, topk=256, ctx=1024)
    dp = binding.DeviceProblem(w)
    dp.call.p.main.page_size = 32
    assert binding.decode_static(dp.call, check=False) == binding.SMLA_ERR_UNSUPPORTED
