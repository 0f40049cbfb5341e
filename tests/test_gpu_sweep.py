"""GPU parity over the whole envelope sweep: H in {1,8,16,32,64,128} x topk in
{64,...,2048} x T in {1,16,64,65,256,1024} x sink off/on (432 points) over one
16384-token FP8 paged context (64 sequences, random distinct indices, 5% masked). Both
schedules (prefill and split-K decode) run every point through the C ABI; the fp64 oracle
checks up to two sampled tokens per point with the stated tolerances (4e-2 * max|O_ref| for
FP8 caches, 1e-2 on LSE, exact O = 0 / LSE = -inf for empty sets)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from sparse_top_mla_gb300 import binding, synth  # noqa: E402
from sparse_top_mla_gb300 import build as smla_build  # noqa: E402

from .test_gpu_parity import check_against  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smla_build.build()
    binding.load()
    yield
    assert binding.device_error() == 0


def test_sweep_full_grid(oracle_mod):
    pool = synth.SweepPool()
    base = None
    done = 0
    for H in synth.SWEEP_H:
        for topk in synth.SWEEP_TOPK:
            for T in synth.SWEEP_T:
                for sink in (False, True):
                    w = pool.point(H, topk, T, sink)
                    dp = binding.DeviceProblem(w, share_caches_with=base)
                    base = base or dp
                    rng = np.random.default_rng(H * 100003 + topk * 101 + T * 7 + int(sink))
                    tokens = np.sort(rng.choice(T, size=min(2, T), replace=False))
                    O_ref, L_ref = oracle_mod.attention(w, tokens=tokens)
                    sel = torch.from_numpy(tokens).to(dp.out.device)
                    for mode in ("prefill", "decode"):
                        dp.run(mode)
                        torch.cuda.synchronize()
                        O = dp.out.index_select(0, sel).float().cpu().double().numpy()
                        L = dp.lse.index_select(0, sel).cpu().double().numpy()
                        check_against(w, O, L, O_ref, L_ref, f"{w.name} mode={mode}")
                    done += 1
    assert done == len(synth.SWEEP_H) * len(synth.SWEEP_TOPK) * len(synth.SWEEP_T) * 2
