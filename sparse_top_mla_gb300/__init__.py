"""sparse_top_mla_gb300 — sparse top-k MLA attention on one GB300 (sm_103a).

The compute lives in libsmla.so (hand-written CUDA, C ABI in include/smla.h); this
package only builds it (``build``), marshals arguments into it (``binding``) and draws
seeded synthetic inputs (``synth``).
"""
from . import binding  # noqa: F401
from .binding import (Call, DeviceProblem, DeviceSet, SmlaError, decode, decode_max_tokens,  # noqa: F401
                      device_error, forward, load, load_crossover, prefill, set_crossover,
                      set_timing_events, supported, workspace_size)
