"""Independent numpy helpers for pinning the oracle (test code only).

Written separately from the C++ oracle: the cache decoders below follow the format
definitions (bfloat16 = top half of an IEEE float32; OCP E4M3FN from its field
formula) and the dense reference is textbook multi-query softmax attention.
"""
import numpy as np

from sparse_top_mla_gb300.synth import D_QK, D_V, FMT_BF16, PAGE


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def e4m3_table() -> np.ndarray:
    """Value of every E4M3FN code from the format's definition: (-1)^s * 2^(e-7) * (1 + m/8)
    for e > 0, (-1)^s * 2^-6 * (m/8) for e = 0, NaN for e = 15, m = 7."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            v = float("nan")
        elif e == 0:
            v = 2.0 ** -6 * (m / 8.0)
        else:
            v = 2.0 ** (e - 7) * (1.0 + m / 8.0)
        vals[code] = -v if s else v
    return vals


_E4M3 = e4m3_table()


def decode_row(s, page: int, r: int) -> np.ndarray:
    off = page * s.page_stride + r * s.row_stride
    if s.fmt == FMT_BF16:
        return bf16_to_f64(s.cache[off:off + 2 * D_QK].view(np.uint16))
    raw = s.cache[off:off + 656]
    scale = raw[512:528].view(np.float32).astype(np.float64)
    lat = _E4M3[raw[:512]] * np.repeat(scale, 128)
    rope = bf16_to_f64(raw[528:656].view(np.uint16))
    return np.concatenate([lat, rope])


def decode_logical(s, seq: int, pos: int) -> np.ndarray:
    return decode_row(s, int(s.block_table[seq, pos // PAGE]), pos % PAGE)


def dense_mqa(q: np.ndarray, K: np.ndarray, sm_scale: float, sink=None):
    """Dense multi-query attention: q [H, 576], K [n, 576] (V = K[:, :512]).
    Returns O [H, 512], LSE [H] (natural log, sink excluded)."""
    S = (q @ K.T) * sm_scale
    m = S.max(axis=1, keepdims=True)
    if sink is not None:
        m = np.maximum(m, np.asarray(sink, dtype=np.float64)[:, None])
    E = np.exp(S - m)
    Z = E.sum(axis=1)
    D = Z + (np.exp(np.asarray(sink, dtype=np.float64) - m[:, 0]) if sink is not None else 0.0)
    O = (E @ K[:, :D_V]) / D[:, None]
    return O, m[:, 0] + np.log(Z)
