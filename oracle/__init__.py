"""CPU oracle of the MoE dispatch / combine path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of ``bench.py`` may import
this package.  It wraps ``ep_oracle.c`` (plain single-threaded C, built with gcc
``-O2 -ffp-contract=off``) through ctypes and numpy; it shares no code with the CUDA library.

Every function takes and returns numpy arrays; bf16 tensors are ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libep_oracle.so")

OVERFLOW = 1
BAD_EXPERT = 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no contraction of multiply-adds)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_long


def _declare(L):
    L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_double.restype = ctypes.c_double
    L.oracle_bf16_from_double.argtypes = [ctypes.c_double]
    L.oracle_bf16_from_double.restype = ctypes.c_uint16
    L.oracle_e2m1_encode.argtypes = [ctypes.c_float]
    L.oracle_e2m1_encode.restype = ctypes.c_uint8
    L.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e2m1_decode.restype = ctypes.c_float
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_decode.restype = ctypes.c_float
    L.oracle_layout.argtypes = [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]
    L.oracle_layout.restype = _I
    L.oracle_rows_max.argtypes = [_I, _I, _I, _I, _I, _L]
    L.oracle_rows_max.restype = _L
    L.oracle_layout_padded.argtypes = [_P, _I, _I, _I, _I, _I, _I, _I, _L, _P, _P, _P, _P, _P]
    L.oracle_layout_padded.restype = _I
    L.oracle_fill_padding_rows.argtypes = [_P, _L, _L, _I, _P, _L, _P]
    L.oracle_fill_padding_rows.restype = None
    L.oracle_fp8_quantize_row.argtypes = [_P, _I, _P, _P]
    L.oracle_fp8_quantize_row.restype = None
    L.oracle_dispatch_fp8.argtypes = [_P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P]
    L.oracle_dispatch_fp8.restype = None
    L.oracle_routing_map_to_topk.argtypes = [_P, _P, _I, _I, _I, _P, _P]
    L.oracle_routing_map_to_topk.restype = None
    L.oracle_indices_to_multihot.argtypes = [_P, _P, _I, _I, _I, _P, _P]
    L.oracle_indices_to_multihot.restype = None
    L.oracle_nvfp4_quantize_row.argtypes = [_P, _I, _P, _P, _P]
    L.oracle_nvfp4_quantize_row.restype = None
    L.oracle_dispatch_nvfp4.argtypes = [_P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P]
    L.oracle_dispatch_nvfp4.restype = None
    L.oracle_dispatch_bf16.argtypes = [_P, _I, _I, _I, _I, _I, _P, _P, _I, _P]
    L.oracle_dispatch_bf16.restype = None
    L.oracle_combine.argtypes = [_P, _P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P]
    L.oracle_combine.restype = None
    L.oracle_combine_bwd.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P]
    L.oracle_combine_bwd.restype = None
    L.oracle_tiny_expert_outputs.argtypes = [_P, _P, _P, _P, _L, _I, _P]
    L.oracle_tiny_expert_outputs.restype = None
    L.oracle_e2m1_encode_n.argtypes = [_P, _P, _L]
    L.oracle_e2m1_encode_n.restype = None
    L.oracle_e4m3_encode_n.argtypes = [_P, _P, _L]
    L.oracle_e4m3_encode_n.restype = None


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------------------------------
# scalar format helpers
# ------------------------------------------------------------------------------------------
def e2m1_encode(v: float) -> int:
    return int(lib().oracle_e2m1_encode(float(v)))


def e2m1_decode(code: int) -> float:
    return float(lib().oracle_e2m1_decode(code))


def e4m3_encode(v: float) -> int:
    return int(lib().oracle_e4m3_encode(float(v)))


def e4m3_decode(code: int) -> float:
    return float(lib().oracle_e4m3_decode(code))


def bf16_from_double(v: float) -> int:
    return int(lib().oracle_bf16_from_double(float(v)))


def bf16_to_double(b: int) -> float:
    return float(lib().oracle_bf16_to_double(int(b)))


def e2m1_encode_array(v: np.ndarray) -> np.ndarray:
    a = _c(v, np.float32)
    out = np.empty(a.shape, np.uint8)
    lib().oracle_e2m1_encode_n(_ptr(a), _ptr(out), a.size)
    return out


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    a = _c(v, np.float32)
    out = np.empty(a.shape, np.uint8)
    lib().oracle_e4m3_encode_n(_ptr(a), _ptr(out), a.size)
    return out


# ------------------------------------------------------------------------------------------
# layout
# ------------------------------------------------------------------------------------------
class Layout(dict):
    """Result of :func:`layout`: row_offsets, expert_ids, src_info, row_of, part_tokens, status
    plus the problem sizes T, K, E, P, C, S, the padding multiple ``pad`` and R (rows in use,
    padding included) / R_max (rows allocated)."""

    def __getattr__(self, k):
        try:
            return self[k]
        except KeyError as e:
            raise AttributeError(k) from e


def rows_max(T: int, K: int, E: int, S: int = 0, pad_multiple: int = 1,
             num_permuted_tokens: int | None = None) -> int:
    """Rows every dispatched buffer holds: the static capacity when one is given, else the most
    rows any routing can need, T*K + S*T + G*(pad_multiple - 1)."""
    return int(lib().oracle_rows_max(T, K, E, S, pad_multiple, num_permuted_tokens or 0))


def layout(topk_ids: np.ndarray, E: int, P: int = 1, C: int | None = None, S: int = 0,
           pad_multiple: int = 1, num_permuted_tokens: int | None = None) -> Layout:
    ids = _c(topk_ids, np.int32)
    T, K = ids.shape
    C = T if C is None else C
    G = E + S
    R_max = rows_max(T, K, E, S, pad_multiple, num_permuted_tokens)
    row_offsets = np.zeros(G + 1, np.int32)
    expert_ids = np.full(max(R_max, 1), -7, np.int32)
    src_info = np.full((max(R_max, 1), 2), -7, np.int32)
    row_of = np.zeros((T, K), np.int32)
    part = np.zeros(P, np.int32)
    st = lib().oracle_layout_padded(_ptr(ids), T, K, E, P, C, S, pad_multiple,
                                    num_permuted_tokens or 0, _ptr(row_offsets), _ptr(expert_ids),
                                    _ptr(src_info), _ptr(row_of), _ptr(part))
    R = int(row_offsets[G])
    return Layout(row_offsets=row_offsets, expert_ids=expert_ids[:R_max], src_info=src_info[:R_max],
                  row_of=row_of, part_tokens=part, status=int(st), T=T, K=K, E=E, P=P, C=C, S=S,
                  pad=pad_multiple, R=R, R_max=R_max)


def _fill_padding(L: Layout, buf: np.ndarray, row: np.ndarray) -> None:
    """Write ``row`` (the bytes an all-zero token dispatches to) into every padding row."""
    assert buf.flags.c_contiguous
    r = np.ascontiguousarray(row).view(np.uint8)
    src = _c(L.src_info, np.int32)
    lib().oracle_fill_padding_rows(_ptr(src), L.R, L.R_max, L.status, _ptr(buf.view(np.uint8)),
                                   r.size, _ptr(r))


# ------------------------------------------------------------------------------------------
# dispatch
# ------------------------------------------------------------------------------------------
def nvfp4_quantize_row(x_row: np.ndarray):
    """(codes uint8 [H/2], scales uint8 [H/16], inv bf16 bits) of one bf16 row."""
    x = _c(x_row, np.uint16)
    H = x.size
    codes = np.zeros(H // 2, np.uint8)
    scales = np.zeros(H // 16, np.uint8)
    inv = np.zeros(1, np.uint16)
    lib().oracle_nvfp4_quantize_row(_ptr(x), H, _ptr(codes), _ptr(scales), _ptr(inv))
    return codes, scales, int(inv[0])


def dispatch_nvfp4(x: np.ndarray, L: Layout, fill: int = 0xA5):
    """NVFP4 dispatch into buffers of R_max rows pre-filled with ``fill`` (rows past R and
    every row when the layout's status is non-zero keep the fill)."""
    x = _c(x, np.uint16)
    T, H = x.shape
    R_max = L.R_max
    fp4 = np.full((R_max, H // 2), fill, np.uint8)
    sc = np.full((R_max, H // 16), fill, np.uint8)
    inv = np.full(R_max, (fill << 8) | fill, np.uint16)
    so = np.full(L.E + L.S + 1, -7, np.int32)
    lib().oracle_dispatch_nvfp4(_ptr(x), T, H, L.K, L.E, L.S, _ptr(L.row_offsets), _ptr(L.row_of),
                                L.status, _ptr(fp4), _ptr(sc), _ptr(inv), _ptr(so))
    zc, zs, zi = nvfp4_quantize_row(np.zeros(H, np.uint16))
    _fill_padding(L, fp4, zc)
    _fill_padding(L, sc, zs)
    _fill_padding(L, inv, np.array([zi], np.uint16))
    return fp4, sc, inv, so


def dispatch_bf16(x: np.ndarray, L: Layout, fill: int = 0xA5A5):
    x = _c(x, np.uint16)
    T, H = x.shape
    out = np.full((L.R_max, H), fill, np.uint16)
    lib().oracle_dispatch_bf16(_ptr(x), T, H, L.K, L.E, L.S, _ptr(L.row_offsets), _ptr(L.row_of),
                               L.status, _ptr(out))
    _fill_padding(L, out, np.zeros(H, np.uint16))
    return out


FP8_BLOCK = 128


def fp8_quantize_row(x_row: np.ndarray):
    """(E4M3 codes uint8 [H], float32 scales [H/128]) of one bf16 row."""
    x = _c(x_row, np.uint16)
    H = x.size
    codes = np.zeros(H, np.uint8)
    scales = np.zeros(H // FP8_BLOCK, np.float32)
    lib().oracle_fp8_quantize_row(_ptr(x), H, _ptr(codes), _ptr(scales))
    return codes, scales


def dispatch_fp8(x: np.ndarray, L: Layout, fill: int = 0xA5):
    """FP8 dispatch into buffers of R_max rows pre-filled with ``fill`` bytes."""
    x = _c(x, np.uint16)
    T, H = x.shape
    codes = np.full((L.R_max, H), fill, np.uint8)
    sc = np.full((L.R_max, 4 * (H // FP8_BLOCK)), fill, np.uint8).view(np.float32)
    lib().oracle_dispatch_fp8(_ptr(x), T, H, L.K, L.E, L.S, _ptr(L.row_offsets), _ptr(L.row_of),
                              L.status, _ptr(codes), _ptr(sc))
    zc, zs = fp8_quantize_row(np.zeros(H, np.uint16))
    _fill_padding(L, codes, zc)
    _fill_padding(L, sc, zs)
    return codes, sc


# ------------------------------------------------------------------------------------------
# routing representations
# ------------------------------------------------------------------------------------------
def routing_map_to_topk(routing_map: np.ndarray, dense_probs: np.ndarray | None, K: int):
    """(topk_ids int32 [T,K], topk_probs float32 [T,K]) from a [T,E] map: ascending expert ids,
    -1 after the last; a token with more than K experts gets the id E in every slot."""
    m = _c(routing_map, np.uint8)
    T, E = m.shape
    ids = np.zeros((T, K), np.int32)
    probs = np.zeros((T, K), np.float32)
    dp = None if dense_probs is None else _c(dense_probs, np.float32)
    lib().oracle_routing_map_to_topk(_ptr(m), _ptr(dp), T, E, K, _ptr(ids), _ptr(probs))
    return ids, probs


def indices_to_multihot(topk_ids: np.ndarray, topk_probs: np.ndarray | None, E: int):
    """(routing_map uint8 [T,E], dense_probs float32 [T,E]) from compact ids and probabilities."""
    ids = _c(topk_ids, np.int32)
    T, K = ids.shape
    m = np.zeros((T, E), np.uint8)
    d = np.zeros((T, E), np.float32)
    p = None if topk_probs is None else _c(topk_probs, np.float32)
    lib().oracle_indices_to_multihot(_ptr(ids), _ptr(p), T, K, E, _ptr(m), _ptr(d))
    return m, d


# ------------------------------------------------------------------------------------------
# combine and backward
# ------------------------------------------------------------------------------------------
def combine(y: np.ndarray, probs: np.ndarray | None, L: Layout, want64: bool = False,
            fill: int = 0xA5A5):
    """Probability-weighted combine (``probs`` given) or dispatch backward (``probs`` None).
    Returns the bf16 output [T, H] (and the binary64 sums when ``want64``)."""
    y = _c(y, np.uint16)
    H = y.shape[1]
    T, K = L.T, L.K
    out = np.full((T, H), fill, np.uint16)
    out64 = np.zeros((T, H), np.float64) if want64 else None
    p = None if probs is None else _c(probs, np.float32)
    lib().oracle_combine(_ptr(y), _ptr(p), T, H, K, L.E, L.S, _ptr(L.row_offsets), _ptr(L.row_of),
                         L.status, _ptr(out), _ptr(out64))
    return (out, out64) if want64 else out


def dispatch_bwd(grad_rows: np.ndarray, L: Layout, want64: bool = False):
    return combine(grad_rows, None, L, want64=want64)


def combine_bwd(g: np.ndarray, y: np.ndarray, probs: np.ndarray, L: Layout, want64: bool = False,
                fill: int = 0xA5A5):
    """(grad_y bf16 [R_max, H], grad_p float64 [T, K]) (+ binary64 grad_y when ``want64``)."""
    g = _c(g, np.uint16)
    y = _c(y, np.uint16)
    p = _c(probs, np.float32)
    T, H = g.shape
    gy = np.full((L.R_max, H), fill, np.uint16)
    gp = np.zeros((T, L.K), np.float64)
    gy64 = np.zeros((L.R_max, H), np.float64) if want64 else None
    lib().oracle_combine_bwd(_ptr(g), _ptr(y), _ptr(p), T, H, L.K, L.E, L.S, _ptr(L.row_offsets),
                             _ptr(L.row_of), L.status, _ptr(gy), _ptr(gp), _ptr(gy64))
    _fill_padding(L, gy, np.zeros(H, np.uint16))   # a padding row's gradient is zero
    return (gy, gp, gy64) if want64 else (gy, gp)


def tiny_expert_outputs(fp4, scales, inv, L: Layout) -> np.ndarray:
    """Expert outputs of the Tiny workload: dequantised dispatched rows x (1 + expert/8)."""
    H = fp4.shape[1] * 2
    y = np.zeros((L.R_max, H), np.uint16)
    lib().oracle_tiny_expert_outputs(_ptr(_c(fp4, np.uint8)), _ptr(_c(scales, np.uint8)),
                                     _ptr(_c(inv, np.uint16)), _ptr(_c(L.expert_ids, np.int32)),
                                     L.R, H, _ptr(y))
    return y


def dequantize_rows(fp4: np.ndarray, scales: np.ndarray, inv_or_g: np.ndarray) -> np.ndarray:
    """Float64 values code * block scale * factor per row (factor given per row in fp64)."""
    lo = (fp4 & 0xF).astype(np.uint8)
    hi = (fp4 >> 4).astype(np.uint8)
    R, h2 = fp4.shape
    codes = np.empty((R, 2 * h2), np.uint8)
    codes[:, 0::2] = lo
    codes[:, 1::2] = hi
    table = np.array([e2m1_decode(c) for c in range(16)], np.float64)
    stab = np.array([e4m3_decode(c) for c in range(256)], np.float64)
    v = table[codes] * np.repeat(stab[scales], 16, axis=1)
    return v * np.asarray(inv_or_g, np.float64).reshape(R, 1)
