"""GB300 MoE token dispatch / combine: a thin Python binding over libep_gb300.so.

Every function here only marshals arguments (torch device tensors -> pointers, sizes and the
current CUDA stream) and calls the C ABI declared in ``include/ep.h``; every step of the path
runs in the library's CUDA kernels.  There is no CPU fallback: importing the binding without
the built library raises.

Entry points (same names as the C ABI, without the ``ep_`` prefix):
``dispatch_layout``, ``dispatch_layout_routed``, ``dispatch_layout_noalloc``, ``dispatch_nvfp4``,
``dispatch_layout_nvfp4``, ``dispatch_layout_padded_nvfp4``, ``dispatch_bf16``, ``dispatch_fp8``, ``combine``, ``combine_bwd``,
``dispatch_bwd``, ``routing_map_to_topk``, ``indices_to_multihot``, ``rows_max``,
``read_status``, ``cvt_e2m1``, ``cvt_e4m3``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# EP_GB300_CHECKED=1 selects the bounds-checked debug build of the same sources, which reports
# an index outside its buffer as EP_STATUS_BOUNDS instead of relying on the caller's layout.
CHECKED = os.environ.get("EP_GB300_CHECKED", "0") == "1"
LIB_PATH = os.path.join(_HERE, "_build", "libep_gb300_checked.so" if CHECKED else "libep_gb300.so")

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_OVERFLOW = 2
EP_ERR_BAD_EXPERT = 3
EP_ERR_CUDA = 5
EP_ERR_TOO_LARGE = 6
EP_ERR_BOUNDS = 7
NOALLOC_WORKSPACE_BYTES = 1 << 20
STATUS_OVERFLOW = 1
STATUS_BAD_EXPERT = 2
STATUS_BOUNDS = 8


class EPError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} (code {code})")
        self.code = code


class _Layout(ctypes.Structure):
    _fields_ = [
        ("row_offsets", ctypes.c_void_p),
        ("expert_ids", ctypes.c_void_p),
        ("src_info", ctypes.c_void_p),
        ("row_of", ctypes.c_void_p),
        ("part_tokens", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("T", ctypes.c_int),
        ("K", ctypes.c_int),
        ("E", ctypes.c_int),
        ("P", ctypes.c_int),
        ("capacity", ctypes.c_int),
        ("fused_shared", ctypes.c_int),
        ("pad_multiple", ctypes.c_int),
        ("row_capacity", ctypes.c_int),
    ]


_P, _I, _L, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_size_t
_LP = ctypes.POINTER(_Layout)

# name -> (restype, argtypes); must match include/ep.h
SIGNATURES = {
    "ep_layout_workspace_bytes": (_Z, [_I, _I, _I, _I]),
    "ep_rows_max": (_Z, [_I, _I, _I, _I, _I, _I]),
    "ep_dispatch_layout": (_I, [_P, _I, _I, _I, _I, _I, _I, _LP, _P]),
    "ep_dispatch_layout_routed": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _LP, _P]),
    "ep_routing_map_to_topk": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "ep_indices_to_multihot": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "ep_dispatch_fp8": (_I, [_P, _I, _LP, _P, _P, _P]),
    "ep_dispatch_layout_noalloc": (_I, [_P, _I, _I, _I, _I, _I, _I, _LP, _P]),
    "ep_dispatch_nvfp4": (_I, [_P, _I, _LP, _P, _P, _P, _P, _P]),
    "ep_dispatch_layout_nvfp4": (_I, [_P, _I, _I, _I, _I, _I, _I, _P, _I, _LP, _P, _P, _P, _P, _P]),
    "ep_dispatch_layout_padded_nvfp4": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _LP, _P, _P, _P,
                                             _P, _P]),
    "ep_dispatch_bf16": (_I, [_P, _I, _LP, _P, _P]),
    "ep_combine": (_I, [_P, _P, _I, _LP, _P, _P]),
    "ep_combine_bwd": (_I, [_P, _P, _P, _I, _LP, _P, _P, _P]),
    "ep_dispatch_bwd": (_I, [_P, _I, _LP, _P, _P]),
    "ep_read_status": (_I, [_LP, _P, ctypes.POINTER(ctypes.c_int32)]),
    "ep_strerror": (ctypes.c_char_p, [_I]),
    "ep_cvt_e2m1": (_I, [_P, _P, _L, _P]),
    "ep_cvt_e4m3": (_I, [_P, _P, _L, _P]),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libep_gb300.so is not built ({LIB_PATH}); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` from the repository root")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


def strerror(code: int) -> str:
    return _lib.ep_strerror(code).decode()


def _check(rc: int, what: str):
    if rc != EP_OK:
        raise EPError(rc, what)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _bits(t: torch.Tensor):
    """bf16 tensors travel as their 16-bit patterns."""
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"expected a bf16 tensor, got {t.dtype}")
    return _ptr(t)


def _need(t: torch.Tensor, rows_at_least: int | None, cols: int | None, dtypes, what: str,
          exact_rows: int | None = None):
    """Shape / dtype check of a tensor handed to the library (the C ABI trusts buffer sizes)."""
    if t.dtype not in dtypes:
        raise TypeError(f"{what}: dtype {t.dtype} not in {dtypes}")
    if cols is not None and (t.dim() != 2 or t.shape[1] != cols):
        raise ValueError(f"{what}: expected [*, {cols}], got {tuple(t.shape)}")
    n = t.shape[0] if t.dim() else 1
    if exact_rows is not None and n != exact_rows:
        raise ValueError(f"{what}: expected {exact_rows} rows, got {n}")
    if rows_at_least is not None and n < rows_at_least:
        raise ValueError(f"{what}: needs at least {rows_at_least} rows, got {n}")


_BF16 = (torch.bfloat16, torch.int16, torch.uint16)


def layout_workspace_bytes(T: int, K: int, n_experts: int, fused_shared: bool = False) -> int:
    return int(_lib.ep_layout_workspace_bytes(T, K, n_experts, int(bool(fused_shared))))


def rows_max(T: int, K: int, n_experts: int, fused_shared: bool = False, pad_multiple: int = 1,
             num_permuted_tokens: int | None = None) -> int:
    """ep_rows_max: rows every dispatched buffer holds (the static capacity when one is given,
    else T*K + S*T + G*(pad_multiple - 1))."""
    n = int(_lib.ep_rows_max(T, K, n_experts, int(bool(fused_shared)), pad_multiple,
                             int(num_permuted_tokens or 0)))
    if n == 0 and T * K > 0:
        raise EPError(EP_ERR_INVALID_ARG, "rows_max sizes")
    return n


class Layout:
    """Device buffers of one dispatch layout (see ``ep_layout_t`` in include/ep.h).

    ``row_offsets`` [G+1], ``expert_ids`` [R_max], ``src_info`` [R_max, 2], ``row_of`` [T, K],
    ``part_tokens`` [P], ``status`` [1] and the zero-initialised ``workspace``; all int32
    except the workspace (uint8).  The buffers are allocated once for a shape (including the
    padding multiple and the static row capacity, which set R_max) and reused by every layout
    call into this object.
    """

    def __init__(self, T: int, K: int, n_experts: int, n_parts: int = 1, fused_shared: bool = False,
                 device=None, pad_multiple: int = 1, num_permuted_tokens: int | None = None):
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        S = int(bool(fused_shared))
        self.T, self.K, self.E, self.P, self.S = T, K, n_experts, n_parts, S
        self.G = n_experts + S
        self.pad = int(pad_multiple)
        self.row_capacity = int(num_permuted_tokens or 0)
        self.R_max = rows_max(T, K, n_experts, S, self.pad, self.row_capacity)
        i32 = dict(dtype=torch.int32, device=dev)
        self.row_offsets = torch.empty(self.G + 1, **i32)
        self.expert_ids = torch.empty(max(self.R_max, 1), **i32)
        self.src_info = torch.empty(max(self.R_max, 1), 2, **i32)
        self.row_of = torch.empty(max(T, 1), K, **i32)
        self.part_tokens = torch.empty(n_parts, **i32)
        self.status = torch.zeros(4, **i32)      # 16 bytes keeps the word aligned
        nb = layout_workspace_bytes(T, K, n_experts, S)
        if nb == 0:
            raise EPError(EP_ERR_INVALID_ARG, "layout sizes")
        self.workspace = torch.zeros(nb, dtype=torch.uint8, device=dev)
        self.capacity = T
        self.c = _Layout(
            row_offsets=self.row_offsets.data_ptr(), expert_ids=self.expert_ids.data_ptr(),
            src_info=self.src_info.data_ptr(), row_of=self.row_of.data_ptr(),
            part_tokens=self.part_tokens.data_ptr(), status=self.status.data_ptr(),
            workspace=self.workspace.data_ptr(), workspace_bytes=nb)

    @property
    def ref(self):
        return ctypes.byref(self.c)

    def shape_key(self):
        return (self.T, self.K, self.E, self.P, self.S, self.pad, self.row_capacity)

    def num_rows(self) -> torch.Tensor:
        """R as a device tensor (no host sync)."""
        return self.row_offsets[self.G]


def dispatch_layout(topk_ids: torch.Tensor, n_experts: int, n_parts: int = 1,
                    capacity: int | None = None, fused_shared: bool = False,
                    out: Layout | None = None, stream=None) -> Layout:
    """ep_dispatch_layout: routing metadata from top-k ids [T, K] int32 (-1 = unused slot)."""
    if topk_ids.dtype != torch.int32 or topk_ids.dim() != 2:
        raise TypeError("topk_ids must be an int32 [T, K] tensor")
    T, K = topk_ids.shape
    if out is not None and out.shape_key() != (T, K, n_experts, n_parts, int(bool(fused_shared)), 1, 0):
        raise ValueError(f"layout buffers were allocated for other sizes {out.shape_key()}")
    L = out if out is not None else Layout(T, K, n_experts, n_parts, fused_shared, topk_ids.device)
    cap = T if capacity is None else int(capacity)
    L.capacity = cap
    rc = _lib.ep_dispatch_layout(_ptr(topk_ids) if T > 0 else None, T, K, n_experts, n_parts, cap,
                                 int(bool(fused_shared)), L.ref, _stream(stream))
    _check(rc, "ep_dispatch_layout")
    return L


def dispatch_layout_noalloc(topk_ids: torch.Tensor, n_experts: int, n_parts: int = 1,
                            capacity: int | None = None, fused_shared: bool = False,
                            out: Layout | None = None, stream=None) -> Layout:
    """ep_dispatch_layout_noalloc: the layout of ``dispatch_layout`` for callers that cannot
    allocate device memory; its scratch is a fixed 1 MiB array inside the library, so the
    layout's own workspace is not used.  ``out`` (the output buffers) must be given: this call
    allocates nothing.  The first call on a device sets the array up (make it before any stream
    capture); calls that overlap on the GPU race on the shared array."""
    if topk_ids.dtype != torch.int32 or topk_ids.dim() != 2:
        raise TypeError("topk_ids must be an int32 [T, K] tensor")
    if out is None:
        raise ValueError("dispatch_layout_noalloc writes into caller-provided buffers: pass out=")
    T, K = topk_ids.shape
    if out.shape_key() != (T, K, n_experts, n_parts, int(bool(fused_shared)), 1, 0):
        raise ValueError(f"layout buffers were allocated for other sizes {out.shape_key()}")
    cap = T if capacity is None else int(capacity)
    out.capacity = cap
    rc = _lib.ep_dispatch_layout_noalloc(_ptr(topk_ids) if T > 0 else None, T, K, n_experts, n_parts,
                                         cap, int(bool(fused_shared)), out.ref, _stream(stream))
    _check(rc, "ep_dispatch_layout_noalloc")
    return out


def dispatch_layout_routed(n_experts: int, topk_ids: torch.Tensor | None = None,
                           routing_map: torch.Tensor | None = None,
                           dense_probs: torch.Tensor | None = None, K: int | None = None,
                           n_parts: int = 1, capacity: int | None = None,
                           fused_shared: bool = False, pad_multiple: int = 1,
                           num_permuted_tokens: int | None = None, out: Layout | None = None,
                           map_out=None, stream=None):
    """ep_dispatch_layout_routed: the layout from compact ids [T, K] or from a dense routing map
    [T, E] (uint8 / bool, which takes precedence when both are given, with optional dense
    probabilities [T, E] fp32), with groups padded to ``pad_multiple`` rows and an optional
    static row capacity ``num_permuted_tokens``.  Returns (Layout, topk_ids, topk_probs): the
    compact ids the layout was made from (the converted map when one was given) and, for a map
    with dense probabilities, the per-slot probabilities combine takes (else None)."""
    if routing_map is not None:
        if routing_map.dtype not in (torch.uint8, torch.bool) or routing_map.dim() != 2:
            raise TypeError("routing_map must be a uint8 / bool [T, E] tensor")
        T, E = routing_map.shape
        if E != n_experts:
            raise ValueError("routing_map has the wrong number of experts")
        if K is None:
            K = topk_ids.shape[1] if topk_ids is not None else None
        if K is None:
            raise ValueError("K (slots per token) is needed with a routing map")
        if dense_probs is not None:
            _need(dense_probs, None, E, (torch.float32,), "dense_probs", exact_rows=T)
        dev = routing_map.device
        if map_out is None:
            map_out = (torch.empty(max(T, 1), K, dtype=torch.int32, device=dev),
                       torch.empty(max(T, 1), K, dtype=torch.float32, device=dev)
                       if dense_probs is not None else None)
        ids, probs = map_out
        _need(ids, T, K, (torch.int32,), "map_topk_ids")
        if probs is not None:
            _need(probs, T, K, (torch.float32,), "map_topk_probs")
        rmap = routing_map.view(torch.uint8) if routing_map.dtype == torch.bool else routing_map
    else:
        if topk_ids is None or topk_ids.dtype != torch.int32 or topk_ids.dim() != 2:
            raise TypeError("topk_ids must be an int32 [T, K] tensor when no routing_map is given")
        T, K = topk_ids.shape
        ids, probs, rmap = topk_ids, None, None
        dev = topk_ids.device
    S = int(bool(fused_shared))
    key = (T, K, n_experts, n_parts, S, int(pad_multiple), int(num_permuted_tokens or 0))
    if out is not None and out.shape_key() != key:
        raise ValueError(f"layout buffers were allocated for other sizes {out.shape_key()}")
    L = out if out is not None else Layout(T, K, n_experts, n_parts, fused_shared, dev,
                                           pad_multiple, num_permuted_tokens)
    cap = T if capacity is None else int(capacity)
    L.capacity = cap
    rc = _lib.ep_dispatch_layout_routed(
        _ptr(topk_ids) if (rmap is None and T > 0) else None,
        _ptr(rmap) if (rmap is not None and T > 0) else None,
        _ptr(dense_probs) if (rmap is not None and T > 0) else None,
        T, K, n_experts, n_parts, cap, S, int(pad_multiple), int(num_permuted_tokens or 0),
        _ptr(ids) if (rmap is not None and T > 0) else None,
        _ptr(probs) if (rmap is not None and T > 0) else None, L.ref, _stream(stream))
    _check(rc, "ep_dispatch_layout_routed")
    return L, ids, probs


def routing_map_to_topk(routing_map: torch.Tensor, dense_probs: torch.Tensor | None, K: int,
                        out=None, stream=None):
    """ep_routing_map_to_topk -> (topk_ids int32 [T, K], topk_probs fp32 [T, K] or None)."""
    if routing_map.dtype not in (torch.uint8, torch.bool) or routing_map.dim() != 2:
        raise TypeError("routing_map must be a uint8 / bool [T, E] tensor")
    T, E = routing_map.shape
    if dense_probs is not None:
        _need(dense_probs, None, E, (torch.float32,), "dense_probs", exact_rows=T)
    if out is None:
        out = (torch.empty(max(T, 1), K, dtype=torch.int32, device=routing_map.device),
               torch.empty(max(T, 1), K, dtype=torch.float32, device=routing_map.device)
               if dense_probs is not None else None)
    ids, probs = out
    _need(ids, T, K, (torch.int32,), "topk_ids")
    if probs is not None:
        _need(probs, T, K, (torch.float32,), "topk_probs")
    rmap = routing_map.view(torch.uint8) if routing_map.dtype == torch.bool else routing_map
    rc = _lib.ep_routing_map_to_topk(_ptr(rmap), _ptr(dense_probs), T, E, K, _ptr(ids), _ptr(probs),
                                     _stream(stream))
    _check(rc, "ep_routing_map_to_topk")
    return ids, probs


def indices_to_multihot(topk_ids: torch.Tensor, topk_probs: torch.Tensor | None, n_experts: int,
                        out=None, stream=None):
    """ep_indices_to_multihot -> (routing_map uint8 [T, E], dense_probs fp32 [T, E] or None)."""
    if topk_ids.dtype != torch.int32 or topk_ids.dim() != 2:
        raise TypeError("topk_ids must be an int32 [T, K] tensor")
    T, K = topk_ids.shape
    if topk_probs is not None:
        _need(topk_probs, None, K, (torch.float32,), "topk_probs", exact_rows=T)
    if out is None:
        out = (torch.empty(max(T, 1), n_experts, dtype=torch.uint8, device=topk_ids.device),
               torch.empty(max(T, 1), n_experts, dtype=torch.float32, device=topk_ids.device)
               if topk_probs is not None else None)
    rmap, dense = out
    _need(rmap, T, n_experts, (torch.uint8,), "routing_map")
    if dense is not None:
        _need(dense, T, n_experts, (torch.float32,), "dense_probs")
    rc = _lib.ep_indices_to_multihot(_ptr(topk_ids), _ptr(topk_probs), T, K, n_experts, _ptr(rmap),
                                     _ptr(dense), _stream(stream))
    _check(rc, "ep_indices_to_multihot")
    return rmap, dense


def dispatch_fp8(x: torch.Tensor, L: Layout, out=None, stream=None):
    """ep_dispatch_fp8 -> (E4M3 codes uint8 [R_max, H], fp32 scales [R_max, H/128])."""
    T, H = x.shape
    _need(x, None, H, _BF16, "input_tokens", exact_rows=L.T)
    if H % 128:
        raise ValueError("FP8 dispatch needs H % 128 == 0")
    if out is None:
        out = (torch.empty(max(L.R_max, 1), H, dtype=torch.uint8, device=x.device),
               torch.empty(max(L.R_max, 1), H // 128, dtype=torch.float32, device=x.device))
    codes, sc = out
    _need(codes, L.R_max, H, (torch.uint8,), "out_fp8")
    _need(sc, L.R_max, H // 128, (torch.float32,), "out_scales")
    rc = _lib.ep_dispatch_fp8(_bits(x), H, L.ref, _ptr(codes), _ptr(sc), _stream(stream))
    _check(rc, "ep_dispatch_fp8")
    return out


def dispatch_nvfp4(x: torch.Tensor, L: Layout, out=None, stream=None):
    """ep_dispatch_nvfp4 -> (fp4 codes uint8 [R_max, H/2], E4M3 scales uint8 [R_max, H/16],
    bf16 inverse global scales [R_max], scales_offsets int32 [G+1])."""
    T, H = x.shape
    _need(x, None, H, _BF16, "input_tokens", exact_rows=L.T)
    if out is None:
        dev = x.device
        out = (torch.empty(max(L.R_max, 1), H // 2, dtype=torch.uint8, device=dev),
               torch.empty(max(L.R_max, 1), H // 16, dtype=torch.uint8, device=dev),
               torch.empty(max(L.R_max, 1), dtype=torch.bfloat16, device=dev),
               torch.empty(L.G + 1, dtype=torch.int32, device=dev))
    fp4, sc, inv, so = out
    _need(fp4, L.R_max, H // 2, (torch.uint8,), "out_fp4")
    _need(sc, L.R_max, H // 16, (torch.uint8,), "out_scales")
    _need(inv, L.R_max, None, _BF16, "out_rowwise_inv_scale")
    _need(so, L.G + 1, None, (torch.int32,), "scales_offsets")
    rc = _lib.ep_dispatch_nvfp4(_bits(x), H, L.ref, _ptr(fp4), _ptr(sc), _bits(inv), _ptr(so),
                                _stream(stream))
    _check(rc, "ep_dispatch_nvfp4")
    return out


def dispatch_layout_nvfp4(topk_ids: torch.Tensor, x: torch.Tensor, n_experts: int, n_parts: int = 1,
                          capacity: int | None = None, fused_shared: bool = False,
                          out_layout: Layout | None = None, out=None, stream=None):
    """ep_dispatch_layout_nvfp4: layout + NVFP4 dispatch in one call (the quantisation overlaps
    the layout).  Returns (Layout, (fp4, scales, inv, scales_offsets))."""
    if topk_ids.dtype != torch.int32 or topk_ids.dim() != 2:
        raise TypeError("topk_ids must be an int32 [T, K] tensor")
    T, K = topk_ids.shape
    Tx, H = x.shape
    if Tx != T:
        raise ValueError("x and topk_ids disagree on the number of tokens")
    S = int(bool(fused_shared))
    L = out_layout
    if L is not None and L.shape_key() != (T, K, n_experts, n_parts, S, 1, 0):
        raise ValueError(f"layout buffers were allocated for other sizes {L.shape_key()}")
    if L is None:
        L = Layout(T, K, n_experts, n_parts, fused_shared, topk_ids.device)
    _need(x, None, H, _BF16, "input_tokens", exact_rows=T)
    if out is None:
        dev = x.device
        out = (torch.empty(max(L.R_max, 1), H // 2, dtype=torch.uint8, device=dev),
               torch.empty(max(L.R_max, 1), H // 16, dtype=torch.uint8, device=dev),
               torch.empty(max(L.R_max, 1), dtype=torch.bfloat16, device=dev),
               torch.empty(L.G + 1, dtype=torch.int32, device=dev))
    fp4, sc, inv, so = out
    _need(fp4, L.R_max, H // 2, (torch.uint8,), "out_fp4")
    _need(sc, L.R_max, H // 16, (torch.uint8,), "out_scales")
    _need(inv, L.R_max, None, _BF16, "out_rowwise_inv_scale")
    _need(so, L.G + 1, None, (torch.int32,), "scales_offsets")
    cap = T if capacity is None else int(capacity)
    L.capacity = cap
    rc = _lib.ep_dispatch_layout_nvfp4(_ptr(topk_ids) if T > 0 else None, T, K, n_experts, n_parts, cap,
                                       S, _bits(x) if T > 0 else None, H, L.ref, _ptr(fp4), _ptr(sc),
                                       _bits(inv), _ptr(so), _stream(stream))
    _check(rc, "ep_dispatch_layout_nvfp4")
    return L, out


def _nvfp4_out(L: Layout, H: int, out, dev):
    if out is None:
        out = (torch.empty(max(L.R_max, 1), H // 2, dtype=torch.uint8, device=dev),
               torch.empty(max(L.R_max, 1), H // 16, dtype=torch.uint8, device=dev),
               torch.empty(max(L.R_max, 1), dtype=torch.bfloat16, device=dev),
               torch.empty(L.G + 1, dtype=torch.int32, device=dev))
    fp4, sc, inv, so = out
    _need(fp4, L.R_max, H // 2, (torch.uint8,), "out_fp4")
    _need(sc, L.R_max, H // 16, (torch.uint8,), "out_scales")
    _need(inv, L.R_max, None, _BF16, "out_rowwise_inv_scale")
    _need(so, L.G + 1, None, (torch.int32,), "scales_offsets")
    return out


def dispatch_layout_padded_nvfp4(topk_ids: torch.Tensor, x: torch.Tensor, n_experts: int,
                                 n_parts: int = 1, capacity: int | None = None,
                                 fused_shared: bool = False, pad_multiple: int = 1,
                                 num_permuted_tokens: int | None = None,
                                 out_layout: Layout | None = None, out=None, stream=None):
    """ep_dispatch_layout_padded_nvfp4: the layout of ``dispatch_layout_routed`` from compact ids
    (groups padded to ``pad_multiple`` rows, optional static row capacity) and the NVFP4
    dispatch in one call; padding rows get the dispatch of an all-zero token.  Returns
    (Layout, (fp4, scales, inv, scales_offsets))."""
    if topk_ids.dtype != torch.int32 or topk_ids.dim() != 2:
        raise TypeError("topk_ids must be an int32 [T, K] tensor")
    T, K = topk_ids.shape
    Tx, H = x.shape
    if Tx != T:
        raise ValueError("x and topk_ids disagree on the number of tokens")
    S = int(bool(fused_shared))
    key = (T, K, n_experts, n_parts, S, int(pad_multiple), int(num_permuted_tokens or 0))
    L = out_layout
    if L is not None and L.shape_key() != key:
        raise ValueError(f"layout buffers were allocated for other sizes {L.shape_key()}")
    if L is None:
        L = Layout(T, K, n_experts, n_parts, fused_shared, topk_ids.device, pad_multiple,
                   num_permuted_tokens)
    _need(x, None, H, _BF16, "input_tokens", exact_rows=T)
    out = _nvfp4_out(L, H, out, x.device)
    fp4, sc, inv, so = out
    cap = T if capacity is None else int(capacity)
    L.capacity = cap
    rc = _lib.ep_dispatch_layout_padded_nvfp4(
        _ptr(topk_ids) if T > 0 else None, T, K, n_experts, n_parts, cap, S, int(pad_multiple),
        int(num_permuted_tokens or 0), _bits(x) if T > 0 else None, H, L.ref, _ptr(fp4), _ptr(sc),
        _bits(inv), _ptr(so), _stream(stream))
    _check(rc, "ep_dispatch_layout_padded_nvfp4")
    return L, out


def dispatch_bf16(x: torch.Tensor, L: Layout, out: torch.Tensor | None = None, stream=None):
    """ep_dispatch_bf16 -> dispatched rows bf16 [R_max, H]."""
    T, H = x.shape
    _need(x, None, H, _BF16, "input_tokens", exact_rows=L.T)
    if out is None:
        out = torch.empty(max(L.R_max, 1), H, dtype=torch.bfloat16, device=x.device)
    _need(out, L.R_max, H, _BF16, "out")
    _check(_lib.ep_dispatch_bf16(_bits(x), H, L.ref, _bits(out), _stream(stream)), "ep_dispatch_bf16")
    return out


def combine(expert_out: torch.Tensor, probs: torch.Tensor, L: Layout, out: torch.Tensor | None = None,
            stream=None):
    """ep_combine -> out bf16 [T, H] = sum_k probs * expert_out[row_of] (+ shared row)."""
    H = expert_out.shape[1]
    _need(expert_out, L.R_max, H, _BF16, "expert_out")
    _need(probs, None, L.K, (torch.float32,), "probs", exact_rows=L.T)
    if out is None:
        out = torch.empty(max(L.T, 1), H, dtype=torch.bfloat16, device=expert_out.device)
    _need(out, L.T, H, _BF16, "out")
    _check(_lib.ep_combine(_bits(expert_out), _ptr(probs), H, L.ref, _bits(out), _stream(stream)),
           "ep_combine")
    return out


def combine_bwd(grad_out: torch.Tensor, expert_out: torch.Tensor, probs: torch.Tensor, L: Layout,
                out=None, stream=None):
    """ep_combine_bwd -> (grad_expert_out bf16 [R_max, H], grad_probs fp32 [T, K])."""
    T, H = grad_out.shape
    _need(grad_out, None, H, _BF16, "grad_out", exact_rows=L.T)
    _need(expert_out, L.R_max, H, _BF16, "expert_out")
    _need(probs, None, L.K, (torch.float32,), "probs", exact_rows=L.T)
    if out is None:
        out = (torch.empty(max(L.R_max, 1), H, dtype=torch.bfloat16, device=grad_out.device),
               torch.empty(max(T, 1), L.K, dtype=torch.float32, device=grad_out.device))
    gy, gp = out
    _need(gy, L.R_max, H, _BF16, "grad_expert_out")
    _need(gp, L.T, L.K, (torch.float32,), "grad_probs")
    rc = _lib.ep_combine_bwd(_bits(grad_out), _bits(expert_out), _ptr(probs), H, L.ref, _bits(gy),
                             _ptr(gp), _stream(stream))
    _check(rc, "ep_combine_bwd")
    return out


def dispatch_bwd(grad_rows: torch.Tensor, L: Layout, out: torch.Tensor | None = None, stream=None):
    """ep_dispatch_bwd -> grad_input bf16 [T, H] = sum_k grad_rows[row_of] (+ shared row)."""
    H = grad_rows.shape[1]
    _need(grad_rows, L.R_max, H, _BF16, "grad_rows")
    if out is None:
        out = torch.empty(max(L.T, 1), H, dtype=torch.bfloat16, device=grad_rows.device)
    _need(out, L.T, H, _BF16, "grad_input")
    _check(_lib.ep_dispatch_bwd(_bits(grad_rows), H, L.ref, _bits(out), _stream(stream)), "ep_dispatch_bwd")
    return out


def read_status(L: Layout, stream=None) -> int:
    """ep_read_status: synchronises the stream and returns the status bits (0 = ok)."""
    v = ctypes.c_int32(0)
    rc = _lib.ep_read_status(L.ref, _stream(stream), ctypes.byref(v))
    if rc == EP_ERR_CUDA or rc == EP_ERR_INVALID_ARG:
        raise EPError(rc, "ep_read_status")
    return int(v.value)


def cvt_e2m1(v: torch.Tensor, stream=None) -> torch.Tensor:
    """ep_cvt_e2m1: E2M1 code of each fp32 element (one code per byte)."""
    out = torch.empty(v.numel(), dtype=torch.uint8, device=v.device)
    _check(_lib.ep_cvt_e2m1(_ptr(v), _ptr(out), v.numel(), _stream(stream)), "ep_cvt_e2m1")
    return out


def cvt_e4m3(v: torch.Tensor, stream=None) -> torch.Tensor:
    """ep_cvt_e4m3: E4M3 code of each fp32 element."""
    out = torch.empty(v.numel(), dtype=torch.uint8, device=v.device)
    _check(_lib.ep_cvt_e4m3(_ptr(v), _ptr(out), v.numel(), _stream(stream)), "ep_cvt_e4m3")
    return out
