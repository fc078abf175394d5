"""Thin ctypes binding of libdsv4 (include/dsv4.h): argument marshalling only.

Every function named ``dsv4_*`` here calls the C entry point of the same name;
all work runs in the library's CUDA kernels. torch provides device memory and
streams. There is no fallback: if the library is missing the import fails.
"""
import ctypes
import os

import torch

from . import accounting  # noqa: F401  (re-exported for users)

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdsv4.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libdsv4.so not built ({_LIB_PATH}); run `python -m compressed_sparse_kv_05_b300.build`")

lib = ctypes.CDLL(_LIB_PATH)

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_WORKSPACE, ERR_CUDA, ERR_SCRATCH = 0, -1, -2, -3, -4, -5, -6
STATIC_SCRATCH_BYTES = 32 << 20
STATUS_CAPACITY, STATUS_BAD_INDEX, STATUS_TIMEOUT, STATUS_RANGE = 1, 2, 4, 8
_ERR_NAMES = {-1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "MISALIGNED", -4: "WORKSPACE", -5: "CUDA", -6: "SCRATCH"}


class Dsv4Error(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {_ERR_NAMES.get(code, code)} ({code})")
        self.code = code


class LayerDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("batch", "d_nope", "d_rope", "ratio", "window", "separate_v", "idx_dim", "capacity")]


class KvPlanes(ctypes.Structure):
    _fields_ = [("nope", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("rope", ctypes.c_void_p)]


class CacheStruct(ctypes.Structure):
    _fields_ = [("k", KvPlanes), ("v", KvPlanes)] + [(n, ctypes.c_void_p) for n in (
        "idx_codes", "idx_scales", "win_k", "win_v", "pend_k", "pend_v", "pend_z", "pend_u", "pend_zu",
        "n_tokens", "status")]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_DESC = ctypes.POINTER(LayerDesc)
_CACHE = ctypes.POINTER(CacheStruct)

_SIGS = {
    "dsv4_compress_append": ([_DESC, _CACHE, _I32, _P, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "dsv4_index_topk": ([_DESC, _CACHE, _I32, _P, _P, _I32, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "dsv4_csa_decode": ([_DESC, _CACHE, _I32, _P, ctypes.c_float, _P, _I32, _P, _P, _P, ctypes.c_size_t, _P],
                        ctypes.c_int),
    "dsv4_hca_decode": ([_DESC, _CACHE, _I32, _P, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "dsv4_hca_decode_static": ([_DESC, _CACHE, _I32, _P, ctypes.c_float, _P, _P, _P], ctypes.c_int),
    "dsv4_index_topk_multi": ([_DESC, _CACHE, _I32, _I32, _P, _P, _I32, _P, _P, _P, ctypes.c_size_t, _P],
                              ctypes.c_int),
    "dsv4_csa_decode_multi": ([_DESC, _CACHE, _I32, _I32, _P, ctypes.c_float, _P, _I32, _P, _P, _P, _P, _P,
                               ctypes.c_size_t, _P], ctypes.c_int),
    "dsv4_hca_decode_multi": ([_DESC, _CACHE, _I32, _I32, _P, ctypes.c_float, _P, _P, _P, _P, _P, ctypes.c_size_t,
                               _P], ctypes.c_int),
    "dsv4_workspace_size_multi": ([_DESC, _I32, _I32, _I32, _I32], ctypes.c_size_t),
    "dsv4_workspace_size": ([_DESC, _I32, _I32, _I32], ctypes.c_size_t),
    "dsv4_decode_plan": ([_DESC, _I32, _I32, _P], ctypes.c_int),
    "dsv4_read_status": ([_CACHE, _P], ctypes.c_int),
    "dsv4_debug_force_timeout": ([_I32], ctypes.c_int),
    "dsv4_project_streams": ([_DESC, _CACHE, _I32, _I32, _P, _P, ctypes.c_float, _P, _P, _P, _P, _P], ctypes.c_int),
    "dsv4_quantize_kv_rows": ([_P, _I64, _I32, _I32, _P, _P, _P, _P], ctypes.c_int),
    "dsv4_quantize_fp4_rows": ([_P, _I64, _I32, _P, _P, _P], ctypes.c_int),
    "dsv4_pool_rows": ([_P, _P, _P, _I64, _I32, _I32, _P, _P], ctypes.c_int),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGS)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(name, code):
    if code < 0:
        raise Dsv4Error(name, code)
    return code


def layer_desc(layer, capacity):
    """LayerDesc for a ``workloads.Layer`` with the given entry capacity."""
    return LayerDesc(layer.batch, layer.d_nope, layer.d_rope, layer.ratio, layer.window,
                     1 if layer.separate_v else 0, layer.idx_dim if layer.kind == "csa" else 0, capacity)


class Cache:
    """Device planes of one layer's cache, allocated (zeroed) through torch."""

    def __init__(self, desc, device="cuda"):
        self.desc = desc
        B, cap, D = desc.batch, desc.capacity, desc.d_nope + desc.d_rope
        kw = dict(device=device)
        z = torch.zeros
        self.k_nope = z((B, cap, desc.d_nope), dtype=torch.uint8, **kw)
        self.k_scale = z((B, cap), dtype=torch.float32, **kw)
        self.k_rope = z((B, cap, max(desc.d_rope, 1)), dtype=torch.int16, **kw)
        sep = bool(desc.separate_v)
        self.v_nope = z((B, cap, desc.d_nope), dtype=torch.uint8, **kw) if sep else None
        self.v_scale = z((B, cap), dtype=torch.float32, **kw) if sep else None
        self.v_rope = z((B, cap, max(desc.d_rope, 1)), dtype=torch.int16, **kw) if sep else None
        Di = desc.idx_dim
        self.idx_codes = z((B, cap, Di // 2), dtype=torch.uint8, **kw) if Di else None
        self.idx_scales = z((B, cap, Di // 16), dtype=torch.uint8, **kw) if Di else None
        W, m = desc.window, desc.ratio
        self.win_k = z((B, max(W, 1), D), dtype=torch.int16, **kw)
        self.win_v = z((B, max(W, 1), D), dtype=torch.int16, **kw) if sep else None
        self.pend_k = z((B, m, D), dtype=torch.int16, **kw)
        self.pend_z = z((B, m, D), dtype=torch.int16, **kw)
        self.pend_v = z((B, m, D), dtype=torch.int16, **kw) if sep else None
        self.pend_u = z((B, m, max(Di, 8)), dtype=torch.int16, **kw) if Di else None
        self.pend_zu = z((B, m, max(Di, 8)), dtype=torch.int16, **kw) if Di else None
        self.n_tokens = z((B,), dtype=torch.int64, **kw)
        self.status = z((4,), dtype=torch.int32, **kw)
        self.struct = CacheStruct(
            KvPlanes(_ptr(self.k_nope), _ptr(self.k_scale), _ptr(self.k_rope)),
            KvPlanes(_ptr(self.v_nope), _ptr(self.v_scale), _ptr(self.v_rope)),
            _ptr(self.idx_codes), _ptr(self.idx_scales), _ptr(self.win_k), _ptr(self.win_v), _ptr(self.pend_k),
            _ptr(self.pend_v), _ptr(self.pend_z), _ptr(self.pend_u), _ptr(self.pend_zu), _ptr(self.n_tokens),
            _ptr(self.status))

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in vars(self).values() if isinstance(t, torch.Tensor))


# ----------------------------------------------------------------------------- entry points

def dsv4_compress_append(desc, cache, T, k, v, z, b, u=None, zu=None, bu=None, stream=None):
    return _check("dsv4_compress_append", lib.dsv4_compress_append(
        ctypes.byref(desc), ctypes.byref(cache.struct), T, _ptr(k), _ptr(v), _ptr(z), _ptr(b), _ptr(u), _ptr(zu),
        _ptr(bu), _stream(stream)))


def dsv4_index_topk(desc, cache, Hi, q_idx, w, k, topk, scores, ws, stream=None):
    return _check("dsv4_index_topk", lib.dsv4_index_topk(
        ctypes.byref(desc), ctypes.byref(cache.struct), Hi, _ptr(q_idx), _ptr(w), k, _ptr(topk), _ptr(scores),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def dsv4_csa_decode(desc, cache, H, q, sm_scale, topk, k, out, lse, ws, stream=None):
    return _check("dsv4_csa_decode", lib.dsv4_csa_decode(
        ctypes.byref(desc), ctypes.byref(cache.struct), H, _ptr(q), float(sm_scale), _ptr(topk), k, _ptr(out),
        _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def dsv4_hca_decode(desc, cache, H, q, sm_scale, out, lse, ws, stream=None):
    return _check("dsv4_hca_decode", lib.dsv4_hca_decode(
        ctypes.byref(desc), ctypes.byref(cache.struct), H, _ptr(q), float(sm_scale), _ptr(out), _ptr(lse),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def dsv4_hca_decode_static(desc, cache, H, q, sm_scale, out, lse, stream=None):
    return _check("dsv4_hca_decode_static", lib.dsv4_hca_decode_static(
        ctypes.byref(desc), ctypes.byref(cache.struct), H, _ptr(q), float(sm_scale), _ptr(out), _ptr(lse),
        _stream(stream)))


def dsv4_index_topk_multi(desc, cache, T, Hi, q_idx, w, k, topk, scores, ws, stream=None):
    return _check("dsv4_index_topk_multi", lib.dsv4_index_topk_multi(
        ctypes.byref(desc), ctypes.byref(cache.struct), T, Hi, _ptr(q_idx), _ptr(w), k, _ptr(topk), _ptr(scores),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def dsv4_csa_decode_multi(desc, cache, T, H, q, sm_scale, topk, k, span_k, span_v, out, lse, ws, stream=None):
    return _check("dsv4_csa_decode_multi", lib.dsv4_csa_decode_multi(
        ctypes.byref(desc), ctypes.byref(cache.struct), T, H, _ptr(q), float(sm_scale), _ptr(topk), k, _ptr(span_k),
        _ptr(span_v), _ptr(out), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def dsv4_hca_decode_multi(desc, cache, T, H, q, sm_scale, span_k, span_v, out, lse, ws, stream=None):
    return _check("dsv4_hca_decode_multi", lib.dsv4_hca_decode_multi(
        ctypes.byref(desc), ctypes.byref(cache.struct), T, H, _ptr(q), float(sm_scale), _ptr(span_k), _ptr(span_v),
        _ptr(out), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def dsv4_workspace_size_multi(desc, T, H, Hi, k):
    return int(lib.dsv4_workspace_size_multi(ctypes.byref(desc), T, H, Hi, k))


def workspace_multi(desc, T, H, Hi=0, k=0, device="cuda"):
    """Device workspace for T queries per sequence (dsv4_workspace_size_multi bytes)."""
    n = dsv4_workspace_size_multi(desc, T, H, Hi, k)
    if n == 0:
        raise Dsv4Error("dsv4_workspace_size_multi", ERR_INVALID_ARG)
    return torch.empty(n, dtype=torch.uint8, device=device)


def dsv4_workspace_size(desc, H, Hi, k):
    return int(lib.dsv4_workspace_size(ctypes.byref(desc), H, Hi, k))


def dsv4_decode_plan(desc, H, k):
    """Launch plan of a decode call (k: top-k width, 0 window-only CSA, -1 HCA) as a dict."""
    plan = (ctypes.c_int32 * 6)()
    _check("dsv4_decode_plan", lib.dsv4_decode_plan(ctypes.byref(desc), H, k, ctypes.cast(plan, ctypes.c_void_p)))
    return dict(zip(("tensor_core", "splits", "tile_rows", "tiles_per_split", "head_groups", "sms"), list(plan)))


def dsv4_project_streams(desc, cache, T, d_model, hidden, weight, rope_base, x, z, u, zu, stream=None):
    return _check("dsv4_project_streams", lib.dsv4_project_streams(
        ctypes.byref(desc), ctypes.byref(cache.struct), T, d_model, _ptr(hidden), _ptr(weight), float(rope_base),
        _ptr(x), _ptr(z), _ptr(u), _ptr(zu), _stream(stream)))


def dsv4_debug_force_timeout(on):
    return _check("dsv4_debug_force_timeout", lib.dsv4_debug_force_timeout(1 if on else 0))


def dsv4_read_status(cache, stream=None):
    return _check("dsv4_read_status", lib.dsv4_read_status(ctypes.byref(cache.struct), _stream(stream)))


def dsv4_quantize_kv_rows(y, rows, d_nope, d_rope, nope, scale, rope, stream=None):
    return _check("dsv4_quantize_kv_rows", lib.dsv4_quantize_kv_rows(
        _ptr(y), rows, d_nope, d_rope, _ptr(nope), _ptr(scale), _ptr(rope), _stream(stream)))


def dsv4_quantize_fp4_rows(y, rows, cols, codes, scales, stream=None):
    return _check("dsv4_quantize_fp4_rows", lib.dsv4_quantize_fp4_rows(
        _ptr(y), rows, cols, _ptr(codes), _ptr(scales), _stream(stream)))


def dsv4_pool_rows(x, z, b, blocks, ratio, dim, y, stream=None):
    return _check("dsv4_pool_rows", lib.dsv4_pool_rows(
        _ptr(x), _ptr(z), _ptr(b), blocks, ratio, dim, _ptr(y), _stream(stream)))


def workspace(desc, H, Hi=0, k=0, device="cuda"):
    """Device workspace for this layer (a torch uint8 tensor of dsv4_workspace_size bytes)."""
    n = dsv4_workspace_size(desc, H, Hi, k)
    if n == 0:
        raise Dsv4Error("dsv4_workspace_size", ERR_INVALID_ARG)
    return torch.empty(n, dtype=torch.uint8, device=device)
