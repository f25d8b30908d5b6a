"""ctypes binding of libcpattn.so (C ABI in include/cpattn.h).

Argument checking and marshalling only: tensors are passed as ``data_ptr()`` on the caller's
current CUDA stream.  Each function raises CpError on a non-OK status, with the library's own
message.  The library must be built (``__graft_entry__.build()``); there is no fallback.
"""

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

CP_OK, CP_ERR_INVALID_ARG, CP_ERR_UNSUPPORTED, CP_ERR_CUDA, CP_ERR_TIMEOUT = range(5)
CP_LAYOUT_CONTIGUOUS, CP_LAYOUT_STRIDED, CP_LAYOUT_TWO_BLOCK, CP_LAYOUT_BALANCED = 0, 1, 2, 3
CP_MAX_SEGMENTS = 2
CP_F32, CP_BF16 = 0, 1
CP_FLAG_KV_DESCENDING = 0x1
CP_FLAG_TEST_STALL = 0x100
CP_MAX_PARTIALS = 128
CP_MAX_CHUNKS = 64

_LAYOUTS = {"contiguous": CP_LAYOUT_CONTIGUOUS, "strided": CP_LAYOUT_STRIDED,
            "two_block": CP_LAYOUT_TWO_BLOCK, "balanced": CP_LAYOUT_BALANCED,
            CP_LAYOUT_CONTIGUOUS: CP_LAYOUT_CONTIGUOUS, CP_LAYOUT_STRIDED: CP_LAYOUT_STRIDED,
            CP_LAYOUT_TWO_BLOCK: CP_LAYOUT_TWO_BLOCK, CP_LAYOUT_BALANCED: CP_LAYOUT_BALANCED}


class CpError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"status {status}: {message}")
        self.status = status


class _PosMap(ctypes.Structure):
    _fields_ = [("base", ctypes.c_int64), ("stride", ctypes.c_int64)]


class _AttnDesc(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("in_dtype", ctypes.c_int32), ("o_dtype", ctypes.c_int32),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("sq", ctypes.c_int64), ("skv", ctypes.c_int64),
        ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("d", ctypes.c_int32),
        ("causal", ctypes.c_int32), ("scale", ctypes.c_float), ("flags", ctypes.c_int32),
        ("q_pos", _PosMap), ("kv_pos", _PosMap),
        ("status", ctypes.c_void_p), ("wait_timeout_ms", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class _AttnBwdDesc(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("d_o", ctypes.c_void_p), ("in_dtype", ctypes.c_int32), ("flags", ctypes.c_int32),
        ("aux", ctypes.c_void_p), ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p),
        ("dv", ctypes.c_void_p), ("sq", ctypes.c_int64), ("skv", ctypes.c_int64),
        ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("d", ctypes.c_int32),
        ("causal", ctypes.c_int32), ("scale", ctypes.c_float), ("wait_timeout_ms", ctypes.c_int32),
        ("q_pos", _PosMap), ("kv_pos", _PosMap), ("status", ctypes.c_void_p),
    ]


class _KvBwdChunk(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dk", ctypes.c_void_p),
                ("dv", ctypes.c_void_p), ("skv", ctypes.c_int64), ("kv_pos", _PosMap)]


class _KvChunk(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("skv", ctypes.c_int64),
                ("kv_pos", _PosMap)]


@dataclass(frozen=True)
class PosMap:
    """Affine global positions of a shard or chunk: pos(i) = base + stride * i."""
    base: int
    stride: int


_lib = None


def library_path():
    return _build.LIB


def load_library():
    """Load libcpattn.so once and declare its signatures; raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise CpError(CP_ERR_UNSUPPORTED, f"{path} is not built; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.cp_version.restype = i32
    lib.cp_version.argtypes = []
    lib.cp_last_error.restype = ctypes.c_char_p
    lib.cp_last_error.argtypes = []
    lib.cp_shard_layout.restype = i32
    lib.cp_shard_layout.argtypes = [i64, i32, i32, i32, ctypes.POINTER(_PosMap), vp, vp]
    lib.cp_shard_segments.restype = i32
    lib.cp_shard_segments.argtypes = [i64, i32, i32, i32, ctypes.POINTER(_PosMap),
                                      ctypes.POINTER(i64), ctypes.POINTER(i32), vp, vp]
    lib.cp_partial_attn.restype = i32
    lib.cp_partial_attn.argtypes = [ctypes.POINTER(_AttnDesc), vp]
    lib.cp_partial_attn_chunks.restype = i32
    lib.cp_partial_attn_chunks.argtypes = [ctypes.POINTER(_AttnDesc), i32, ctypes.POINTER(_KvChunk), vp]
    lib.cp_attn_bwd_prep.restype = i32
    lib.cp_attn_bwd_prep.argtypes = [vp, i32, vp, i32, vp, i64, i32, i32, vp, vp]
    lib.cp_partial_attn_bwd.restype = i32
    lib.cp_partial_attn_bwd.argtypes = [ctypes.POINTER(_AttnBwdDesc), vp]
    lib.cp_partial_attn_bwd_chunks.restype = i32
    lib.cp_partial_attn_bwd_chunks.argtypes = [ctypes.POINTER(_AttnBwdDesc), i32, ctypes.POINTER(_KvBwdChunk), vp]
    lib.cp_partial_attn_bwd_noalloc.restype = i32
    lib.cp_partial_attn_bwd_noalloc.argtypes = [ctypes.POINTER(_AttnBwdDesc), vp, i32, vp, vp]
    lib.cp_merge_partials.restype = i32
    lib.cp_merge_partials.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), i64, i32, i32,
                                      vp, i32, vp, vp]
    lib.cp_ulysses_reshard.restype = i32
    lib.cp_ulysses_reshard.argtypes = [i32, i32, i64, i32, ctypes.POINTER(i32), i32, i32, i32,
                                       ctypes.POINTER(vp), ctypes.POINTER(vp), vp]
    _lib = lib
    return lib


def _check(status):
    if status != CP_OK:
        msg = load_library().cp_last_error().decode(errors="replace")
        raise CpError(status, msg)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dtype_code(dt):
    if dt == torch.float32:
        return CP_F32
    if dt == torch.bfloat16:
        return CP_BF16
    raise CpError(CP_ERR_INVALID_ARG, f"unsupported dtype {dt}")


def _need_cuda(t, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise CpError(CP_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise CpError(CP_ERR_INVALID_ARG, f"{name} must be contiguous")


def version():
    return load_library().cp_version()


def shard_layout(seq_len, cp, rank, kind="contiguous", positions=False, device=None, stream=None):
    """Affine position map of rank ``rank``; with ``positions=True`` also an int32 CUDA tensor
    of the positions, filled by the library's kernel."""
    lib = load_library()
    m = _PosMap()
    out = None
    ptr = None
    if positions:
        if seq_len % cp != 0 or cp <= 0:
            _check(lib.cp_shard_layout(seq_len, cp, rank, _LAYOUTS.get(kind, -1), ctypes.byref(m),
                                       None, None))
        device = device or torch.device("cuda", torch.cuda.current_device())
        out = torch.empty(seq_len // cp, dtype=torch.int32, device=device)
        ptr = ctypes.c_void_p(out.data_ptr())
    _check(lib.cp_shard_layout(int(seq_len), int(cp), int(rank), _LAYOUTS.get(kind, -1),
                               ctypes.byref(m), ptr, _stream(stream) if positions else None))
    pm = PosMap(m.base, m.stride)
    return (pm, out) if positions else pm


def shard_segments(seq_len, cp, rank, kind="contiguous", positions=False, device=None, stream=None):
    """The shard of rank ``rank`` as a list of ``(PosMap, length)`` affine segments in local
    order (two for the two-block layout, one otherwise; the balanced layout's shards differ in
    length); with ``positions=True`` also an int32 CUDA tensor of every local token's position,
    filled by the library's kernel."""
    lib = load_library()
    maps = (_PosMap * CP_MAX_SEGMENTS)()
    lens = (ctypes.c_int64 * CP_MAX_SEGMENTS)()
    n = ctypes.c_int32(0)
    out = None
    ptr = None
    if positions:
        # validate first so that a bad shape fails before anything is allocated
        _check(lib.cp_shard_segments(int(seq_len), int(cp), int(rank), _LAYOUTS.get(kind, -1),
                                     maps, lens, ctypes.byref(n), None, None))
        device = device or torch.device("cuda", torch.cuda.current_device())
        out = torch.empty(sum(int(lens[i]) for i in range(n.value)), dtype=torch.int32, device=device)
        ptr = ctypes.c_void_p(out.data_ptr())
    _check(lib.cp_shard_segments(int(seq_len), int(cp), int(rank), _LAYOUTS.get(kind, -1),
                                 maps, lens, ctypes.byref(n), ptr,
                                 _stream(stream) if positions else None))
    segs = [(PosMap(maps[i].base, maps[i].stride), int(lens[i])) for i in range(n.value)]
    return (segs, out) if positions else segs


def sub_chunk_map(shard: PosMap, index: int, length: int) -> PosMap:
    """Map of local rows [index*length, (index+1)*length) of a shard."""
    return PosMap(shard.base + shard.stride * index * length, shard.stride)


def partial_attn(q, k, v, q_pos: PosMap, kv_pos: PosMap, causal=True, scale=0.0, o=None,
                 lse=None, o_dtype=None, flags=0, status=None, wait_timeout_ms=0, stream=None):
    """(O, LSE) partial of query shard ``q`` [Sq, Hq, D] against one KV chunk [Skv, Hkv, D]."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need_cuda(t, n)
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape:
        raise CpError(CP_ERR_INVALID_ARG, "q must be [Sq, Hq, D]; k and v [Skv, Hkv, D]")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise CpError(CP_ERR_INVALID_ARG, "q, k, v must share a dtype")
    sq, hq, d = q.shape
    skv, hkv, dk = k.shape
    if dk != d:
        raise CpError(CP_ERR_INVALID_ARG, "head_dim mismatch")
    if o is None:
        o = torch.empty((sq, hq, d), dtype=o_dtype or torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((sq, hq), dtype=torch.float32, device=q.device)
    _need_cuda(o, "o")
    _need_cuda(lse, "lse")
    if tuple(o.shape) != (sq, hq, d) or tuple(lse.shape) != (sq, hq) or lse.dtype != torch.float32:
        raise CpError(CP_ERR_INVALID_ARG, "o must be [Sq, Hq, D]; lse fp32 [Sq, Hq]")
    desc = _AttnDesc()
    desc.q, desc.k, desc.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    desc.in_dtype = _dtype_code(q.dtype)
    desc.o_dtype = _dtype_code(o.dtype)
    desc.o, desc.lse = o.data_ptr(), lse.data_ptr()
    desc.sq, desc.skv, desc.hq, desc.hkv, desc.d = sq, skv, hq, hkv, d
    desc.causal = 1 if causal else 0
    desc.scale = float(scale)
    desc.flags = int(flags)
    desc.q_pos = _PosMap(q_pos.base, q_pos.stride)
    desc.kv_pos = _PosMap(kv_pos.base, kv_pos.stride)
    if status is not None:
        _need_cuda(status, "status")
        if status.dtype != torch.int32:
            raise CpError(CP_ERR_INVALID_ARG, "status must be int32")
        desc.status = status.data_ptr()
    desc.wait_timeout_ms = int(wait_timeout_ms)
    _check(lib.cp_partial_attn(ctypes.byref(desc), _stream(stream)))
    return o, lse


def partial_attn_chunks(q, chunks, q_pos: PosMap, causal=True, scale=0.0, o=None, lse=None,
                        o_dtype=None, flags=0, status=None, wait_timeout_ms=0, stream=None):
    """Attention of query shard ``q`` against KV chunks consumed in the given (arrival) order in
    one launch, the running softmax state carried across them.

    chunks: list of (k, v, kv_pos) with k, v [Skv_c, Hkv, D] CUDA tensors and kv_pos a PosMap.
    Returns (o, lse) over the union of the chunks' keys.
    """
    lib = load_library()
    _need_cuda(q, "q")
    n = len(chunks)
    if n < 1 or n > CP_MAX_CHUNKS:
        raise CpError(CP_ERR_INVALID_ARG, f"between 1 and {CP_MAX_CHUNKS} chunks")
    sq, hq, d = q.shape
    hkv = None
    arr = (_KvChunk * n)()
    for i, (k, v, kv_pos) in enumerate(chunks):
        _need_cuda(k, "k")
        _need_cuda(v, "v")
        if k.dim() != 3 or v.shape != k.shape or k.shape[2] != d or k.dtype != q.dtype or v.dtype != q.dtype:
            raise CpError(CP_ERR_INVALID_ARG, "each chunk's k and v must be [Skv, Hkv, D] in q's dtype")
        if hkv is None:
            hkv = k.shape[1]
        elif k.shape[1] != hkv:
            raise CpError(CP_ERR_INVALID_ARG, "all chunks must have the same KV head count")
        arr[i].k, arr[i].v, arr[i].skv = k.data_ptr(), v.data_ptr(), k.shape[0]
        arr[i].kv_pos = _PosMap(kv_pos.base, kv_pos.stride)
    if o is None:
        o = torch.empty((sq, hq, d), dtype=o_dtype or torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((sq, hq), dtype=torch.float32, device=q.device)
    _need_cuda(o, "o")
    _need_cuda(lse, "lse")
    if tuple(o.shape) != (sq, hq, d) or tuple(lse.shape) != (sq, hq) or lse.dtype != torch.float32:
        raise CpError(CP_ERR_INVALID_ARG, "o must be [Sq, Hq, D]; lse fp32 [Sq, Hq]")
    desc = _AttnDesc()
    desc.q = q.data_ptr()
    desc.in_dtype = _dtype_code(q.dtype)
    desc.o_dtype = _dtype_code(o.dtype)
    desc.o, desc.lse = o.data_ptr(), lse.data_ptr()
    desc.sq, desc.hq, desc.hkv, desc.d = sq, hq, hkv, d
    desc.causal = 1 if causal else 0
    desc.scale = float(scale)
    desc.flags = int(flags)
    desc.q_pos = _PosMap(q_pos.base, q_pos.stride)
    if status is not None:
        _need_cuda(status, "status")
        desc.status = status.data_ptr()
    desc.wait_timeout_ms = int(wait_timeout_ms)
    _check(lib.cp_partial_attn_chunks(ctypes.byref(desc), n, arr, _stream(stream)))
    return o, lse


def bwd_aux_floats(sq, hq):
    """Size of the per-row backward workspace (``CP_BWD_AUX_FLOATS``)."""
    return 2 * int(hq) * ((int(sq) + 127) // 128 * 128)


def attn_bwd_prep(o, d_o, lse, aux=None, stream=None):
    """Per-row quantities of the backward pass of a query shard from its final ``o`` and ``lse``
    and the output gradient ``d_o`` (all [Sq, Hq, D] / [Sq, Hq]); returns the fp32 workspace."""
    lib = load_library()
    for t, n in ((o, "o"), (d_o, "d_o"), (lse, "lse")):
        _need_cuda(t, n)
    if o.dim() != 3 or d_o.shape != o.shape or tuple(lse.shape) != tuple(o.shape[:2]):
        raise CpError(CP_ERR_INVALID_ARG, "o and d_o must be [Sq, Hq, D], lse [Sq, Hq]")
    if lse.dtype != torch.float32:
        raise CpError(CP_ERR_INVALID_ARG, "lse must be fp32")
    sq, hq, d = o.shape
    if aux is None:
        aux = torch.empty(bwd_aux_floats(sq, hq), dtype=torch.float32, device=o.device)
    _need_cuda(aux, "aux")
    if aux.dtype != torch.float32 or aux.numel() < bwd_aux_floats(sq, hq):
        raise CpError(CP_ERR_INVALID_ARG, "aux must be fp32 with bwd_aux_floats(sq, hq) elements")
    _check(lib.cp_attn_bwd_prep(ctypes.c_void_p(o.data_ptr()), _dtype_code(o.dtype),
                                ctypes.c_void_p(d_o.data_ptr()), _dtype_code(d_o.dtype),
                                ctypes.c_void_p(lse.data_ptr()), sq, hq, d,
                                ctypes.c_void_p(aux.data_ptr()), _stream(stream)))
    return aux


def partial_attn_bwd(q, k, v, d_o, aux, q_pos: PosMap, kv_pos: PosMap, dq, dk, dv, causal=True,
                     scale=0.0, status=None, wait_timeout_ms=0, flags=0, stream=None):
    """Adds one (query shard, KV chunk) pair's share of the attention gradients into ``dq``
    [Sq, Hq, D] and ``dk``, ``dv`` [Skv, Hkv, D] (fp32, accumulated in place)."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (d_o, "d_o"), (aux, "aux"), (dq, "dq"), (dk, "dk"),
                 (dv, "dv")):
        _need_cuda(t, n)
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape or d_o.shape != q.shape:
        raise CpError(CP_ERR_INVALID_ARG, "q, d_o must be [Sq, Hq, D]; k and v [Skv, Hkv, D]")
    if not (q.dtype == k.dtype == v.dtype == d_o.dtype):
        raise CpError(CP_ERR_INVALID_ARG, "q, k, v, d_o must share a dtype")
    sq, hq, d = q.shape
    skv, hkv, dk_ = k.shape
    if dk_ != d:
        raise CpError(CP_ERR_INVALID_ARG, "head_dim mismatch")
    if dq.shape != q.shape or dk.shape != k.shape or dv.shape != k.shape or \
            any(t.dtype != torch.float32 for t in (dq, dk, dv, aux)):
        raise CpError(CP_ERR_INVALID_ARG, "dq, dk, dv must be fp32 and shaped like q, k, v")
    if aux.numel() < bwd_aux_floats(sq, hq):
        raise CpError(CP_ERR_INVALID_ARG, "aux is smaller than bwd_aux_floats(sq, hq)")
    desc = _AttnBwdDesc()
    desc.q, desc.k, desc.v, desc.d_o = q.data_ptr(), k.data_ptr(), v.data_ptr(), d_o.data_ptr()
    desc.in_dtype = _dtype_code(q.dtype)
    desc.aux = aux.data_ptr()
    desc.dq, desc.dk, desc.dv = dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    desc.sq, desc.skv, desc.hq, desc.hkv, desc.d = sq, skv, hq, hkv, d
    desc.causal = 1 if causal else 0
    desc.scale = float(scale)
    desc.q_pos = _PosMap(q_pos.base, q_pos.stride)
    desc.kv_pos = _PosMap(kv_pos.base, kv_pos.stride)
    if status is not None:
        _need_cuda(status, "status")
        if status.dtype != torch.int32:
            raise CpError(CP_ERR_INVALID_ARG, "status must be int32")
        desc.status = status.data_ptr()
    desc.wait_timeout_ms = int(wait_timeout_ms)
    desc.flags = int(flags)
    _check(lib.cp_partial_attn_bwd(ctypes.byref(desc), _stream(stream)))
    return dq, dk, dv


# Largest workspace partial_attn_bwd_noalloc can use (``CP_NOALLOC_AUX_MAX_FLOATS``).
NOALLOC_AUX_MAX_FLOATS = 4194304


def partial_attn_bwd_noalloc(q, k, v, d_o, o, lse, q_pos: PosMap, kv_pos: PosMap, dq, dk, dv, causal=True,
                             scale=0.0, status=None, wait_timeout_ms=0, stream=None):
    """``attn_bwd_prep`` and ``partial_attn_bwd`` in one call whose per-row workspace lives in the
    library's own fixed device array, so that nothing is allocated: for callers that may not
    allocate device memory.  ``o`` and ``lse`` are the shard's final output and LSE; the gradients
    are accumulated into ``dq``, ``dk``, ``dv`` as by ``partial_attn_bwd``.  Calls that may overlap
    on the GPU share the array and race; calls on one stream are safe.  Raises ``CpError`` when
    ``bwd_aux_floats(Sq, Hq)`` is above ``NOALLOC_AUX_MAX_FLOATS``."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (d_o, "d_o"), (o, "o"), (lse, "lse"), (dq, "dq"), (dk, "dk"),
                 (dv, "dv")):
        _need_cuda(t, n)
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape or d_o.shape != q.shape or o.shape != q.shape:
        raise CpError(CP_ERR_INVALID_ARG, "q, d_o, o must be [Sq, Hq, D]; k and v [Skv, Hkv, D]")
    if not (q.dtype == k.dtype == v.dtype == d_o.dtype):
        raise CpError(CP_ERR_INVALID_ARG, "q, k, v, d_o must share a dtype")
    sq, hq, d = q.shape
    skv, hkv, dk_ = k.shape
    if dk_ != d:
        raise CpError(CP_ERR_INVALID_ARG, "head_dim mismatch")
    if tuple(lse.shape) != (sq, hq) or lse.dtype != torch.float32:
        raise CpError(CP_ERR_INVALID_ARG, "lse must be fp32 [Sq, Hq]")
    if dq.shape != q.shape or dk.shape != k.shape or dv.shape != k.shape or \
            any(t.dtype != torch.float32 for t in (dq, dk, dv)):
        raise CpError(CP_ERR_INVALID_ARG, "dq, dk, dv must be fp32 and shaped like q, k, v")
    desc = _AttnBwdDesc()
    desc.q, desc.k, desc.v, desc.d_o = q.data_ptr(), k.data_ptr(), v.data_ptr(), d_o.data_ptr()
    desc.in_dtype = _dtype_code(q.dtype)
    desc.aux = None
    desc.dq, desc.dk, desc.dv = dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    desc.sq, desc.skv, desc.hq, desc.hkv, desc.d = sq, skv, hq, hkv, d
    desc.causal = 1 if causal else 0
    desc.scale = float(scale)
    desc.q_pos = _PosMap(q_pos.base, q_pos.stride)
    desc.kv_pos = _PosMap(kv_pos.base, kv_pos.stride)
    if status is not None:
        _need_cuda(status, "status")
        if status.dtype != torch.int32:
            raise CpError(CP_ERR_INVALID_ARG, "status must be int32")
        desc.status = status.data_ptr()
    desc.wait_timeout_ms = int(wait_timeout_ms)
    _check(lib.cp_partial_attn_bwd_noalloc(ctypes.byref(desc), ctypes.c_void_p(o.data_ptr()), _dtype_code(o.dtype),
                                           ctypes.c_void_p(lse.data_ptr()), _stream(stream)))
    return dq, dk, dv


def partial_attn_bwd_chunks(q, d_o, aux, q_pos: PosMap, chunks, dq, causal=True, scale=0.0, status=None,
                            wait_timeout_ms=0, flags=0, stream=None):
    """The backward of query shard ``q`` against a list of chunks ``(k, v, kv_pos, dk, dv)`` in one
    call: the same as ``partial_attn_bwd`` per chunk (accumulating into ``dq`` and each chunk's
    ``dk``, ``dv``), with one launch per 32 chunks."""
    lib = load_library()
    for t, n in ((q, "q"), (d_o, "d_o"), (aux, "aux"), (dq, "dq")):
        _need_cuda(t, n)
    if q.dim() != 3 or d_o.shape != q.shape or dq.shape != q.shape or dq.dtype != torch.float32:
        raise CpError(CP_ERR_INVALID_ARG, "q, d_o [Sq, Hq, D]; dq fp32 of the same shape")
    sq, hq, d = q.shape
    if aux.dtype != torch.float32 or aux.numel() < bwd_aux_floats(sq, hq):
        raise CpError(CP_ERR_INVALID_ARG, "aux must be fp32 with bwd_aux_floats(sq, hq) elements")
    if not 1 <= len(chunks) <= CP_MAX_CHUNKS:
        raise CpError(CP_ERR_INVALID_ARG, f"1..{CP_MAX_CHUNKS} chunks expected")
    arr = (_KvBwdChunk * len(chunks))()
    hkv = None
    for i, (k, v, kv_pos, dk, dv) in enumerate(chunks):
        for t, n in ((k, "k"), (v, "v"), (dk, "dk"), (dv, "dv")):
            _need_cuda(t, n)
        if k.dim() != 3 or v.shape != k.shape or k.shape[2] != d or k.dtype != q.dtype or v.dtype != q.dtype:
            raise CpError(CP_ERR_INVALID_ARG, f"chunk {i}: k and v must be [Skv, Hkv, D] of q's dtype")
        if dk.shape != k.shape or dv.shape != k.shape or dk.dtype != torch.float32 or dv.dtype != torch.float32:
            raise CpError(CP_ERR_INVALID_ARG, f"chunk {i}: dk and dv must be fp32 shaped like k")
        if hkv is None:
            hkv = k.shape[1]
        elif k.shape[1] != hkv:
            raise CpError(CP_ERR_INVALID_ARG, "every chunk must have the same KV head count")
        arr[i].k, arr[i].v, arr[i].dk, arr[i].dv = k.data_ptr(), v.data_ptr(), dk.data_ptr(), dv.data_ptr()
        arr[i].skv = k.shape[0]
        arr[i].kv_pos = _PosMap(kv_pos.base, kv_pos.stride)
    desc = _AttnBwdDesc()
    desc.q, desc.d_o = q.data_ptr(), d_o.data_ptr()
    desc.in_dtype = _dtype_code(q.dtype)
    desc.aux = aux.data_ptr()
    desc.dq = dq.data_ptr()
    desc.sq, desc.hq, desc.hkv, desc.d = sq, hq, hkv, d
    desc.causal = 1 if causal else 0
    desc.scale = float(scale)
    desc.q_pos = _PosMap(q_pos.base, q_pos.stride)
    if status is not None:
        _need_cuda(status, "status")
        if status.dtype != torch.int32:
            raise CpError(CP_ERR_INVALID_ARG, "status must be int32")
        desc.status = status.data_ptr()
    desc.wait_timeout_ms = int(wait_timeout_ms)
    desc.flags = int(flags)
    _check(lib.cp_partial_attn_bwd_chunks(ctypes.byref(desc), len(chunks), arr, _stream(stream)))
    return dq


def merge_partials(o_parts, lse_parts, out_dtype=torch.bfloat16, o=None, lse=None, stream=None):
    """Exact attention from partials (lists of fp32 [Sq, H, D] and fp32 [Sq, H])."""
    lib = load_library()
    n = len(o_parts)
    if n != len(lse_parts) or n < 1:
        raise CpError(CP_ERR_INVALID_ARG, "need matching non-empty partial lists")
    if n > CP_MAX_PARTIALS:
        raise CpError(CP_ERR_INVALID_ARG, f"at most {CP_MAX_PARTIALS} partials")
    sq, h, d = o_parts[0].shape
    for x, y in zip(o_parts, lse_parts):
        _need_cuda(x, "o part")
        _need_cuda(y, "lse part")
        if x.dtype != torch.float32 or y.dtype != torch.float32:
            raise CpError(CP_ERR_INVALID_ARG, "partials must be fp32")
        if tuple(x.shape) != (sq, h, d) or tuple(y.shape) != (sq, h):
            raise CpError(CP_ERR_INVALID_ARG, "partials must share shape [Sq, H, D] / [Sq, H]")
    if o is None:
        o = torch.empty((sq, h, d), dtype=out_dtype, device=o_parts[0].device)
    if lse is None:
        lse = torch.empty((sq, h), dtype=torch.float32, device=o_parts[0].device)
    _need_cuda(o, "o")
    _need_cuda(lse, "lse")
    arr_o = (ctypes.c_void_p * n)(*[x.data_ptr() for x in o_parts])
    arr_l = (ctypes.c_void_p * n)(*[y.data_ptr() for y in lse_parts])
    _check(lib.cp_merge_partials(n, arr_o, arr_l, sq, h, d, ctypes.c_void_p(o.data_ptr()),
                                 _dtype_code(o.dtype), ctypes.c_void_p(lse.data_ptr()),
                                 _stream(stream)))
    return o, lse


def ulysses_reshard(direction, tensors, cp, seq_len, layout="contiguous", out=None, stream=None):
    """Reshard ``tensors`` (a list over tensor kinds, each a list of cp per-rank tensors).

    direction "seq_to_head": inputs [S/cp, H_t, D] -> outputs [S, H_t/cp, D];
    direction "head_to_seq": inputs [S, H_t/cp, D] -> outputs [S/cp, H_t, D].
    Returns the outputs in the same nesting.
    """
    lib = load_library()
    dirc = {"seq_to_head": 0, "head_to_seq": 1}[direction]
    nt = len(tensors)
    heads = []
    outs = []
    for t, per_rank in enumerate(tensors):
        if len(per_rank) != cp:
            raise CpError(CP_ERR_INVALID_ARG, "one tensor per rank expected")
        x0 = per_rank[0]
        d = x0.shape[2]
        h_t = x0.shape[1] if dirc == 0 else x0.shape[1] * cp
        heads.append(h_t)
        for x in per_rank:
            _need_cuda(x, "reshard input")
        if out is not None:
            outs.append(out[t])
        elif dirc == 0:
            outs.append([torch.empty((seq_len, h_t // cp, d), dtype=x0.dtype, device=x0.device)
                         for _ in range(cp)])
        else:
            outs.append([torch.empty((seq_len // cp, h_t, d), dtype=x0.dtype, device=x0.device)
                         for _ in range(cp)])
    d = tensors[0][0].shape[2]
    dtype = tensors[0][0].dtype
    arr_in = (ctypes.c_void_p * (nt * cp))(*[x.data_ptr() for per in tensors for x in per])
    arr_out = (ctypes.c_void_p * (nt * cp))(*[y.data_ptr() for per in outs for y in per])
    arr_h = (ctypes.c_int32 * nt)(*heads)
    _check(lib.cp_ulysses_reshard(dirc, cp, seq_len, nt, arr_h, d, _dtype_code(dtype),
                                  _LAYOUTS[layout], arr_in, arr_out, _stream(stream)))
    return outs
