"""The C ABI library: it loads, exports every function include/cpattn.h declares, and rejects
invalid arguments on the host (no GPU work is issued by any of these calls)."""

import ctypes

import pytest

import helpers

helpers.ensure_built()

import context_blockwise_attention_gb300 as cpa  # noqa: E402
from context_blockwise_attention_gb300 import api  # noqa: E402


def test_exports_every_declared_function():
    declared = helpers.header_functions()
    assert {"cp_shard_layout", "cp_partial_attn", "cp_merge_partials", "cp_ulysses_reshard",
            "cp_last_error", "cp_version"} <= set(declared)
    raw = ctypes.CDLL(cpa.library_path())
    for name in declared:
        assert hasattr(raw, name), f"{name} declared in cpattn.h but not exported"


def test_version():
    assert cpa.version() == 4


def test_desc_layout_matches_header():
    # the ctypes mirror must match the C struct size (pointers 8, int64 8, int32/float 4)
    assert ctypes.sizeof(api._AttnDesc) == 136
    assert ctypes.sizeof(api._PosMap) == 16
    assert ctypes.sizeof(api._KvChunk) == 40


def _layout(seq, cp, rank, kind):
    lib = cpa.load_library()
    m = api._PosMap()
    st = lib.cp_shard_layout(seq, cp, rank, kind, ctypes.byref(m), None, None)
    return st, m


@pytest.mark.parametrize("seq,cp,rank,kind", [
    (100, 8, 0, 0),   # not divisible
    (64, 0, 0, 0),    # cp 0
    (64, 4, 4, 0),    # rank out of range
    (64, 4, -1, 1),
    (-8, 4, 0, 0),
    (64, 4, 0, 7),    # unknown kind
])
def test_layout_rejects(seq, cp, rank, kind):
    st, _ = _layout(seq, cp, rank, kind)
    assert st == api.CP_ERR_INVALID_ARG
    assert cpa.load_library().cp_last_error()


def test_layout_host_map_page_examples():
    # host-only part (no positions buffer): the affine map
    st, m = _layout(32768, 4, 1, api.CP_LAYOUT_CONTIGUOUS)
    assert st == 0 and (m.base, m.stride) == (8192, 1)
    st, m = _layout(64, 4, 1, api.CP_LAYOUT_STRIDED)
    assert st == 0 and (m.base, m.stride) == (1, 4)


def _desc(**kw):
    d = api._AttnDesc()
    d.q = d.k = d.v = 0x1000
    d.o = 0x2000
    d.lse = 0x3000
    d.in_dtype = api.CP_BF16
    d.o_dtype = api.CP_F32
    d.sq, d.skv, d.hq, d.hkv, d.d = 128, 128, 8, 2, 128
    d.causal = 1
    d.q_pos = api._PosMap(0, 1)
    d.kv_pos = api._PosMap(0, 1)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("field,value", [
    ("d", 96), ("hq", 5), ("hkv", 0), ("in_dtype", 5), ("o_dtype", 9), ("causal", 2),
    ("q", 0), ("k", 0), ("o", 0), ("lse", 0), ("q", 0x1008), ("sq", -1), ("flags", 0x40),
    ("q_pos", api._PosMap(0, 0)), ("kv_pos", api._PosMap(-5, 1)), ("scale", -1.0),
    ("wait_timeout_ms", -3),
    # global positions must stay below 2e9: the shard's last position, then the chunk's
    ("q_pos", api._PosMap(2_000_000_000 - 100, 1)), ("kv_pos", api._PosMap(7, 16_000_000)),
])
def test_partial_attn_rejects(field, value):
    lib = cpa.load_library()
    d = _desc(**{field: value})
    assert lib.cp_partial_attn(ctypes.byref(d), None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_last_error()


def test_partial_attn_null_desc():
    assert cpa.load_library().cp_partial_attn(None, None) == api.CP_ERR_INVALID_ARG


def test_merge_rejects():
    lib = cpa.load_library()
    arr = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    out = ctypes.c_void_p(0x4000)
    assert lib.cp_merge_partials(0, arr, arr, 8, 2, 64, out, 0, None, None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_merge_partials(129, arr, arr, 8, 2, 64, out, 0, None, None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_merge_partials(2, arr, arr, 8, 2, 48, out, 0, None, None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_merge_partials(2, arr, arr, 8, 2, 64, out, 3, None, None) == api.CP_ERR_INVALID_ARG
    bad = (ctypes.c_void_p * 2)(0x1000, 0)
    assert lib.cp_merge_partials(2, bad, arr, 8, 2, 64, out, 0, None, None) == api.CP_ERR_INVALID_ARG


def test_reshard_rejects():
    lib = cpa.load_library()
    ptrs = (ctypes.c_void_p * 4)(0x1000, 0x2000, 0x3000, 0x4000)
    heads = (ctypes.c_int32 * 1)(8)
    ok_args = dict(dir=0, cp=4, seq=64, nt=1, d=64, dtype=1, layout=0)

    def call(**kw):
        a = dict(ok_args, **kw)
        return lib.cp_ulysses_reshard(a["dir"], a["cp"], a["seq"], a["nt"], heads, a["d"],
                                      a["dtype"], a["layout"], ptrs, ptrs, None)
    assert call(dir=2) == api.CP_ERR_INVALID_ARG
    assert call(seq=66) == api.CP_ERR_INVALID_ARG
    assert call(cp=3) == api.CP_ERR_INVALID_ARG        # 8 heads not divisible by 3 (and 66 % 3)
    assert call(dtype=4) == api.CP_ERR_INVALID_ARG
    assert call(layout=3) == api.CP_ERR_INVALID_ARG
    assert call(nt=0) == api.CP_ERR_INVALID_ARG
    heads[0] = 6  # not a multiple of cp=4
    assert call() == api.CP_ERR_INVALID_ARG


def test_python_wrapper_rejects_cpu_tensors():
    import torch
    q = torch.zeros(4, 2, 64)
    with pytest.raises(cpa.CpError):
        cpa.partial_attn(q, q, q, cpa.PosMap(0, 1), cpa.PosMap(0, 1))


def test_partial_attn_chunks_rejects():
    lib = cpa.load_library()
    d = _desc()
    ch = (api._KvChunk * 2)()
    for c in ch:
        c.k, c.v, c.skv, c.kv_pos = 0x1000, 0x2000, 128, api._PosMap(0, 1)
    assert lib.cp_partial_attn_chunks(ctypes.byref(d), 0, ch, None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_partial_attn_chunks(ctypes.byref(d), 65, ch, None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_partial_attn_chunks(ctypes.byref(d), 2, None, None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_partial_attn_chunks(None, 2, ch, None) == api.CP_ERR_INVALID_ARG
    ch[1].kv_pos = api._PosMap(0, 0)
    assert lib.cp_partial_attn_chunks(ctypes.byref(d), 2, ch, None) == api.CP_ERR_INVALID_ARG
    ch[1].kv_pos = api._PosMap(0, 1)
    ch[1].k = 0
    assert lib.cp_partial_attn_chunks(ctypes.byref(d), 2, ch, None) == api.CP_ERR_INVALID_ARG
    ch[1].k = 0x1008
    assert lib.cp_partial_attn_chunks(ctypes.byref(d), 2, ch, None) == api.CP_ERR_INVALID_ARG
    assert b"chunk 1" in lib.cp_last_error()


def _segments(seq, cp, rank, kind):
    lib = cpa.load_library()
    maps = (api._PosMap * api.CP_MAX_SEGMENTS)()
    lens = (ctypes.c_int64 * api.CP_MAX_SEGMENTS)()
    n = ctypes.c_int32(-1)
    st = lib.cp_shard_segments(seq, cp, rank, kind, maps, lens, ctypes.byref(n), None, None)
    return st, [(maps[i].base, maps[i].stride, lens[i]) for i in range(max(n.value, 0))]


@pytest.mark.parametrize("seq,cp,rank,kind", [
    (60, 4, 0, 2),    # two blocks need seq % (2 cp) == 0
    (12, 8, 0, 2),    # not even a multiple of cp
    (64, 4, 4, 2),
    (64, 4, 0, 9),
])
def test_segments_reject(seq, cp, rank, kind):
    st, _ = _segments(seq, cp, rank, kind)
    assert st == api.CP_ERR_INVALID_ARG and cpa.load_library().cp_last_error()


def test_segments_reject_null_outputs_and_single_map_call():
    lib = cpa.load_library()
    maps = (api._PosMap * api.CP_MAX_SEGMENTS)()
    n = ctypes.c_int32()
    assert lib.cp_shard_segments(64, 4, 0, 2, maps, None, ctypes.byref(n), None, None) == \
        api.CP_ERR_INVALID_ARG
    # the two-block split is not one affine map
    assert _layout(64, 4, 0, api.CP_LAYOUT_TWO_BLOCK)[0] == api.CP_ERR_INVALID_ARG


def test_segments_host_maps_equal_oracle_positions():
    # host-only: the segments' affine maps, expanded, are the oracle's positions exactly
    import numpy as np
    import oracle
    for kind_name, kind in (("contiguous", 0), ("strided", 1), ("two_block", 2), ("balanced", 3)):
        for seq, cp in ((64, 4), (48, 8), (32768, 8), (131072, 4), (16, 1), (65537, 7)):
            if kind != 3 and seq % (2 * cp if kind == 2 else cp):
                continue
            for r in range(cp):
                st, segs = _segments(seq, cp, r, kind)
                assert st == 0
                assert len(segs) == (2 if kind == 2 else 1)
                got = np.concatenate([b + s * np.arange(n, dtype=np.int64) for b, s, n in segs])
                assert np.array_equal(got, oracle.shard_positions(seq, cp, r, kind_name))
    st, _ = _layout(64, 4, 0, 0)
    assert st == 0


def test_reshard_rejects_two_block_odd_length():
    lib = cpa.load_library()
    ptrs = (ctypes.c_void_p * 4)(0x1000, 0x2000, 0x3000, 0x4000)
    heads = (ctypes.c_int32 * 1)(8)
    # 36 % 4 == 0 but 36 % 8 != 0
    assert lib.cp_ulysses_reshard(0, 4, 36, 1, heads, 64, 1, api.CP_LAYOUT_TWO_BLOCK, ptrs, ptrs,
                                  None) == api.CP_ERR_INVALID_ARG


def test_bwd_desc_layout_matches_header():
    assert ctypes.sizeof(api._AttnBwdDesc) == 152
    assert api._AttnBwdDesc.aux.offset == 40 and api._AttnBwdDesc.q_pos.offset == 112


def _bwd_desc(**kw):
    d = api._AttnBwdDesc()
    d.q = d.k = d.v = d.d_o = 0x1000
    d.aux = d.dq = d.dk = d.dv = 0x2000
    d.in_dtype = api.CP_BF16
    d.sq, d.skv, d.hq, d.hkv, d.d = 128, 128, 8, 2, 128
    d.causal = 1
    d.q_pos = api._PosMap(0, 1)
    d.kv_pos = api._PosMap(0, 1)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("field,value", [
    ("d", 96), ("hq", 5), ("hkv", 0), ("in_dtype", 4), ("causal", 3), ("q", 0), ("aux", 0),
    ("dq", 0), ("dk", 0x2004), ("sq", -1), ("skv", -2), ("flags", 1), ("flags", 0x200),
    ("q_pos", api._PosMap(0, 0)), ("kv_pos", api._PosMap(-1, 1)), ("scale", float("inf")),
    ("wait_timeout_ms", -1),
])
def test_partial_attn_bwd_rejects(field, value):
    lib = cpa.load_library()
    d = _bwd_desc(**{field: value})
    assert lib.cp_partial_attn_bwd(ctypes.byref(d), None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_last_error()
    assert lib.cp_partial_attn_bwd(None, None) == api.CP_ERR_INVALID_ARG


def test_bwd_prep_rejects():
    lib = cpa.load_library()
    p = ctypes.c_void_p(0x1000)
    assert lib.cp_attn_bwd_prep(p, 7, p, 1, p, 16, 2, 64, p, None) == api.CP_ERR_INVALID_ARG   # o dtype
    assert lib.cp_attn_bwd_prep(p, 0, p, 1, p, 16, 2, 96, p, None) == api.CP_ERR_INVALID_ARG   # d
    assert lib.cp_attn_bwd_prep(p, 0, p, 1, p, 16, 0, 64, p, None) == api.CP_ERR_INVALID_ARG   # hq
    assert lib.cp_attn_bwd_prep(p, 0, p, 1, None, 16, 2, 64, p, None) == api.CP_ERR_INVALID_ARG  # lse
    assert lib.cp_attn_bwd_prep(p, 0, p, 1, p, 16, 2, 64, ctypes.c_void_p(0x1004), None) == \
        api.CP_ERR_INVALID_ARG  # aux alignment
    assert cpa.bwd_aux_floats(130, 3) == 2 * 3 * 256


def test_bwd_test_stall_needs_bf16():
    lib = cpa.load_library()
    d = _bwd_desc(flags=api.CP_FLAG_TEST_STALL, in_dtype=api.CP_F32)
    assert lib.cp_partial_attn_bwd(ctypes.byref(d), None) == api.CP_ERR_INVALID_ARG


def test_bwd_chunks_rejects():
    lib = cpa.load_library()
    assert ctypes.sizeof(api._KvBwdChunk) == 56
    d = _bwd_desc()
    arr = (api._KvBwdChunk * 2)()
    for i in range(2):
        arr[i].k = arr[i].v = 0x1000
        arr[i].dk = arr[i].dv = 0x2000
        arr[i].skv = 128
        arr[i].kv_pos = api._PosMap(0, 1)
    assert lib.cp_partial_attn_bwd_chunks(ctypes.byref(d), 0, arr, None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_partial_attn_bwd_chunks(ctypes.byref(d), 65, arr, None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_partial_attn_bwd_chunks(ctypes.byref(d), 2, None, None) == api.CP_ERR_INVALID_ARG
    assert lib.cp_partial_attn_bwd_chunks(None, 2, arr, None) == api.CP_ERR_INVALID_ARG
    arr[1].dv = 0
    assert lib.cp_partial_attn_bwd_chunks(ctypes.byref(d), 2, arr, None) == api.CP_ERR_INVALID_ARG
    arr[1].dv = 0x2000
    arr[1].kv_pos = api._PosMap(0, 0)
    assert lib.cp_partial_attn_bwd_chunks(ctypes.byref(d), 2, arr, None) == api.CP_ERR_INVALID_ARG


def test_balanced_layout_rejects():
    # too few tokens for every rank to get one; not one map of S/cp tokens; no Ulysses reshard
    assert _segments(7, 7, 0, api.CP_LAYOUT_BALANCED)[0] == api.CP_ERR_INVALID_ARG
    assert _layout(64, 4, 0, api.CP_LAYOUT_BALANCED)[0] == api.CP_ERR_INVALID_ARG
    lib = cpa.load_library()
    ptrs = (ctypes.c_void_p * 4)(0x1000, 0x2000, 0x3000, 0x4000)
    heads = (ctypes.c_int32 * 1)(8)
    assert lib.cp_ulysses_reshard(0, 4, 64, 1, heads, 64, 1, api.CP_LAYOUT_BALANCED, ptrs, ptrs,
                                  None) == api.CP_ERR_INVALID_ARG

