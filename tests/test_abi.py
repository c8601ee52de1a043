"""Host-side checks of the C ABI (no GPU): the library loads and exports every
symbol the header declares, the planner's integer logic, and argument
validation that must reject bad calls before any launch."""
import ctypes
import math
import os
import re

import pytest
import torch

from mla_paged_kv_02_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        import __graft_entry__

        __graft_entry__.build_cuda()
    return _lib.load()


def declared_symbols(debug=False):
    """Entry points declared by the product headers (or, with debug, by the debug
    build's own header)."""
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h") and f.endswith("_debug.h") == debug:
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(mla_\w+)\s*\(", text, flags=re.M))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert names == set(_lib.EXPORTED), names
    for n in names:
        assert hasattr(lib, n)


def test_debug_build_exports_its_hook_and_every_product_symbol(lib):
    dbg = _lib.load_debug()
    hooks = declared_symbols(debug=True)
    assert hooks == {"mla_debug_set_wait_limit_ns"}
    for n in hooks | set(_lib.EXPORTED):
        assert hasattr(dbg, n)
    assert not hasattr(lib, "mla_debug_set_wait_limit_ns")  # the product build has no test hook
    assert dbg.mla_debug_set_wait_limit_ns(0) == _lib.MLA_OK


def test_status_strings(lib):
    for code in range(7):
        assert _lib.status_string(code).startswith("MLA_")


def page_rule_reference(max_seq_len, sm_count):
    """The split-count rule of the Triton MLA path (vLLM PR #46819 summary, key code excerpt):
    next power of two of max(1, max_seq_len // 512), capped at 2 * sm_count."""
    ideal = 1 << (max(1, max_seq_len // 512) - 1).bit_length()
    return min(ideal, sm_count * 2)


@pytest.mark.parametrize("B,H,q,L", [(4, 16, 1, 200), (64, 128, 1, 4096), (64, 32, 4, 81920),
                                     (64, 32, 8, 81920), (128, 128, 2, 32768),
                                     (256, 16, 1, 131072), (1, 1, 1, 1)])
def test_plan_invariants(lib, B, H, q, L):
    for sms in (148, 152):
        pl = _lib.plan(B, H, q, L, num_sms=sms)
        assert pl.num_kv_splits >= 1
        assert pl.chunk_tokens % 64 == 0 and pl.chunk_tokens >= 64
        assert pl.num_kv_splits * pl.chunk_tokens >= L
        assert (pl.num_kv_splits - 1) * pl.chunk_tokens < L  # no split lies wholly past L
        assert pl.row_groups == math.ceil(H * q / pl.rows_per_cta)
        rows = B * H * q
        want = rows * pl.num_kv_splits * 513 * 4 if pl.num_kv_splits > 1 else 0
        assert pl.partial_bytes == want
        assert pl.workspace_bytes == 256 + want
        # partials stay small next to the KV stream
        assert pl.partial_bytes <= 0.1 * B * L * 576 * 2 + 256 * 1024 * 1024


def test_force_splits_reproduces_reference_rule(lib):
    for L in (512, 4096, 81920, 131072):
        s = page_rule_reference(L, 148)
        pl = _lib.plan(64, 32, 4, L, num_sms=148, force_splits=s)
        pages = math.ceil(L / 64)
        chunk_pages = math.ceil(pages / min(s, pages))
        assert pl.chunk_tokens == chunk_pages * 64
        assert pl.num_kv_splits == math.ceil(pages / chunk_pages)


def test_plan_rejects_unsupported(lib):
    p = _lib.Plan()
    f = lib.mla_decode_plan
    assert f(4, 16, 9, 100, 64, 0, 148, 0, ctypes.byref(p)) == _lib.MLA_ERR_UNSUPPORTED  # q_len > 8
    assert f(4, 16, 1, 100, 32, 0, 148, 0, ctypes.byref(p)) == _lib.MLA_ERR_UNSUPPORTED  # page 32
    assert f(4, 16, 4, 3, 64, 0, 148, 0, ctypes.byref(p)) == _lib.MLA_ERR_INVALID_ARG  # L < q
    assert f(0, 16, 1, 100, 64, 0, 148, 0, ctypes.byref(p)) == _lib.MLA_ERR_INVALID_ARG
    assert f(4, 16, 1, 100, 64, 7, 148, 0, ctypes.byref(p)) == _lib.MLA_ERR_UNSUPPORTED  # kv dtype
    assert f(4, 16, 1, 100, 64, 0, 148, 0, None) == _lib.MLA_ERR_INVALID_ARG


def _call_decode(lib, pl, **over):
    args = dict(q_nope=0x10000, qs=512, q_pe=0x20000, ps=64, kv=0x30000, pages=8, bt=0x40000,
                bts=4, seq=0x50000, scale=0.07, kvs=None, out=0x60000, odt=0, lse=None,
                ws=0x70000, wsb=pl.workspace_bytes)
    args.update(over)
    P = ctypes.c_void_p
    return lib.mla_decode(ctypes.byref(pl), P(args["q_nope"]), args["qs"], P(args["q_pe"]), args["ps"],
                          P(args["kv"]), args["pages"], P(args["bt"]), args["bts"], P(args["seq"]),
                          args["scale"], P(args["kvs"]), P(args["out"]), args["odt"], P(args["lse"]),
                          P(args["ws"]), args["wsb"], None)


def test_decode_validation_rejects_before_launch(lib):
    pl = _lib.plan(2, 16, 1, 200, num_sms=148, force_splits=2)
    E = _lib.MLA_ERR_INVALID_ARG
    assert _call_decode(lib, pl, q_nope=0) == E
    assert _call_decode(lib, pl, seq=0) == E
    assert _call_decode(lib, pl, ws=0) == E
    assert _call_decode(lib, pl, qs=500) == E  # stride shorter than a row
    assert _call_decode(lib, pl, ps=60) == E  # stride not a multiple of 8 elements
    assert _call_decode(lib, pl, kv=0x30008) == E  # TMA needs a 16-byte aligned cache
    assert _call_decode(lib, pl, ws=0x70010) == E  # workspace alignment
    assert _call_decode(lib, pl, bts=3) == E  # block table narrower than ceil(200/64)
    assert _call_decode(lib, pl, pages=0) == E
    assert _call_decode(lib, pl, scale=float("nan")) == E
    assert _call_decode(lib, pl, scale=0.0) == E
    assert _call_decode(lib, pl, odt=5) == E
    assert _call_decode(lib, pl, wsb=pl.workspace_bytes - 1) == _lib.MLA_ERR_WORKSPACE_TOO_SMALL
    bad = _lib.Plan.from_buffer_copy(pl)
    bad.q_len = 9
    assert _call_decode(lib, bad) == E
    bad = _lib.Plan.from_buffer_copy(pl)
    bad.chunk_tokens = 100
    assert _call_decode(lib, bad) == E
    bad = _lib.Plan.from_buffer_copy(pl)
    bad.num_kv_splits = 1  # one split of 128 tokens cannot cover max_seq_len 200
    assert _call_decode(lib, bad) == E


def test_edited_plan_is_refused_before_launch(lib):
    # The kernels size their partial writes from num_kv_splits: a plan edited
    # after mla_decode_plan (more splits, byte counts left alone) must be
    # refused by every entry point that takes a plan, before any launch.
    pl = _lib.plan(2, 16, 1, 4096, num_sms=148, force_splits=2)
    E = _lib.MLA_ERR_INVALID_ARG
    bad = _lib.Plan.from_buffer_copy(pl)
    bad.num_kv_splits = 8
    bad.chunk_tokens = 512
    assert _call_decode(lib, bad, wsb=1 << 30) == E
    assert lib.mla_combine(ctypes.byref(bad), ctypes.c_void_p(0x60000), 0, None, ctypes.c_void_p(0x70000),
                           1 << 30, None) == E
    P = ctypes.c_void_p
    assert lib.mla_decode_noalloc(ctypes.byref(bad), P(0x10000), 512, P(0x20000), 64, P(0x30000), 8,
                                  P(0x40000), 64, P(0x50000), 0.07, None, P(0x60000), 0, None, None) == E
    for field, value in (("partial_bytes", pl.partial_bytes * 2), ("workspace_bytes", pl.workspace_bytes + 64),
                         ("row_groups", 2), ("num_kv_splits", 200)):
        bad = _lib.Plan.from_buffer_copy(pl)
        setattr(bad, field, value)
        assert _call_decode(lib, bad, wsb=1 << 30) == E, field


def test_plan_rejects_batch_beyond_grid_limit(lib):
    # The batch is a grid dimension of the split kernel (limit 65535).
    p = _lib.Plan()
    assert lib.mla_decode_plan(65536, 16, 1, 100, 64, 0, 148, 0, ctypes.byref(p)) == _lib.MLA_ERR_UNSUPPORTED
    assert lib.mla_decode_plan(65535, 16, 1, 100, 64, 0, 148, 0, ctypes.byref(p)) == _lib.MLA_OK
    assert lib.mla_decode_plan(4, 16, 1, (1 << 30) + 1, 64, 0, 148, 0, ctypes.byref(p)) == _lib.MLA_ERR_UNSUPPORTED


def test_decode_varlen_validation_rejects_before_launch(lib):
    # The per-request q_len entry point: a missing q_lens array, and every
    # host-checkable problem of mla_decode, return before any launch.
    pl = _lib.plan(2, 16, 4, 200, num_sms=148, force_splits=2)
    P = ctypes.c_void_p
    E = _lib.MLA_ERR_INVALID_ARG

    def call(q_lens=0x80000, q_nope=0x10000):
        return lib.mla_decode_varlen(ctypes.byref(pl), P(q_nope), 512, P(0x20000), 64, P(0x30000), 8,
                                     P(0x40000), 4, P(0x50000), P(q_lens), 0.07, None, P(0x60000), 0,
                                     None, P(0x70000), pl.workspace_bytes, None)

    assert call(q_lens=0) == E
    assert call(q_nope=0) == E


def test_fp8_entry_point_validation(lib):
    # mla_decode_fp8: an FP8 query needs an FP8 cache plan; query row strides
    # are 16-byte multiples (e4m3: 16 elements); an FP8 output is accepted only
    # here, not by mla_decode.
    P = ctypes.c_void_p
    pl8 = _lib.plan(2, 16, 1, 200, kv_fp8=True, num_sms=148, force_splits=2)
    plb = _lib.plan(2, 16, 1, 200, num_sms=148, force_splits=2)

    def call(pl, qs=512, ps=64, odt=_lib.MLA_OUT_FP8_E4M3):
        return lib.mla_decode_fp8(ctypes.byref(pl), P(0x10000), qs, P(0x20000), ps, None, P(0x30000), 8,
                                  P(0x40000), 4, P(0x50000), 0.07, None, P(0x60000), odt, None, None,
                                  P(0x70000), pl.workspace_bytes, None)

    assert call(plb) == _lib.MLA_ERR_UNSUPPORTED
    assert call(pl8, qs=520) == _lib.MLA_ERR_INVALID_ARG  # 520 bytes: not a 16-byte multiple
    assert call(pl8, ps=72) == _lib.MLA_ERR_INVALID_ARG
    assert call(pl8, odt=7) == _lib.MLA_ERR_INVALID_ARG
    assert _call_decode(lib, plb, odt=_lib.MLA_OUT_FP8_E4M3) == _lib.MLA_ERR_INVALID_ARG


def test_length_aware_plan():
    # mla_decode_plan_lengths: host-only, never more splits than the length-blind
    # plan for the longest request, the same geometry rules, and fewer splits when
    # a few long requests dominate a batch of uneven lengths.
    g = torch.Generator().manual_seed(3)
    equal = [81920] * 64
    p_len = _lib.plan_lengths(32, 4, equal, num_sms=152)
    p_uni = _lib.plan(64, 32, 4, 81920, num_sms=152)
    assert p_len.num_kv_splits == p_uni.num_kv_splits == 7  # the MTP-3 shape
    assert p_len.workspace_bytes == p_uni.workspace_bytes
    uneven = torch.randint(1, 131073, (256,), generator=g).tolist()
    p_len = _lib.plan_lengths(16, 1, uneven, num_sms=152)
    p_uni = _lib.plan(256, 16, 1, max(uneven), num_sms=152)
    assert p_len.max_seq_len == max(uneven)
    assert 1 <= p_len.num_kv_splits < p_uni.num_kv_splits
    assert p_len.num_kv_splits * p_len.chunk_tokens >= max(uneven)
    # a single request spreads over every cluster slot
    one = _lib.plan_lengths(64, 2, [131072 - 5], num_sms=152)
    assert one.num_kv_splits == _lib.plan(1, 64, 2, 131072 - 5, num_sms=152).num_kv_splits
    for bad in ([3, 1], []):  # a length below q_len, an empty batch
        with pytest.raises(_lib.MlaError):
            _lib.plan_lengths(16, 2, bad, num_sms=152)
    lib = _lib.load()
    pl = _lib.Plan()
    assert lib.mla_decode_plan_lengths(4, 16, 1, None, 64, 0, 152, ctypes.byref(pl)) == _lib.MLA_ERR_INVALID_ARG
