"""The device timeout path of the split kernel, without breaking anything.

Every wait in the kernel is bounded (1 s in the product build).  The debug build
of the same sources (libmla_decode_debug.so) lets a test shorten that limit to a
few microseconds, so that ordinary waits of a healthy call run out: the kernel
must report MLA_ERR_TIMEOUT through the workspace's error word, write the rows it
gave up on as NaN, and leave the context usable, so that the next call on the
same workspace succeeds and matches the oracle.  No wait is skipped, no barrier
removed and no input made invalid.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
from mla_paged_kv_02_gb300 import _lib, api, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    if not os.path.exists(_lib.DEBUG_LIB_PATH):
        import __graft_entry__

        __graft_entry__.build_cuda()
    lib = _lib.load_debug()
    yield lib
    lib.mla_debug_set_wait_limit_ns(0)


def _decode(lib, pl, inp, out, lse, ws):
    args = _lib._decode_args(pl, inp.q_nope.view(-1, 512), inp.q_pe.view(-1, 64), inp.kv_cache, inp.block_table,
                             inp.seq_lens, inp.softmax_scale, api.kv_scale_tensor(inp), out, lse, ws, None)
    return lib.mla_decode(*args)


def _check(lib, ws):
    info = (ctypes.c_int32 * 4)()
    st = lib.mla_decode_check_error(ctypes.c_void_p(ws.data_ptr()), _lib._stream(None), info)
    return st, list(info)


@pytest.mark.parametrize("kv_fp8", [False, True])
def test_timeout_is_reported_isolated_and_recoverable(dbg, kv_fp8):
    inp = synth.make_inputs("tiny", seed=90 + kv_fp8, kv_lens=[3, 300, 1000, 2000], q_len=2, batch=4,
                            num_heads=64, kv_fp8=kv_fp8)
    ref_o, ref_l = oracle.decode(inp)
    dev = inp.to("cuda")
    pl = api.plan_for(dev, force_splits=2)
    ws = api.alloc_workspace(pl, "cuda")
    out, lse = api.alloc_outputs(dev, out_fp32=True)

    assert dbg.mla_debug_set_wait_limit_ns(2000) == _lib.MLA_OK  # 2 us: ordinary waits run out
    try:
        assert _decode(dbg, pl, dev, out, lse, ws) == _lib.MLA_OK
        st, info = _check(dbg, ws)
    finally:
        dbg.mla_debug_set_wait_limit_ns(0)
    assert st == _lib.MLA_ERR_TIMEOUT, (st, info)
    assert info[0] == _lib.MLA_ERR_TIMEOUT
    # the rows of every cluster that gave up are NaN (never silently wrong)
    o = out.cpu().numpy()
    bad = np.isnan(o).any(axis=(1, 2, 3))
    assert bad.any()
    for b in np.nonzero(~bad)[0]:  # a request whose clusters all finished is still right
        assert np.max(np.abs(o[b] - ref_o[b])) <= 1e-2 * np.max(np.abs(ref_o[b])) + 1e-3

    # The context and the workspace stay usable: the next call succeeds.
    assert _decode(dbg, pl, dev, out, lse, ws) == _lib.MLA_OK
    st, info = _check(dbg, ws)
    assert st == _lib.MLA_OK, info
    o, l = out.double().cpu().numpy(), lse.double().cpu().numpy()
    tol = 2e-2 if kv_fp8 else 1e-2
    assert np.max(np.abs(o - ref_o)) <= tol * np.max(np.abs(ref_o)) + 1e-3
    assert np.max(np.abs(l - ref_l)) <= 1e-3
    # and so does the product library in the same process
    out2, lse2, _ = api.decode(dev, pl=pl, workspace=ws, out_fp32=True)
    torch.cuda.synchronize()
    assert torch.equal(out2, out) and torch.equal(lse2, lse)
