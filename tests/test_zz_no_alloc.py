"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers of this library (a plug-in inside a host framework that owns every
device allocation, or code handed only input and output pointers) have no way to
provide the workspace mla_decode needs.  mla_decode_noalloc runs the same kernels
on a fixed scratch array inside the library instead.  These tests call it through
the C ABI and check that it matches mla_decode, on two calls in a row (the array
keeps the previous call's contents), and that a plan too large for the array is
refused.  The file is named so pytest collects it last.
"""
import os

import numpy as np
import pytest
import torch

from mla_paged_kv_02_gb300 import _lib, api, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(_lib.LIB_PATH):
        import __graft_entry__

        __graft_entry__.build_cuda()
    _lib.load()


def within_tolerance(out, lse, ref_o, ref_l, fp8=False):
    """The bound the parity tests use: max|out-ref| <= rel*max|ref| + 1e-3, |lse-ref| <= 1e-3."""
    rel = 2e-2 if fp8 else 1e-2
    o, r = out.float().cpu().numpy(), ref_o.float().cpu().numpy()
    l, rl = lse.cpu().numpy(), ref_l.cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    assert np.max(np.abs(o - r)) <= rel * np.max(np.abs(r)) + 1e-3
    assert np.max(np.abs(l - rl)) <= 1e-3


def run_noalloc(inp, pl, out_fp32):
    out, lse = api.alloc_outputs(inp, out_fp32)
    st = _lib.decode_noalloc(pl, inp.q_nope.view(-1, 512), inp.q_pe.view(-1, 64), inp.kv_cache,
                             inp.block_table, inp.seq_lens, inp.softmax_scale, api.kv_scale_tensor(inp),
                             out, lse)
    assert st == _lib.MLA_OK, _lib.status_string(st)
    torch.cuda.synchronize()
    return out, lse


CASES = [
    ("tiny", dict(), 2, True),
    ("mtp", dict(kv_lens=[4, 700, 3000, 4096], q_len=4, batch=4, num_heads=32, sharp=4.0), 3, False),
    ("fp8", dict(kv_lens=[2, 1500, 3000], q_len=2, batch=3, num_heads=128, kv_fp8=True), 5, True),
]


@pytest.mark.parametrize("name,kw,splits,out_fp32", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_decode_on_two_calls_in_a_row(name, kw, splits, out_fp32):
    for call, seed in enumerate((11, 12)):  # two calls in a row on the same scratch array
        inp = synth.make_inputs("tiny", seed=seed, device="cuda", **kw)
        pl = api.plan_for(inp, force_splits=splits)
        assert pl.workspace_bytes <= (32 << 20)
        ref_o, ref_l, _ = api.decode(inp, pl=pl, out_fp32=out_fp32)
        out, lse = run_noalloc(inp, pl, out_fp32)
        within_tolerance(out, lse, ref_o, ref_l, fp8=inp.kv_fp8)


def test_noalloc_error_of_one_call_does_not_leak_into_the_next():
    # The caller cannot read the error word, so each call clears it.  A call
    # with a device-side input error (one seq_len above the planned maximum)
    # writes that request's rows as NaN; the next, valid call on the same
    # scratch array must be finite and match mla_decode.
    inp = synth.make_inputs("tiny", seed=21, device="cuda", kv_lens=[3, 90, 300], q_len=2, batch=3,
                            num_heads=16)
    pl = api.plan_for(inp, force_splits=3)
    bad = synth.Inputs(**{**inp.__dict__})
    bad.seq_lens = inp.seq_lens.clone()
    bad.seq_lens[1] = pl.max_seq_len + 1
    out, lse = run_noalloc(bad, pl, True)
    assert torch.isnan(out[1]).all() and torch.isnan(lse[1]).all()
    assert torch.isfinite(out[0]).all() and torch.isfinite(out[2]).all()
    ref_o, ref_l, _ = api.decode(inp, pl=pl, out_fp32=True)
    out, lse = run_noalloc(inp, pl, True)
    within_tolerance(out, lse, ref_o, ref_l)


def test_noalloc_refuses_a_plan_larger_than_its_scratch():
    pl = _lib.plan(64, 128, 8, 131072, num_sms=152, force_splits=64)
    assert pl.workspace_bytes > (32 << 20)
    inp = synth.make_inputs("tiny", seed=1, device="cuda")
    out, lse = api.alloc_outputs(inp)
    st = _lib.decode_noalloc(pl, inp.q_nope.view(-1, 512), inp.q_pe.view(-1, 64), inp.kv_cache,
                             inp.block_table, inp.seq_lens, inp.softmax_scale, None, out, lse)
    assert st == _lib.MLA_ERR_WORKSPACE_TOO_SMALL
