"""GPU parity of the sequence-sharded (DCP) decode: every shard's partial against
the oracle's token-range form, and the merged shards against the single-pass
oracle, through the C ABI (mla_decode_shard, mla_combine_shards).

One GPU runs the shards one after another: each call sees only its own paged
cache, block table and token range, exactly as a rank would; the all-gather of
a real multi-GPU run is replaced by stacking the partials (its layout is tested
on gloo ranks in test_dcp.py).  Bounds as in test_gpu_parity: bf16
max|out-ref| <= 1e-2*max|ref| + 1e-3, |lse-ref| <= 1e-3; FP8 the same with 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from mla_paged_kv_02_gb300 import _lib, api, dcp, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import os

    if not os.path.exists(_lib.LIB_PATH):
        import __graft_entry__

        __graft_entry__.build_cuda()
    _lib.load()


def _bound(fp8):
    return 2e-2 if fp8 else 1e-2


def check_partial(part, ref, fp8, what):
    """Shard partial [B,q,H,513] against the oracle's range form: rows that see
    nothing in the shard are exactly 0 / -inf, the others within the bound."""
    got = part.double().cpu().numpy()
    empty = np.isneginf(ref[..., 512])
    assert np.array_equal(np.isneginf(got[..., 512]), empty), f"{what}: empty rows differ"
    assert np.all(got[..., :512][empty] == 0), f"{what}: empty rows not zero"
    live = ~empty
    o, r = got[..., :512][live], ref[..., :512][live]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(got[..., 512][live]))
    err_o = float(np.max(np.abs(o - r))) if o.size else 0.0
    err_l = float(np.max(np.abs(got[..., 512][live] - ref[..., 512][live]))) if o.size else 0.0
    ref_max = float(np.max(np.abs(r))) if o.size else 0.0
    print(f"{what}: max|o-ref|={err_o:.3e} (norm {err_o / max(ref_max, 1e-30):.3e}) max|lse-ref|={err_l:.3e}")
    assert err_o <= _bound(fp8) * ref_max + 1e-3 and err_l <= 1e-3, what


def check_out(out, lse, ref_o, ref_l, fp8, what):
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l)), what
    err_o = float(np.max(np.abs(o - ref_o)))
    err_l = float(np.max(np.abs(l - ref_l)))
    ref_max = float(np.max(np.abs(ref_o)))
    print(f"{what}: max|out-ref|={err_o:.3e} (norm {err_o / ref_max:.3e}) max|lse-ref|={err_l:.3e}")
    assert err_o <= _bound(fp8) * ref_max + 1e-3 and err_l <= 1e-3, what


def run_shard(dev, bt, lo, hi, splits, kv_cache=None):
    """mla_decode_shard for one rank holding [lo[b], hi[b]) of every request."""
    sl = torch.tensor([h - l for l, h in zip(lo, hi)], dtype=torch.int32, device="cuda")
    ss = torch.tensor(lo, dtype=torch.int32, device="cuda")
    max_local = max(int(sl.max()), dev.q_len)
    pl = _lib.plan(dev.batch, dev.num_heads, dev.q_len, max_local, kv_fp8=dev.kv_fp8, force_splits=splits)
    ws = api.alloc_workspace(pl, "cuda")
    part = torch.full((dev.batch, dev.q_len, dev.num_heads, 513), float("nan"), device="cuda")
    st = _lib.decode_shard(pl, dev.q_nope.view(-1, 512), dev.q_pe.view(-1, 64),
                           dev.kv_cache if kv_cache is None else kv_cache, bt, sl, ss, dev.seq_lens,
                           dev.softmax_scale, api.kv_scale_tensor(dev), part, ws)
    assert st == _lib.MLA_OK, _lib.status_string(st)
    st, info = _lib.check_error(ws)
    assert st == _lib.MLA_OK, info
    return part


def merge(parts, dev):
    out = torch.empty((dev.batch, dev.q_len, dev.num_heads, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((dev.batch, dev.q_len, dev.num_heads), dtype=torch.float32, device="cuda")
    st = _lib.combine_shards(torch.stack(parts), out, lse)
    assert st == _lib.MLA_OK
    torch.cuda.synchronize()
    return out, lse


CASES = [(2, 1, False, 0), (3, 4, False, 3), (2, 2, True, 0), (4, 8, False, 1), (3, 4, True, 2)]


@pytest.mark.parametrize("world,q_len,fp8,splits", CASES,
                         ids=[f"w{w}-q{q}-{'fp8' if f else 'bf16'}-s{s}" for w, q, f, s in CASES])
def test_page_aligned_shards_match_the_oracle(world, q_len, fp8, splits):
    lens = [q_len, 70, 300, 1000 + q_len, 64, 2 * q_len + 127]
    inp = synth.make_inputs("tiny", seed=40 + world + q_len, kv_lens=lens, q_len=q_len, batch=len(lens),
                            num_heads=32, sharp=4.0, kv_fp8=fp8)
    ref_o, ref_l = oracle.decode(inp)
    dev = inp.to("cuda")
    parts = []
    for r in range(world):
        bounds = dcp.shard_bounds(lens, world, r)
        lo, hi = [s for s, _ in bounds], [e for _, e in bounds]
        part = run_shard(dev, dcp.local_block_table(dev.block_table, bounds), lo, hi, splits)
        check_partial(part, oracle.decode_range(inp, lo, hi), fp8, f"rank {r}/{world} partial")
        parts.append(part)
    out, lse = merge(parts, dev)
    check_out(out, lse, ref_o, ref_l, fp8, f"{world} shards merged")


def _repage(inp, lo, hi, nan_tail):
    """A rank's own paged cache for arbitrary (unaligned) ranges: the rank's
    tokens of request b copied into fresh local pages from slot 0 on (test-side
    data movement); unused slots hold NaN when ``nan_tail``."""
    pages, bts = [], []
    nxt = 0
    fill = float("nan") if nan_tail else 0.0
    for b in range(inp.batch):
        n = hi[b] - lo[b]
        npg = -(-n // 64)
        rows = torch.full((npg * 64, 576), fill, dtype=torch.float32)
        if inp.kv_fp8:
            rows = torch.full((npg * 64, 576), 0x7F if nan_tail else 0, dtype=torch.uint8)
        for t in range(n):
            g = lo[b] + t
            src = inp.kv_cache[int(inp.block_table[b, g // 64]), g % 64]
            rows[t] = src if inp.kv_fp8 else src.float()
        if npg:
            pages.append(rows.view(npg, 64, 576) if inp.kv_fp8 else rows.view(npg, 64, 576).to(torch.bfloat16))
        bts.append(list(range(nxt, nxt + npg)))
        nxt += npg
    width = max(1, max(len(x) for x in bts))
    bt = torch.full((inp.batch, width), -1, dtype=torch.int32)
    for b, x in enumerate(bts):
        bt[b, :len(x)] = torch.tensor(x, dtype=torch.int32)
    kv = torch.cat(pages) if pages else torch.zeros((1, 64, 576), dtype=inp.kv_cache.dtype)
    return kv, bt


@pytest.mark.parametrize("fp8", [False, True])
def test_unaligned_shards_with_their_own_caches(fp8):
    # Ranges that start mid-page, an empty shard for a short request, and a last
    # shard holding only positions the first MTP query rows may not see.
    q_len = 4
    lens = [4, 90, 333, 700]
    cuts = [[0, 2, 4, 4], [0, 31, 77, 90], [0, 100, 329, 333], [0, 1, 650, 700]]  # per request, 3 shards
    inp = synth.make_inputs("tiny", seed=50 + fp8, kv_lens=lens, q_len=q_len, batch=4, num_heads=16, sharp=4.0,
                            kv_fp8=fp8)
    ref_o, ref_l = oracle.decode(inp)
    dev = inp.to("cuda")
    parts = []
    for r in range(3):
        lo = [c[r] for c in cuts]
        hi = [c[r + 1] for c in cuts]
        kv, bt = _repage(inp, lo, hi, nan_tail=True)
        part = run_shard(dev, bt.cuda(), lo, hi, 0, kv_cache=kv.cuda())
        check_partial(part, oracle.decode_range(inp, lo, hi), fp8, f"unaligned rank {r}")
        parts.append(part)
    out, lse = merge(parts, dev)
    check_out(out, lse, ref_o, ref_l, fp8, "unaligned shards merged")


def test_two_shards_at_a_long_context():
    # An MTP-3 shape at 16k tokens split over two ranks, against the oracle.
    inp = synth.make_inputs("mtp3", seed=60, kv_lens=[16384] * 6, batch=6, sharp=4.0, page_offset=0.05)
    ref_o, ref_l = oracle.decode(inp)
    dev = inp.to("cuda")
    lens = [int(x) for x in inp.seq_lens]
    parts = []
    for r in range(2):
        bounds = dcp.shard_bounds(lens, 2, r)
        lo, hi = [s for s, _ in bounds], [e for _, e in bounds]
        parts.append(run_shard(dev, dcp.local_block_table(dev.block_table, bounds), lo, hi, 0))
    out, lse = merge(parts, dev)
    check_out(out, lse, ref_o, ref_l, False, "mtp3 16k, 2 shards")


def test_bad_shard_range_is_reported_and_isolated():
    inp = synth.make_inputs("tiny", seed=70, kv_lens=[50, 200, 300], q_len=2, batch=3, num_heads=16)
    dev = inp.to("cuda")
    lo, hi = [0, 0, 0], [50, 200, 300]
    sl = torch.tensor([50, 200, 300], dtype=torch.int32, device="cuda")
    ss = torch.tensor([0, 10, 0], dtype=torch.int32, device="cuda")  # request 1: 10 + 200 > L
    pl = _lib.plan(3, 16, 2, 300)
    ws = api.alloc_workspace(pl, "cuda")
    part = torch.zeros((3, 2, 16, 513), device="cuda")
    st = _lib.decode_shard(pl, dev.q_nope.view(-1, 512), dev.q_pe.view(-1, 64), dev.kv_cache, dev.block_table,
                           sl, ss, dev.seq_lens, dev.softmax_scale, None, part, ws)
    assert st == _lib.MLA_OK
    st, info = _lib.check_error(ws)
    assert st == _lib.MLA_ERR_DEVICE_INPUT and info[1] == 1 and info[2] == -3 and info[3] == 10
    assert torch.isnan(part[1]).all()
    ref = oracle.decode_range(inp, lo, hi)
    check_partial(part[[0, 2]], ref[[0, 2]], False, "valid requests")


def test_dcp_decode_through_nccl_on_one_rank():
    # dcp.decode end to end with a real NCCL process group.  One GPU gives one
    # rank (ranks on one GPU would wait on one another's kernels), so the
    # all-gather is NCCL's with a world of one: the shard is the whole sequence
    # and the merged result must equal the oracle's and mla_decode's.
    import torch.distributed as dist

    if not dist.is_nccl_available():
        pytest.skip("torch built without NCCL")
    inp = synth.make_inputs("tiny", seed=80, kv_lens=[3, 70, 200, 641], q_len=2, batch=4, num_heads=32, sharp=4.0)
    ref_o, ref_l = oracle.decode(inp)
    dev = inp.to("cuda")
    store = dist.HashStore()
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        bounds = dcp.shard_bounds(dev.seq_lens.tolist(), 1, 0)
        bt = dcp.local_block_table(dev.block_table, bounds)
        sl = torch.tensor([e - s for s, e in bounds], dtype=torch.int32, device="cuda")
        ss = torch.tensor([s for s, _ in bounds], dtype=torch.int32, device="cuda")
        pl = _lib.plan(dev.batch, dev.num_heads, dev.q_len, max(int(sl.max()), dev.q_len), force_splits=0)
        ws = api.alloc_workspace(pl, "cuda")
        out = torch.empty((dev.batch, dev.q_len, dev.num_heads, 512), dtype=torch.float32, device="cuda")
        lse = torch.empty((dev.batch, dev.q_len, dev.num_heads), dtype=torch.float32, device="cuda")
        parts = dcp.decode(pl, dev.q_nope, dev.q_pe, dev.kv_cache, bt, sl, ss, dev.seq_lens, dev.softmax_scale,
                           api.kv_scale_tensor(dev), out, lse, ws, group=dist.group.WORLD)
        torch.cuda.synchronize()
        assert parts.shape == (1, dev.batch, dev.q_len, dev.num_heads, 513)
        assert _lib.check_error(ws)[0] == _lib.MLA_OK
    finally:
        dist.destroy_process_group()
    check_out(out, lse, ref_o, ref_l, False, "DCP through NCCL, world 1")
    o2, l2, _ = api.decode(dev, out_fp32=True)
    torch.cuda.synchronize()
    assert torch.allclose(out, o2, rtol=0, atol=1e-5) and torch.allclose(lse, l2, rtol=0, atol=1e-5)
