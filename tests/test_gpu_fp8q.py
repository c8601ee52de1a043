"""GPU parity of mla_decode_fp8: an FP8 (e4m3) query over an FP8 cache, QK^T on the
FP8 tensor path, and an optional FP8 output, against the oracle run on the same
dequantised values (query = code * q_scale, cache = code * kv_scale).

Bound: the FP8 form of the task's bound, max|out-ref| <= 2e-2*max|ref| + 1e-3
and max|lse-ref| <= 1e-3.  An FP8 output is an integer decision taken on the
kernel's float32 value: its codes must equal, bit for bit, the oracle's E4M3
encoding of the same call's float32 output divided by out_scale in float32,
that float32 output must meet the bound against the oracle, and the dequantised
codes must meet it widened by half an E4M3 step of each element.
"""
import numpy as np
import pytest
import torch

import oracle
from mla_paged_kv_02_gb300 import _lib, api, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import os

    if not os.path.exists(_lib.LIB_PATH):
        import __graft_entry__

        __graft_entry__.build_cuda()
    _lib.load()


def run_fp8(dev, splits=0, out_kind="fp32", out_scale=None, pl=None):
    if pl is None:  # the benchmark's plan (from the batch's lengths) unless a split count is forced
        pl = api.plan_for(dev, force_splits=splits)
    ws = api.alloc_workspace(pl, "cuda")
    shape = (dev.batch, dev.q_len, dev.num_heads, 512)
    dt = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8}[out_kind]
    out = torch.empty(shape, dtype=dt, device="cuda")
    lse = torch.empty(shape[:-1], dtype=torch.float32, device="cuda")
    qs = torch.tensor([dev.q_scale], dtype=torch.float32, device="cuda")
    kvs = torch.tensor([dev.kv_scale], dtype=torch.float32, device="cuda")
    osc = None if out_scale is None else torch.tensor([out_scale], dtype=torch.float32, device="cuda")
    st = _lib.decode_fp8(pl, dev.q_nope.view(-1, 512), dev.q_pe.view(-1, 64), qs, dev.kv_cache, dev.block_table,
                         dev.seq_lens, dev.softmax_scale, kvs, out, osc, lse, ws)
    assert st == _lib.MLA_OK, _lib.status_string(st)
    st, info = _lib.check_error(ws)
    assert st == _lib.MLA_OK, info
    return out, lse, pl


def compare(out, lse, ref_o, ref_l, what):
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l)), what
    err_o = float(np.max(np.abs(o - ref_o)))
    err_l = float(np.max(np.abs(l - ref_l)))
    ref_max = float(np.max(np.abs(ref_o)))
    norm = err_o / max(ref_max, 1e-30)
    print(f"{what}: max|out-ref|={err_o:.3e} (norm {norm:.3e}) max|lse-ref|={err_l:.3e}")
    assert err_o <= 2e-2 * ref_max + 1e-3, what
    assert err_l <= 1e-3, what
    return norm


def e4m3_step(x):
    """Spacing of the E4M3 grid at |x| (2^-9 in the subnormal range)."""
    a = np.maximum(np.abs(x), 2.0 ** -6)
    return 2.0 ** (np.floor(np.log2(a)) - 3)


def check_fp8_out(codes, out32, lse, ref_o, ref_l, out_scale, what):
    """codes: the FP8 output; out32: the same call with an fp32 output.  The
    kernel takes the rounding decision on the float32 quotient out / out_scale,
    so the codes must equal the oracle's E4M3 encoding of that same float32
    quotient, bit for bit; the fp32 output meets the FP8 bound against the
    oracle; and the dequantised codes meet it widened by half an E4M3 step."""
    got = codes.cpu().numpy()
    o32 = out32.cpu().numpy().astype(np.float32)
    q32 = (o32 / np.float32(out_scale)).astype(np.float32)
    want = oracle.e4m3_encode(q32.astype(np.float64))
    mism = int(np.count_nonzero(got != want))
    ref_max = float(np.max(np.abs(ref_o)))
    err32 = float(np.max(np.abs(o32 - ref_o)))
    deq = oracle.e4m3_to_f64(got) * out_scale
    slack = 0.5 * e4m3_step(ref_o / out_scale) * out_scale
    err = np.abs(deq - ref_o)
    print(f"{what}: {mism} codes differ from the encoding of the fp32 output, max|out32-ref|={err32:.3e}, "
          f"max|deq-ref|={float(err.max()):.3e}")
    assert mism == 0, what
    assert err32 <= 2e-2 * ref_max + 1e-3, what
    assert np.all(err <= 2e-2 * ref_max + 1e-3 + slack), what
    assert float(np.max(np.abs(lse.double().cpu().numpy() - ref_l))) <= 1e-3, what


def small(seed, q_len, lens, H=128, **kw):
    return synth.make_inputs("tiny", seed=seed, kv_lens=list(lens), q_len=q_len, batch=len(lens), num_heads=H,
                             kv_fp8=True, q_fp8=True, **kw)


@pytest.mark.parametrize("q_len", [1, 2, 4])
def test_fp8_query_small(q_len):
    inp = small(1200 + q_len, q_len, [q_len, 100, 1100, 3000], H=64 if q_len == 4 else 128, sharp=3.0)
    ref_o, ref_l = oracle.decode(inp)
    dev = inp.to("cuda")
    for s in (0, 1, 3):
        out, lse, pl = run_fp8(dev, splits=s)
        compare(out, lse, ref_o, ref_l, f"fp8q q={q_len} s={pl.num_kv_splits}")


@pytest.mark.parametrize("variant", ["sharp", "page_offset", "needle"])
def test_fp8_query_structural(variant):
    kw = {"sharp": dict(sharp=20.0), "page_offset": dict(page_offset=0.05, sharp=4.0),
          "needle": dict(needle=True)}[variant]
    inp = small(1300, 2, [2, 200, 641, 1002], H=128, **kw)
    ref_o, ref_l = oracle.decode(inp)
    dev = inp.to("cuda")
    for s in (0, 1, 5):
        out, lse, pl = run_fp8(dev, splits=s)
        compare(out, lse, ref_o, ref_l, f"fp8q {variant} s={pl.num_kv_splits}")


def test_fp8_query_mtp_mask_and_nan_tails():
    # Short sequences where the causal mask inside the query block matters, and
    # NaN codes in every slot past L and in spare pages (never part of the result).
    lens = [4, 5, 63, 64, 65, 130]
    clean = small(1400, 4, lens, H=32, spare_pages=3)
    dirty = small(1400, 4, lens, H=32, spare_pages=3, nan_tail=True)
    ref_o, ref_l = oracle.decode(clean)
    for s in (0, 1, 3):
        o1, l1, _ = run_fp8(clean.to("cuda"), splits=s)
        o2, l2, _ = run_fp8(dirty.to("cuda"), splits=s)
        compare(o1, l1, ref_o, ref_l, f"fp8q mtp short s={s}")
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("splits", [1, 3])
def test_fp8_output(splits):
    inp = small(1500, 2, [2, 300, 1500], H=64, sharp=4.0, page_offset=0.05)
    ref_o, ref_l = oracle.decode(inp)
    dev = inp.to("cuda")
    out_scale = float(np.max(np.abs(ref_o))) / 200.0  # the output spans most of the E4M3 range
    codes, lse, _ = run_fp8(dev, splits=splits, out_kind="fp8", out_scale=out_scale)
    out32, _, _ = run_fp8(dev, splits=splits, out_kind="fp32")
    assert codes.dtype == torch.uint8
    check_fp8_out(codes, out32, lse, ref_o, ref_l, out_scale, f"fp8 out s={splits}")


def test_fp8_output_saturates():
    inp = small(1510, 1, [1, 90], H=16, sharp=2.0)
    ref_o, ref_l = oracle.decode(inp)
    out_scale = float(np.max(np.abs(ref_o))) / 1000.0  # the largest outputs exceed 448 codes
    codes, lse, _ = run_fp8(inp.to("cuda"), splits=1, out_kind="fp8", out_scale=out_scale)
    got = codes.cpu().numpy()
    want = oracle.e4m3_encode(ref_o / out_scale)
    big = np.abs(ref_o / out_scale) > 480
    assert big.any()
    assert np.array_equal(got[big], want[big])  # saturated codes 0x7E / 0xFE on both sides
    assert set(np.unique(got[big]).tolist()) <= {0x7E, 0xFE}


def test_fp8_query_needs_an_fp8_cache():
    inp = small(1520, 1, [1, 90], H=16)
    dev = inp.to("cuda")
    pl = _lib.plan(dev.batch, dev.num_heads, 1, 90)  # a bf16-cache plan
    ws = api.alloc_workspace(pl, "cuda")
    out = torch.empty((2, 1, 16, 512), device="cuda")
    lse = torch.empty((2, 1, 16), device="cuda")
    st = _lib.decode_fp8(pl, dev.q_nope.view(-1, 512), dev.q_pe.view(-1, 64), None, dev.kv_cache, dev.block_table,
                         dev.seq_lens, dev.softmax_scale, None, out, None, lse, ws)
    assert st == _lib.MLA_ERR_UNSUPPORTED


def test_fp8_query_full_size_every_request():
    # The FP8 workload (B=128, H=128, q_len=2, lognormal lengths) with an FP8
    # query, in the planner's launch configuration, every request against the oracle.
    inp = synth.make_inputs("fp8", seed=list(synth.WORKLOADS).index("fp8"), device="cuda", q_fp8=True)
    out, lse, pl = run_fp8(inp)
    host = inp.to("cpu")
    del inp
    ref_o, ref_l = oracle.decode(host)
    norm = compare(out, lse, ref_o, ref_l, f"fp8q full B={host.batch} splits={pl.num_kv_splits}")
    assert norm <= 2e-2
