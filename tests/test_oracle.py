"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: a library
routine (torch float64 SDPA / logsumexp / float8 decode), a different
formulation (un-absorbed MHA with explicit W_UK keys), a closed form, or an
invariant the definition implies.  A dropped term (k_pe), a wrong sign, an
off-by-one in the causal mask, a transposed operand or a wrong page lookup
fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from mla_paged_kv_02_gb300 import synth


def small(seed=0, B=3, H=4, q_len=1, kv_lens=(1, 37, 130), fp8=False, **kw):
    return synth.make_inputs("tiny", seed=seed, kv_lens=list(kv_lens), q_len=q_len, kv_fp8=fp8,
                             batch=B, num_heads=H, **kw)


def gather_rows_torch(inp, b, n):
    """Logical rows 0..n-1 of request b, gathered with torch indexing (not the oracle)."""
    t = torch.arange(n)
    pages = inp.block_table[b].long()[t // inp.page_size]
    rows = inp.kv_cache[pages, t % inp.page_size]
    if inp.kv_fp8:
        return rows.view(torch.float8_e4m3fn).to(torch.float64) * inp.kv_scale
    return rows.to(torch.float64)


def sdpa_reference(inp):
    """Library-routine form: torch float64 SDPA per (request, query index) with a boolean
    causal mask, and logsumexp of the masked scaled scores."""
    B, q, H = inp.batch, inp.q_len, inp.num_heads
    out = np.zeros((B, q, H, 512))
    lse = np.zeros((B, q, H))
    Q = torch.cat([inp.q_nope, inp.q_pe], dim=-1).to(torch.float64)
    for b in range(B):
        L = int(inp.seq_lens[b])
        X = gather_rows_torch(inp, b, L)  # [L, 576]
        for i in range(q):
            vis = L - q + 1 + i
            mask = torch.arange(L) < vis
            qi = Q[b, i]  # [H, 576]
            o = F.scaled_dot_product_attention(
                qi[None, :, None, :], X[None, None].expand(1, H, L, 576),
                X[None, None, :, :512].expand(1, H, L, 512),
                attn_mask=mask[None, None, None, :], scale=inp.softmax_scale)
            out[b, i] = o[0, :, 0].numpy()
            s = (qi @ X.T) * inp.softmax_scale
            s = s.masked_fill(~mask[None, :], -math.inf)
            lse[b, i] = torch.logsumexp(s, dim=-1).numpy()
    return out, lse


@pytest.mark.parametrize("q_len,kv_lens", [(1, (1, 37, 130)), (2, (2, 63, 65)), (4, (4, 64, 129)),
                                           (8, (8, 9, 200))])
def test_matches_torch_sdpa_f64(q_len, kv_lens):
    inp = small(seed=q_len, q_len=q_len, kv_lens=kv_lens)
    out, lse = oracle.decode(inp)
    ref_o, ref_l = sdpa_reference(inp)
    assert np.max(np.abs(out - ref_o)) <= 1e-12
    assert np.max(np.abs(lse - ref_l)) <= 1e-12


def test_matches_torch_sdpa_fp8_cache():
    inp = small(seed=11, q_len=2, kv_lens=(2, 70, 128), fp8=True)
    out, lse = oracle.decode(inp)
    ref_o, ref_l = sdpa_reference(inp)
    assert np.max(np.abs(out - ref_o)) <= 1e-12
    assert np.max(np.abs(lse - ref_l)) <= 1e-12


def test_sharp_queries_match_sdpa():
    inp = small(seed=5, q_len=4, kv_lens=(4, 100, 190), sharp=20.0)
    out, lse = oracle.decode(inp)
    ref_o, ref_l = sdpa_reference(inp)
    assert np.max(np.abs(out - ref_o)) <= 1e-11
    assert np.max(np.abs(lse - ref_l)) <= 1e-11


def test_unabsorbed_mha_equivalence():
    """Absorbed q_nope = W_UK^T q_orig gives the same result as explicit keys
    K = W_UK c_kv (qk_nope=128) | k_pe with V = c_kv."""
    inp = small(seed=3, q_len=2, kv_lens=(2, 50, 140), H=3)
    rng = np.random.default_rng(7)
    w_uk = rng.standard_normal((inp.num_heads, 128, 512)) / math.sqrt(512)
    q_orig = rng.standard_normal((inp.batch, inp.q_len, inp.num_heads, 128))
    q_abs = np.einsum("hed,bqhe->bqhd", w_uk, q_orig)
    q_pe = oracle.bf16_to_f64(inp.q_pe)
    out_a, lse_a = oracle.decode(inp, q=np.concatenate([q_abs, q_pe], axis=-1))
    out_u, lse_u = oracle.decode_unabsorbed(inp, q_orig, w_uk)
    assert np.max(np.abs(out_a - out_u)) <= 1e-10
    assert np.max(np.abs(lse_a - lse_u)) <= 1e-10


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_split_form_equals_single_pass(splits):
    inp = small(seed=4, q_len=4, kv_lens=(4, 129, 300, 64), B=4)
    out, lse = oracle.decode(inp)
    L = int(inp.seq_lens.max())
    chunk = max(64, ((L + splits - 1) // splits + 63) // 64 * 64)
    o2, l2, part = oracle.decode_split(inp, splits, chunk)
    assert np.max(np.abs(out - o2)) <= 1e-12
    assert np.max(np.abs(lse - l2)) <= 1e-12
    # empty splits carry o = 0 and lse = -inf
    for j in range(splits):
        if j * chunk >= L:
            assert np.all(np.isneginf(part[..., j, 512]))
            assert np.all(part[..., j, :512] == 0)


def test_single_token_returns_its_row():
    inp = small(seed=6, kv_lens=(1, 1, 1))
    out, lse = oracle.decode(inp)
    for b in range(inp.batch):
        x = gather_rows_torch(inp, b, 1)[0].numpy()
        np.testing.assert_array_equal(out[b, 0], np.broadcast_to(x[:512], out[b, 0].shape))
        qv = torch.cat([inp.q_nope[b, 0], inp.q_pe[b, 0]], -1).double().numpy()
        np.testing.assert_allclose(lse[b, 0], inp.softmax_scale * (qv @ x), rtol=0, atol=1e-12)


def test_zero_query_gives_mean_and_log_count():
    inp = small(seed=8, q_len=2, kv_lens=(2, 77, 131))
    q = np.zeros((inp.batch, inp.q_len, inp.num_heads, 576))
    out, lse = oracle.decode(inp, q=q)
    for b in range(inp.batch):
        L = int(inp.seq_lens[b])
        X = gather_rows_torch(inp, b, L).numpy()
        for i in range(inp.q_len):
            vis = L - inp.q_len + 1 + i
            np.testing.assert_allclose(out[b, i], np.broadcast_to(X[:vis, :512].mean(0), out[b, i].shape),
                                       rtol=0, atol=1e-14)
            np.testing.assert_allclose(lse[b, i], math.log(vis), rtol=0, atol=1e-13)


def test_identical_rows_return_that_row():
    inp = small(seed=9, q_len=1, kv_lens=(5, 70, 129))
    row = inp.kv_cache[int(inp.block_table[0, 0]), 0].clone()
    inp.kv_cache[:] = row
    out, lse = oracle.decode(inp)
    x = row.double().numpy()
    Q = torch.cat([inp.q_nope, inp.q_pe], -1).double().numpy()
    for b in range(inp.batch):
        L = int(inp.seq_lens[b])
        np.testing.assert_allclose(out[b, 0], np.broadcast_to(x[:512], out[b, 0].shape), rtol=0,
                                   atol=1e-14)
        s = inp.softmax_scale * (Q[b, 0] @ x)
        np.testing.assert_allclose(lse[b, 0], s + math.log(L), rtol=0, atol=1e-12)


def test_weights_sum_to_one():
    """A c_kv column that is 1 in every row returns sum_t w_t, which must be 1."""
    inp = small(seed=10, q_len=4, kv_lens=(4, 90, 199), sharp=5.0)
    inp.kv_cache[:, :, 17] = 1.0
    out, _ = oracle.decode(inp)
    assert np.max(np.abs(out[..., 17] - 1.0)) <= 1e-12


def test_mtp_rows_equal_truncated_single_query_calls():
    """Row i of a q_len call with length L equals a q_len=1 call with L - q_len + 1 + i."""
    q_len = 4
    inp = small(seed=12, q_len=q_len, kv_lens=(4, 66, 129))
    out, lse = oracle.decode(inp)
    for i in range(q_len):
        sub = synth.Inputs(**{**inp.__dict__})
        sub.q_len = 1
        sub.q_nope = inp.q_nope[:, i:i + 1].contiguous()
        sub.q_pe = inp.q_pe[:, i:i + 1].contiguous()
        sub.seq_lens = inp.seq_lens - q_len + 1 + i
        o1, l1 = oracle.decode(sub)
        np.testing.assert_array_equal(out[:, i], o1[:, 0])
        np.testing.assert_array_equal(lse[:, i], l1[:, 0])


def test_page_permutation_is_bitwise_invariant():
    inp = small(seed=13, q_len=2, kv_lens=(2, 128, 190), spare_pages=3)
    out, lse = oracle.decode(inp)
    perm = synth.permute_pages(inp, seed=99)
    assert not torch.equal(perm.block_table, inp.block_table)
    o2, l2 = oracle.decode(perm)
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(lse, l2)


def test_nan_tail_slots_are_never_read():
    clean = small(seed=14, q_len=2, kv_lens=(2, 70, 131), spare_pages=2)
    dirty = small(seed=14, q_len=2, kv_lens=(2, 70, 131), spare_pages=2, nan_tail=True)
    assert torch.isnan(dirty.kv_cache.float()).any()
    o1, l1 = oracle.decode(clean)
    o2, l2 = oracle.decode(dirty)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_request_subset_matches_full():
    inp = small(seed=15, q_len=2, kv_lens=(2, 40, 100, 7), B=4)
    out, lse = oracle.decode(inp)
    o2, l2 = oracle.decode(inp, reqs=[3, 1])
    for b in (1, 3):
        np.testing.assert_array_equal(out[b], o2[b])
        np.testing.assert_array_equal(lse[b], l2[b])
    assert np.all(np.isnan(o2[0])) and np.all(np.isnan(o2[2]))


def test_e4m3_decoder_matches_torch_on_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_f64(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2  # 0x7F and 0xFF
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_bf16_decoder_matches_torch():
    g = torch.Generator().manual_seed(0)
    x = (torch.randn(4096, generator=g) * 3).to(torch.bfloat16)
    np.testing.assert_array_equal(oracle.bf16_to_f64(x), x.to(torch.float64).numpy())


def test_rejects_short_sequences():
    inp = small(seed=16, q_len=4, kv_lens=(4, 50, 60))
    inp.seq_lens[0] = 3  # L < q_len
    with pytest.raises(ValueError):
        oracle.decode(inp)


# ---------------------------------------------------------------------------
# Token-range (sequence shard) form and the LSE merge of shard partials: the
# decode-context-parallel reading of the Triton MLA and sparse-MLA summaries
# (vLLM PR #46819 key code excerpt, q_num_heads = num_heads * dcp_world_size;
# vLLM PR #47327, implementation breakdown 1, DCP-aware workspace), where each
# rank attends over its own token range and the ranks' partials are merged.

def _sdpa_on_range(inp, lo, hi):
    """torch float64 SDPA / logsumexp of every row restricted to the positions of
    [lo[b], hi[b]) it may see; rows with nothing to see give 0 / -inf."""
    B, q, H = inp.batch, inp.q_len, inp.num_heads
    out = np.zeros((B, q, H, 512))
    lse = np.full((B, q, H), -np.inf)
    Q = torch.cat([inp.q_nope, inp.q_pe], dim=-1).to(torch.float64)
    for b in range(B):
        L = int(inp.seq_lens[b])
        X = gather_rows_torch(inp, b, L)
        for i in range(q):
            t = torch.arange(L)
            mask = (t < L - q + 1 + i) & (t >= lo[b]) & (t < hi[b])
            if not bool(mask.any()):
                continue
            qi = Q[b, i]
            o = F.scaled_dot_product_attention(
                qi[None, :, None, :], X[None, None].expand(1, H, L, 576),
                X[None, None, :, :512].expand(1, H, L, 512),
                attn_mask=mask[None, None, None, :], scale=inp.softmax_scale)
            out[b, i] = o[0, :, 0].numpy()
            s = (qi @ X.T) * inp.softmax_scale
            lse[b, i] = torch.logsumexp(s.masked_fill(~mask[None, :], -math.inf), dim=-1).numpy()
    return out, lse


def test_range_form_matches_torch_sdpa_on_the_range():
    inp = small(seed=20, q_len=4, kv_lens=(4, 70, 200, 129), B=4)
    lo, hi = [0, 10, 64, 100], [4, 69, 190, 129]  # row-dependent visibility cuts inside some ranges
    part = oracle.decode_range(inp, lo, hi)
    ref_o, ref_l = _sdpa_on_range(inp, lo, hi)
    assert np.max(np.abs(part[..., :512] - ref_o)) <= 1e-12
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(part[..., 512]), fin)
    assert np.max(np.abs(part[..., 512][fin] - ref_l[fin])) <= 1e-12


@pytest.mark.parametrize("cuts", [(1,), (2,), (3,), (4,)])
def test_ranges_tiling_the_sequence_merge_to_the_single_pass(cuts):
    R = cuts[0]
    inp = small(seed=21 + R, q_len=4, kv_lens=(4, 65, 300, 131), B=4, sharp=3.0)
    out, lse = oracle.decode(inp)
    g = np.random.default_rng(R)
    parts = []
    bounds = []
    for b in range(inp.batch):
        L = int(inp.seq_lens[b])
        inner = np.sort(g.integers(0, L + 1, size=R - 1))  # ragged, possibly empty pieces
        bounds.append(np.concatenate([[0], inner, [L]]).astype(int))
    for k in range(R):
        lo = [int(bounds[b][k]) for b in range(inp.batch)]
        hi = [int(bounds[b][k + 1]) for b in range(inp.batch)]
        parts.append(oracle.decode_range(inp, lo, hi))
    o2, l2 = oracle.lse_merge(np.stack(parts))
    assert np.max(np.abs(o2 - out)) <= 1e-12
    assert np.max(np.abs(l2 - lse)) <= 1e-12
    # the shard order does not matter
    o3, l3 = oracle.lse_merge(np.stack(parts[::-1]))
    assert np.max(np.abs(o3 - o2)) <= 1e-14 and np.max(np.abs(l3 - l2)) <= 1e-13


def test_whole_range_is_the_single_pass_bitwise():
    inp = small(seed=26, q_len=2, kv_lens=(2, 77, 140))
    out, lse = oracle.decode(inp)
    part = oracle.decode_range(inp, [0] * inp.batch, [int(x) for x in inp.seq_lens])
    np.testing.assert_array_equal(part[..., :512], out)
    np.testing.assert_array_equal(part[..., 512], lse)


def test_range_closed_forms():
    inp = small(seed=27, q_len=2, kv_lens=(2, 50, 100))
    L = [int(x) for x in inp.seq_lens]
    # one visible token t = L - 2 (seen by both query rows): out = its c_kv, lse = its score
    lo = [x - 2 for x in L]
    hi = [x - 1 for x in L]
    part = oracle.decode_range(inp, lo, hi)
    Q = torch.cat([inp.q_nope, inp.q_pe], -1).double().numpy()
    for b in range(inp.batch):
        x = gather_rows_torch(inp, b, L[b])[L[b] - 2].numpy()
        for i in range(inp.q_len):
            np.testing.assert_array_equal(part[b, i, :, :512], np.broadcast_to(x[:512], (inp.num_heads, 512)))
            np.testing.assert_allclose(part[b, i, :, 512], inp.softmax_scale * (Q[b, i] @ x), rtol=0, atol=1e-12)
    # the last position, L - 1, is visible to query row q_len-1 only: row 0 is empty
    part = oracle.decode_range(inp, [x - 1 for x in L], L)
    assert np.all(np.isneginf(part[:, 0, :, 512])) and np.all(part[:, 0, :, :512] == 0)
    assert np.all(np.isfinite(part[:, 1, :, 512]))
    # merging nothing but empty partials gives 0 / -inf
    o, l = oracle.lse_merge(np.stack([part[:, :1], part[:, :1]]))
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_range_rejects_ranges_outside_the_sequence():
    inp = small(seed=28, q_len=1, kv_lens=(5, 60))
    with pytest.raises(ValueError):
        oracle.decode_range(inp, [0, 10], [6, 60])  # past L for request 0
    with pytest.raises(ValueError):
        oracle.decode_range(inp, [3, 10], [2, 60])  # hi < lo


# ---------------------------------------------------------------------------
# FP8 query and FP8 output (the TokenSpeed MLA summary: the decode takes FP8
# scales, "output_scale" among them, in implementation breakdown 1, and its
# review names the follow-up "Fix decode FP8 numerics: pass output_scale and
# assert FP8 Q").  The query is E4M3 codes times one per-tensor q_scale; an FP8
# output is the E4M3 code of out / out_scale (round to nearest even, saturating).

def test_e4m3_encoder_matches_torch_rounding():
    # A dense sweep over the whole finite range, with every grid point, every
    # midpoint between neighbours (ties) and the float32 values on either side
    # of it, in both signs.  The values are float32 (torch rounds a float64 to
    # float32 first, and the kernel quantises float32 values), so both sides
    # round each value once.
    codes = torch.arange(0x7F, dtype=torch.int32).to(torch.uint8)
    grid = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    mids = (grid[1:] + grid[:-1]) / 2
    g = np.random.default_rng(0)
    rand = np.concatenate([g.uniform(0, 464, 20000), np.exp(g.uniform(np.log(1e-4), np.log(464), 20000))])
    xs = np.concatenate([grid, mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                         rand.astype(np.float32), [np.float32(464.0)]]).astype(np.float32)
    xs = np.concatenate([xs, -xs])
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(xs.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encoder_saturates_and_round_trips():
    big = np.array([464.0000001, 480.0, 1e9, np.inf])
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    assert oracle.e4m3_encode(np.array([np.nan]))[0] == 0x7F
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.e4m3_encode(oracle.e4m3_to_f64(finite)), finite)


@pytest.mark.parametrize("q_len", [1, 2])
def test_fp8_query_matches_torch_sdpa_on_dequantised_values(q_len):
    inp = small(seed=30 + q_len, q_len=q_len, kv_lens=(q_len, 70, 190), fp8=True, q_fp8=True, sharp=3.0)
    assert inp.q_nope.dtype == torch.uint8 and inp.q_scale != 1.0
    out, lse = oracle.decode(inp)
    # torch's own float8 decode of the same codes, times the scale
    deq = synth.Inputs(**{**inp.__dict__})
    deq.q_nope = inp.q_nope.view(torch.float8_e4m3fn).to(torch.float64) * inp.q_scale
    deq.q_pe = inp.q_pe.view(torch.float8_e4m3fn).to(torch.float64) * inp.q_scale
    deq.q_fp8 = False
    ref_o, ref_l = sdpa_reference(deq)
    assert np.max(np.abs(out - ref_o)) <= 1e-12
    assert np.max(np.abs(lse - ref_l)) <= 1e-12
