"""CPU oracle for absorbed-form MLA decode over a paged latent KV cache.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm use it; the product path never does.
It is plain C (``mla_oracle.c``) evaluated in fp64, loaded through ctypes, and
shares no code with the CUDA library.  See ``mla_oracle.c`` for the definition
it evaluates and the sources it follows.

Every function here is pinned by tests/test_oracle.py against things other
than itself: torch's float64 scaled_dot_product_attention and logsumexp on tiny
inputs, the un-absorbed (explicit W_UK) MHA form, closed forms (single token,
zero query, identical rows), the causal equivalence of MTP rows, page
permutation invariance, and torch's float8_e4m3fn decode on all 256 codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "libmla_oracle.so")
_lib = None

KV_LORA_RANK = 512
QK_ROPE_DIM = 64
KV_ROW = 576


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-shared", "-fPIC", "-o", tmp, _SRC,
             "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.oracle_mla_decode.argtypes = [I, I, I, I, P, P, I, D, P, I, P, D, P, I, P, P, I]
        lib.oracle_mla_decode.restype = I
        lib.oracle_mla_decode_split.argtypes = [I, I, I, I, P, P, I, D, P, I, P, D, I, I, P, P, P, I]
        lib.oracle_mla_decode_split.restype = I
        lib.oracle_mla_decode_unabsorbed.argtypes = [I, I, I, I, P, I, P, P, P, I, D, P, I, P, D,
                                                     P, P, I]
        lib.oracle_mla_decode_unabsorbed.restype = I
        lib.oracle_mla_decode_range.argtypes = [I, I, I, I, P, P, I, D, P, I, P, D, P, P, P, I]
        lib.oracle_mla_decode_range.restype = I
        lib.oracle_lse_merge.argtypes = [ctypes.c_int64, I, P, P, P]
        lib.oracle_lse_merge.restype = None
        lib.oracle_e4m3_encode_array.argtypes = [P, P, ctypes.c_int64]
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_bf16_array_to_double.argtypes = [P, P, ctypes.c_int64]
        lib.oracle_e4m3_array_to_double.argtypes = [P, P, ctypes.c_int64]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """Decode bf16 values (given as a bf16 or int16 tensor) to float64 with the C decoder."""
    bits = np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy()).view(np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_bf16_array_to_double(_ptr(bits), _ptr(out), bits.size)
    return out


def e4m3_to_f64(codes: torch.Tensor | np.ndarray) -> np.ndarray:
    """Decode e4m3 byte codes to float64 with the C decoder."""
    if isinstance(codes, torch.Tensor):
        codes = codes.detach().cpu().contiguous().view(torch.uint8).numpy()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    _load().oracle_e4m3_array_to_double(_ptr(codes), _ptr(out), codes.size)
    return out


def e4m3_encode(x) -> np.ndarray:
    """Round float64 values to OCP E4M3 codes (nearest, ties to even, saturating to
    +-448) with the C encoder."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def query_f64(inp) -> np.ndarray:
    """[B, q, H, 576] float64 query rows q_nope | q_pe: bf16 values, or, for an FP8
    query, e4m3 codes times the per-tensor q_scale (decoded by the C decoder)."""
    if getattr(inp, "q_fp8", False):
        qn = e4m3_to_f64(inp.q_nope) * float(inp.q_scale)
        qp = e4m3_to_f64(inp.q_pe) * float(inp.q_scale)
    else:
        qn = bf16_to_f64(inp.q_nope)
        qp = bf16_to_f64(inp.q_pe)
    return np.concatenate([qn, qp], axis=-1)


class _Host:
    """Host (numpy) views of an input problem, restricted to what the oracle reads."""

    def __init__(self, inp, q: Optional[np.ndarray] = None):
        self.B, self.H, self.q_len, self.ps = inp.batch, inp.num_heads, inp.q_len, inp.page_size
        if q is None:
            q = query_f64(inp)
        self.q = np.ascontiguousarray(q, dtype=np.float64)
        kv = inp.kv_cache.detach().cpu().contiguous()
        if inp.kv_fp8:
            self.kv = kv.view(torch.uint8).numpy()
        else:
            self.kv = kv.view(torch.int16).numpy()
        self.kv_fp8 = int(bool(inp.kv_fp8))
        self.kv_scale = float(inp.kv_scale)
        self.bt = np.ascontiguousarray(inp.block_table.detach().cpu().numpy().astype(np.int32))
        self.seq = np.ascontiguousarray(inp.seq_lens.detach().cpu().numpy().astype(np.int32))
        self.scale = float(inp.softmax_scale)


def decode(inp, reqs: Optional[Sequence[int]] = None, threads: Optional[int] = None,
           q: Optional[np.ndarray] = None, softmax_scale: Optional[float] = None):
    """Single-pass oracle.  Returns (out [B,q,H,512] f64, lse [B,q,H] f64); rows of
    requests outside ``reqs`` are left NaN."""
    h = _Host(inp, q)
    scale = h.scale if softmax_scale is None else float(softmax_scale)
    out = np.full((h.B, h.q_len, h.H, KV_LORA_RANK), np.nan)
    lse = np.full((h.B, h.q_len, h.H), np.nan)
    r = None if reqs is None else np.ascontiguousarray(np.asarray(reqs, dtype=np.int32))
    rc = _load().oracle_mla_decode(
        h.B, h.H, h.q_len, h.ps, _ptr(h.q), _ptr(h.kv), h.kv_fp8, h.kv_scale, _ptr(h.bt),
        h.bt.shape[1], _ptr(h.seq), scale, _ptr(r), 0 if r is None else r.size, _ptr(out),
        _ptr(lse), threads or default_threads())
    if rc:
        raise ValueError(f"oracle_mla_decode rejected its arguments (code {rc})")
    return out, lse


def decode_split(inp, num_splits: int, chunk_tokens: int, threads: Optional[int] = None):
    """Split form: returns (out, lse, partials [B,q,H,s,513])."""
    h = _Host(inp)
    out = np.zeros((h.B, h.q_len, h.H, KV_LORA_RANK))
    lse = np.zeros((h.B, h.q_len, h.H))
    part = np.zeros((h.B, h.q_len, h.H, num_splits, KV_LORA_RANK + 1))
    rc = _load().oracle_mla_decode_split(
        h.B, h.H, h.q_len, h.ps, _ptr(h.q), _ptr(h.kv), h.kv_fp8, h.kv_scale, _ptr(h.bt),
        h.bt.shape[1], _ptr(h.seq), h.scale, num_splits, chunk_tokens, _ptr(part), _ptr(out),
        _ptr(lse), threads or default_threads())
    if rc:
        raise ValueError(f"oracle_mla_decode_split rejected its arguments (code {rc})")
    return out, lse, part


def decode_unabsorbed(inp, q_orig: np.ndarray, w_uk: np.ndarray, threads: Optional[int] = None):
    """Explicit-MHA form with keys W_UK,h c_kv | k_pe; q_orig [B,q,H,d], w_uk [H,d,512]."""
    h = _Host(inp)
    q_orig = np.ascontiguousarray(q_orig, dtype=np.float64)
    w_uk = np.ascontiguousarray(w_uk, dtype=np.float64)
    d = q_orig.shape[-1]
    out = np.zeros((h.B, h.q_len, h.H, KV_LORA_RANK))
    lse = np.zeros((h.B, h.q_len, h.H))
    rc = _load().oracle_mla_decode_unabsorbed(
        h.B, h.H, h.q_len, h.ps, _ptr(q_orig), d, _ptr(w_uk), _ptr(h.q), _ptr(h.kv), h.kv_fp8,
        h.kv_scale, _ptr(h.bt), h.bt.shape[1], _ptr(h.seq), h.scale, _ptr(out), _ptr(lse),
        threads or default_threads())
    if rc:
        raise ValueError(f"oracle_mla_decode_unabsorbed rejected its arguments (code {rc})")
    return out, lse


def decode_range(inp, range_lo: Sequence[int], range_hi: Sequence[int], threads: Optional[int] = None):
    """Token-range (sequence shard) form: every row (b, i, h) attends to the positions of
    [range_lo[b], range_hi[b]) it may see.  Returns partials [B, q, H, 513] (512
    normalised outputs, then the range's LSE; an empty range gives 0 and -inf)."""
    h = _Host(inp)
    lo = np.ascontiguousarray(np.asarray(range_lo, dtype=np.int32))
    hi = np.ascontiguousarray(np.asarray(range_hi, dtype=np.int32))
    assert lo.shape == (h.B,) and hi.shape == (h.B,)
    part = np.zeros((h.B, h.q_len, h.H, KV_LORA_RANK + 1))
    rc = _load().oracle_mla_decode_range(
        h.B, h.H, h.q_len, h.ps, _ptr(h.q), _ptr(h.kv), h.kv_fp8, h.kv_scale, _ptr(h.bt),
        h.bt.shape[1], _ptr(h.seq), h.scale, _ptr(lo), _ptr(hi), _ptr(part),
        threads or default_threads())
    if rc:
        raise ValueError(f"oracle_mla_decode_range rejected its arguments (code {rc})")
    return part


def lse_merge(parts: np.ndarray):
    """LSE merge of partials stacked shard-major, parts [R, ..., 513] -> (out [..., 512], lse [...])."""
    parts = np.ascontiguousarray(parts, dtype=np.float64)
    R = parts.shape[0]
    lead = parts.shape[1:-1]
    rows = int(np.prod(lead)) if lead else 1
    out = np.zeros(lead + (KV_LORA_RANK,))
    lse = np.zeros(lead)
    _load().oracle_lse_merge(rows, R, _ptr(parts), _ptr(out), _ptr(lse))
    return out, lse
