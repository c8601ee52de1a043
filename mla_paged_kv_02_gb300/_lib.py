"""ctypes binding for libmla_decode.so (argument marshalling only).

Every step of the decode runs in the CUDA library; this module only turns torch
tensors into pointers, sizes and strides and returns the C status.  It raises
if the shared library is missing: there is no Python or CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_decode.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE_TOO_SMALL = 3
MLA_ERR_CUDA = 4
MLA_ERR_DEVICE_INPUT = 5
MLA_ERR_TIMEOUT = 6

MLA_KV_BF16 = 0
MLA_KV_FP8_E4M3 = 1
MLA_OUT_BF16 = 0
MLA_OUT_FP32 = 1
MLA_OUT_FP8_E4M3 = 2

# Every symbol include/mla_decode.h declares.
EXPORTED = (
    "mla_decode_plan",
    "mla_decode_plan_lengths",
    "mla_workspace_init",
    "mla_decode",
    "mla_split_kv",
    "mla_combine",
    "mla_decode_check_error",
    "mla_decode_noalloc",
    "mla_decode_varlen",
    "mla_decode_fp8",
    "mla_decode_shard",
    "mla_combine_shards",
    "mla_status_string",
)


class Plan(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("num_heads", ctypes.c_int),
        ("q_len", ctypes.c_int),
        ("max_seq_len", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("kv_dtype", ctypes.c_int),
        ("num_sms", ctypes.c_int),
        ("num_kv_splits", ctypes.c_int),
        ("chunk_tokens", ctypes.c_int),
        ("rows_per_cta", ctypes.c_int),
        ("row_groups", ctypes.c_int),
        ("reserved", ctypes.c_int * 3),
        ("partial_bytes", ctypes.c_size_t),
        ("workspace_bytes", ctypes.c_size_t),
    ]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_ if f != "reserved"}


class MlaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


_lib = None
_debug_lib = None
DEBUG_LIB_PATH = os.path.join(_HERE, "libmla_decode_debug.so")


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    _lib = _open(LIB_PATH)
    return _lib


def load_debug() -> ctypes.CDLL:
    """The debug build (same kernels, plus mla_debug_set_wait_limit_ns); tests only."""
    global _debug_lib
    if _debug_lib is None:
        lib = _open(DEBUG_LIB_PATH)
        lib.mla_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.mla_debug_set_wait_limit_ns.restype = ctypes.c_int
        _debug_lib = lib
    return _debug_lib


def _open(path: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library {path} is missing; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    PP = ctypes.POINTER(Plan)
    lib.mla_decode_plan.argtypes = [I, I, I, I, I, I, I, I, PP]
    lib.mla_decode_plan_lengths.argtypes = [I, I, I, P, I, I, I, PP]
    lib.mla_workspace_init.argtypes = [P, SZ, P]
    decode_args = [PP, P, I64, P, I64, P, I, P, I, P, F, P, P, I, P, P, SZ, P]
    lib.mla_decode.argtypes = decode_args
    lib.mla_split_kv.argtypes = decode_args
    lib.mla_combine.argtypes = [PP, P, I, P, P, SZ, P]
    lib.mla_decode_check_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
    lib.mla_decode_noalloc.argtypes = [PP, P, I64, P, I64, P, I, P, I, P, F, P, P, I, P, P]
    lib.mla_decode_varlen.argtypes = [PP, P, I64, P, I64, P, I, P, I, P, P, F, P, P, I, P, P, SZ, P]
    lib.mla_decode_fp8.argtypes = [PP, P, I64, P, I64, P, P, I, P, I, P, F, P, P, I, P, P, P, SZ, P]
    lib.mla_decode_shard.argtypes = [PP, P, I64, P, I64, P, I, P, I, P, P, P, F, P, P, P, SZ, P]
    lib.mla_combine_shards.argtypes = [I64, I, P, P, I, P, P]
    lib.mla_status_string.argtypes = [I]
    lib.mla_status_string.restype = ctypes.c_char_p
    for name in EXPORTED:
        if name != "mla_status_string":
            getattr(lib, name).restype = I
    return lib


def status_string(status: int) -> str:
    return load().mla_status_string(int(status)).decode()


def plan(batch: int, num_heads: int, q_len: int, max_seq_len: int, kv_fp8: bool = False,
         num_sms: int = 0, force_splits: int = 0, page_size: int = 64) -> Plan:
    p = Plan()
    st = load().mla_decode_plan(batch, num_heads, q_len, max_seq_len, page_size,
                                MLA_KV_FP8_E4M3 if kv_fp8 else MLA_KV_BF16, num_sms, force_splits,
                                ctypes.byref(p))
    if st != MLA_OK:
        raise MlaError(st, "mla_decode_plan")
    return p


def plan_lengths(num_heads: int, q_len: int, seq_lens, kv_fp8: bool = False, num_sms: int = 0,
                 page_size: int = 64) -> Plan:
    """mla_decode_plan_lengths: the split count from the batch's own lengths
    (any int sequence or tensor; copied to host int32)."""
    lens = torch.as_tensor(seq_lens).to(device="cpu", dtype=torch.int32).contiguous()
    p = Plan()
    st = load().mla_decode_plan_lengths(int(lens.numel()), num_heads, q_len, ctypes.c_void_p(lens.data_ptr()),
                                        page_size, MLA_KV_FP8_E4M3 if kv_fp8 else MLA_KV_BF16, num_sms,
                                        ctypes.byref(p))
    if st != MLA_OK:
        raise MlaError(st, "mla_decode_plan_lengths")
    return p


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def workspace_init(workspace: torch.Tensor, stream=None) -> int:
    return load().mla_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream))


def _decode_args(pl: Plan, q_nope, q_pe, kv_cache, block_table, seq_lens, softmax_scale, kv_scale,
                 out, lse, workspace, stream):
    return (ctypes.byref(pl), _ptr(q_nope), q_nope.stride(-2), _ptr(q_pe), q_pe.stride(-2),
            _ptr(kv_cache), kv_cache.shape[0], _ptr(block_table), block_table.stride(0),
            _ptr(seq_lens), float(softmax_scale), _ptr(kv_scale), _ptr(out),
            MLA_OUT_FP32 if out.dtype == torch.float32 else MLA_OUT_BF16, _ptr(lse),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))


def decode(pl: Plan, q_nope, q_pe, kv_cache, block_table, seq_lens, softmax_scale, kv_scale, out,
           lse, workspace, stream=None) -> int:
    """mla_decode; returns the C status (0 = launched)."""
    return load().mla_decode(*_decode_args(pl, q_nope, q_pe, kv_cache, block_table, seq_lens,
                                           softmax_scale, kv_scale, out, lse, workspace, stream))


def decode_varlen(pl: Plan, q_nope, q_pe, kv_cache, block_table, seq_lens, q_lens, softmax_scale, kv_scale,
                  out, lse, workspace, stream=None) -> int:
    """mla_decode_varlen: per-request q_len (layouts padded to the plan's q_len)."""
    a = _decode_args(pl, q_nope, q_pe, kv_cache, block_table, seq_lens, softmax_scale, kv_scale, out, lse,
                     workspace, stream)
    return load().mla_decode_varlen(*a[:10], _ptr(q_lens), *a[10:])


def split_kv(pl: Plan, q_nope, q_pe, kv_cache, block_table, seq_lens, softmax_scale, kv_scale, out,
             lse, workspace, stream=None) -> int:
    return load().mla_split_kv(*_decode_args(pl, q_nope, q_pe, kv_cache, block_table, seq_lens,
                                             softmax_scale, kv_scale, out, lse, workspace, stream))


def combine(pl: Plan, out, lse, workspace, stream=None) -> int:
    return load().mla_combine(ctypes.byref(pl), _ptr(out),
                              MLA_OUT_FP32 if out.dtype == torch.float32 else MLA_OUT_BF16,
                              _ptr(lse), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))


def check_error(workspace, stream=None):
    """Returns (status, [code, request, index, value]) and clears the sticky error word."""
    info = (ctypes.c_int32 * 4)()
    st = load().mla_decode_check_error(_ptr(workspace), _stream(stream), info)
    return st, list(info)


def decode_noalloc(pl: Plan, q_nope, q_pe, kv_cache, block_table, seq_lens, softmax_scale, kv_scale,
                   out, lse, stream=None) -> int:
    """mla_decode_noalloc: the library's own fixed scratch array stands in for the workspace."""
    return load().mla_decode_noalloc(
        ctypes.byref(pl), _ptr(q_nope), q_nope.stride(-2), _ptr(q_pe), q_pe.stride(-2), _ptr(kv_cache),
        kv_cache.shape[0], _ptr(block_table), block_table.stride(0), _ptr(seq_lens), float(softmax_scale),
        _ptr(kv_scale), _ptr(out), MLA_OUT_FP32 if out.dtype == torch.float32 else MLA_OUT_BF16, _ptr(lse),
        _stream(stream))


def decode_shard(pl: Plan, q_nope, q_pe, kv_cache, block_table, shard_lens, shard_start, seq_lens,
                 softmax_scale, kv_scale, shard_partial, workspace, stream=None) -> int:
    """mla_decode_shard: this rank's (o, lse) partial [B, q, H, 513] over its token range."""
    return load().mla_decode_shard(
        ctypes.byref(pl), _ptr(q_nope), q_nope.stride(-2), _ptr(q_pe), q_pe.stride(-2), _ptr(kv_cache),
        kv_cache.shape[0], _ptr(block_table), block_table.stride(0), _ptr(shard_lens), _ptr(shard_start),
        _ptr(seq_lens), float(softmax_scale), _ptr(kv_scale), _ptr(shard_partial), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))


def combine_shards(shard_partials, out, lse, stream=None) -> int:
    """mla_combine_shards: merge [R, rows..., 513] shard partials into out / lse."""
    R = shard_partials.shape[0]
    rows = shard_partials[0].numel() // 513
    return load().mla_combine_shards(rows, R, _ptr(shard_partials), _ptr(out),
                                     MLA_OUT_FP32 if out.dtype == torch.float32 else MLA_OUT_BF16, _ptr(lse),
                                     _stream(stream))


def out_dtype_code(out: torch.Tensor) -> int:
    if out.dtype == torch.float32:
        return MLA_OUT_FP32
    if out.dtype == torch.uint8:
        return MLA_OUT_FP8_E4M3
    return MLA_OUT_BF16


def decode_fp8(pl: Plan, q_nope, q_pe, q_scale, kv_cache, block_table, seq_lens, softmax_scale, kv_scale, out,
               out_scale, lse, workspace, stream=None) -> int:
    """mla_decode_fp8: e4m3 query codes (uint8) with a device q_scale; ``out`` as
    uint8 selects an FP8 output (codes of out / out_scale)."""
    return load().mla_decode_fp8(
        ctypes.byref(pl), _ptr(q_nope), q_nope.stride(-2), _ptr(q_pe), q_pe.stride(-2), _ptr(q_scale),
        _ptr(kv_cache), kv_cache.shape[0], _ptr(block_table), block_table.stride(0), _ptr(seq_lens),
        float(softmax_scale), _ptr(kv_scale), _ptr(out), out_dtype_code(out), _ptr(out_scale), _ptr(lse),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
