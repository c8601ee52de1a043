"""Torch plumbing around the C ABI: allocate out/lse/workspace and call mla_decode.

Allocation happens here, once, with torch; the library itself never allocates.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from . import _lib


def plan_for(inp, force_splits: int = 0, num_sms: int = 0, max_seq_len: Optional[int] = None) -> _lib.Plan:
    """The plan for ``inp``: from its own lengths (mla_decode_plan_lengths) unless
    a split count is forced or the plan must cover longer calls (max_seq_len)."""
    if force_splits == 0 and max_seq_len is None:
        return _lib.plan_lengths(inp.num_heads, inp.q_len, inp.seq_lens, kv_fp8=inp.kv_fp8, num_sms=num_sms)
    return _lib.plan(inp.batch, inp.num_heads, inp.q_len,
                     max_seq_len if max_seq_len is not None else inp.max_seq_len,
                     kv_fp8=inp.kv_fp8, num_sms=num_sms, force_splits=force_splits)


def alloc_workspace(pl: _lib.Plan, device, stream=None) -> torch.Tensor:
    ws = torch.empty(pl.workspace_bytes, dtype=torch.uint8, device=device)
    st = _lib.workspace_init(ws, stream)
    if st != _lib.MLA_OK:
        raise _lib.MlaError(st, "mla_workspace_init")
    return ws


def alloc_outputs(inp, out_fp32: Optional[bool] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    fp32 = inp.out_fp32 if out_fp32 is None else out_fp32
    dev = inp.q_nope.device
    out = torch.empty((inp.batch, inp.q_len, inp.num_heads, 512),
                      dtype=torch.float32 if fp32 else torch.bfloat16, device=dev)
    lse = torch.empty((inp.batch, inp.q_len, inp.num_heads), dtype=torch.float32, device=dev)
    return out, lse


def kv_scale_tensor(inp) -> Optional[torch.Tensor]:
    if not inp.kv_fp8:
        return None
    return torch.tensor([inp.kv_scale], dtype=torch.float32, device=inp.q_nope.device)


def decode(inp, pl: Optional[_lib.Plan] = None, force_splits: int = 0, out_fp32: Optional[bool] = None,
           workspace: Optional[torch.Tensor] = None, stream=None, check: bool = True,
           q_lens: Optional[torch.Tensor] = None):
    """Run one decode on ``inp`` (tensors already on the GPU).  Returns (out, lse, plan).

    ``q_lens`` (int32 [B] on the GPU) selects mla_decode_varlen: request b uses
    its first q_lens[b] query tokens of the padded ``inp.q_len``."""
    if pl is None:
        pl = plan_for(inp, force_splits=force_splits)
    if workspace is None:
        workspace = alloc_workspace(pl, inp.q_nope.device, stream)
    out, lse = alloc_outputs(inp, out_fp32)
    kvs = kv_scale_tensor(inp)
    if q_lens is None:
        st = _lib.decode(pl, inp.q_nope.view(-1, 512), inp.q_pe.view(-1, 64), inp.kv_cache,
                         inp.block_table, inp.seq_lens, inp.softmax_scale, kvs, out, lse, workspace, stream)
    else:
        st = _lib.decode_varlen(pl, inp.q_nope.view(-1, 512), inp.q_pe.view(-1, 64), inp.kv_cache,
                                inp.block_table, inp.seq_lens, q_lens, inp.softmax_scale, kvs, out, lse,
                                workspace, stream)
    if st != _lib.MLA_OK:
        raise _lib.MlaError(st, "mla_decode")
    if check:
        st, info = _lib.check_error(workspace, stream)
        if st != _lib.MLA_OK:
            raise _lib.MlaError(st, f"mla_decode device check {info}")
    return out, lse, pl
