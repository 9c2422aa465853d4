"""Test-side driver for the CUDA path: runs the three C-ABI calls on one
workload and returns host copies of everything they wrote."""

from __future__ import annotations

import numpy as np
import torch

import paged_kv_attention_prepare_gb300 as pa


def to_dev(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def run_step(w, vals, *, workspace_bytes=None, qsl_capacity=None, dev="cuda",
             shared_blocks=None, fused=False):
    """prep -> cache write -> attention on the GPU, on copies of the pools.

    ``vals`` holds the generator's tensors (any device).  Returns a dict with
    host numpy index arrays, the written pools (torch, on the GPU), the
    attention output (torch, on the GPU) and the status word.
    ``shared_blocks`` (the PA_ATTN_SHARED_BLOCKS flag) defaults to whether
    the workload's tables share blocks.  ``fused`` runs the index build and
    the cache write as one call (pa_prepare_and_write)."""
    if shared_blocks is None:
        shared_blocks = w.shares_blocks
    i32 = torch.int32
    R, T = w.num_reqs, w.num_tokens
    cap = R + 1 if qsl_capacity is None else qsl_capacity
    nst, nct, bt = (to_dev(w.num_scheduled_tokens), to_dev(w.num_computed_tokens),
                    to_dev(w.block_table))
    out = {k: torch.full((T,), -7, dtype=i32, device=dev)
           for k in ("req_indices", "positions", "slot_mapping")}
    out["query_start_loc"] = torch.full((cap,), -7, dtype=i32, device=dev)
    out["seq_lens"] = torch.full((R,), -7, dtype=i32, device=dev)
    out["logits_indices"] = torch.full((R,), -7, dtype=i32, device=dev)
    kc = vals["key_cache"].to(dev).clone()
    vc = vals["value_cache"].to(dev).clone()
    key = vals["key"].to(dev) if vals["key"].device.type != "cuda" else vals["key"]
    value = vals["value"].to(dev) if vals["value"].device.type != "cuda" else vals["value"]
    ks, vs = vals.get("k_scale"), vals.get("v_scale")   # FP8 pools only
    if ks is not None:
        ks, vs = ks.to(dev), vs.to(dev)
    idx = (out["req_indices"], out["positions"], out["slot_mapping"], out["query_start_loc"],
           out["seq_lens"], out["logits_indices"])
    if fused:
        pa.pa_prepare_and_write(nst, nct, bt, w.block_size, T, w.num_blocks, *idx, key, value,
                                kc, vc, k_scale=ks, v_scale=vs)
    else:
        pa.pa_prepare_inputs(nst, nct, bt, w.block_size, T, w.num_blocks, *idx)
        pa.pa_cache_write(key, value, kc, vc, out["slot_mapping"], k_scale=ks, v_scale=vs)
    q = vals["q"].to(dev).contiguous()
    o = torch.full_like(q, float("nan"))
    if workspace_bytes is None:
        workspace_bytes = pa.pa_attention_workspace_size(R, T, w.max_query_len, w.max_seq_len,
                                                         w.num_q_heads, w.num_kv_heads,
                                                         w.head_dim)
    ws = torch.empty(max(int(workspace_bytes), 1), dtype=torch.uint8, device=dev)
    pa.pa_attention(q, kc, vc, bt, out["query_start_loc"][: R + 1], out["seq_lens"],
                    w.max_query_len, w.max_seq_len, w.scale, o,
                    ws if workspace_bytes else None, k_scale=ks, v_scale=vs,
                    shared_blocks=shared_blocks)
    status, detail = pa.pa_get_status()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res.update(key_cache=kc, value_cache=vc, out=o, status=status, detail=detail)
    return res
