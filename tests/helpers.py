"""Test-side helpers: hand-built small cases and independent restatements
used to pin the oracle.  Nothing here is imported by the library."""

from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


ATOL = 1e-2


def attention_tolerance(ref: np.ndarray, out_dtype: torch.dtype) -> np.ndarray:
    """Per-element bound on |gpu - oracle| for an attention output of type
    ``out_dtype``: 1e-2 (bf16/fp16 output, fp32 accumulation).  Where the
    type's spacing near the exact value is so coarse that no value of the type
    need lie within 1e-2 of it (|o| >= 4 in bf16, |o| >= 32 in fp16: half a
    spacing is 1/64 or more), the bound is that half spacing plus the
    arithmetic's share, which grows with the output: 2^-10 |o| + 2e-3 (the
    softmax weights carry 11 significant bits or more)."""
    bits = 8 if out_dtype == torch.bfloat16 else 11      # significant bits of the type
    a = np.abs(ref)
    e = np.floor(np.log2(np.maximum(a, np.finfo(np.float64).tiny)))
    coarse = np.exp2(e - bits) + a * 2.0 ** -10 + 2e-3
    return np.where(np.exp2(e - bits) + 2e-3 > ATOL, coarse, ATOL)


# (test, output dtype, largest error where the bound is 1e-2, largest error
# elsewhere, elements compared) of every check_attention_close call; written
# out at the end of a session when PA_ERROR_LOG names a file
ERRORS: list = []


def check_attention_close(got: np.ndarray, ref: np.ndarray, out_dtype: torch.dtype) -> float:
    """Assert every element of ``got`` within ``attention_tolerance`` of the
    oracle's ``ref``; returns the largest absolute error."""
    assert np.isfinite(got).all()
    if got.size == 0:
        return 0.0
    err = np.abs(got - ref)
    tol = attention_tolerance(ref, out_dtype)
    plain = tol <= ATOL
    ERRORS.append((os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], str(out_dtype),
                   float(err[plain].max()) if plain.any() else 0.0,
                   float(err[~plain].max()) if (~plain).any() else 0.0, int(err.size)))
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (f"{len(bad)} elements past the bound; max abs error {err.max()} "
                           f"at {np.unravel_index(np.argmax(err), err.shape)}; first bad "
                           f"{tuple(bad[0])}: got {got[tuple(bad[0])]}, oracle {ref[tuple(bad[0])]}")
    return float(err.max())


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype)


def scatter_to_pool(contig_k, contig_v, ctx_lens, block_size, num_blocks, rng, dtype):
    """Lay per-request contiguous K/V (lists of [L_r, Hkv, D] float tensors) into
    a pool at random physical blocks.  Returns (key_cache, value_cache, table)."""
    need = [-(-int(l) // block_size) for l in ctx_lens]
    perm = rng.permutation(num_blocks)
    hkv, d = contig_k[0].shape[1], contig_k[0].shape[2]
    kc = torch.randn(num_blocks, block_size, hkv, d, dtype=torch.float32).to(dtype)
    vc = torch.randn(num_blocks, block_size, hkv, d, dtype=torch.float32).to(dtype)
    width = max(need) if need else 1
    bt = np.full((len(ctx_lens), max(width, 1)), -1, np.int32)
    k = 0
    for r, l in enumerate(ctx_lens):
        blocks = perm[k : k + need[r]]
        k += need[r]
        bt[r, : need[r]] = blocks
        for j in range(int(l)):
            kc[blocks[j // block_size], j % block_size] = contig_k[r][j]
            vc[blocks[j // block_size], j % block_size] = contig_v[r][j]
    return kc, vc, bt


def brute_prepare(nst, nct, bt, bs):
    """Token-centric restatement of the index build: for each flat token find
    its request by walking the running sum, then apply the slot rule."""
    total = int(sum(nst))
    starts, acc = [], 0
    for n in nst:
        starts.append(acc)
        acc += int(n)
    req, pos, slot = [], [], []
    for t in range(total):
        r = max(i for i in range(len(nst)) if starts[i] <= t)
        p = int(nct[r]) + (t - starts[r])
        blk, off = divmod(p, bs)
        req.append(r)
        pos.append(p)
        slot.append(int(bt[r][blk]) * bs + off)
    qsl = starts + [acc]
    return {
        "req_indices": req, "positions": pos, "slot_mapping": slot,
        "query_start_loc": qsl,
        "seq_lens": [int(c) + int(n) for c, n in zip(nct, nst)],
        "logits_indices": [qsl[i + 1] - 1 for i in range(len(nst))],
    }


def brute_attention(q, kc, vc, bt, qsl, seq_lens, bs, scale):
    """Pure-Python softmax attention with math.fsum, one (token, head) at a
    time.  q: float64 [T,Hq,D]; kc/vc: float64 [NB,bs,Hkv,D]."""
    t_all, hq, d = q.shape
    hkv = kc.shape[2]
    out = np.zeros_like(q)
    for r in range(len(seq_lens)):
        n = qsl[r + 1] - qsl[r]
        for i in range(n):
            t = qsl[r] + i
            p = seq_lens[r] - n + i
            for h in range(hq):
                kvh = (h * hkv) // hq
                keys = [(bt[r][j // bs], j % bs) for j in range(p + 1)]
                logits = [scale * math.fsum(q[t, h, e] * kc[b, o, kvh, e] for e in range(d))
                          for b, o in keys]
                top = max(logits)
                wts = [math.exp(x - top) for x in logits]
                z = math.fsum(wts)
                for e in range(d):
                    out[t, h, e] = math.fsum(w * vc[b, o, kvh, e]
                                             for w, (b, o) in zip(wts, keys)) / z
    return out


def dense_causal_numpy(qr, kr, vr, first_pos, scale):
    """Dense causal attention with NumPy matmuls.  qr [n,Hq,D], kr/vr [L,Hkv,D]
    contiguous (unpaged); query i sits at position first_pos + i."""
    n, hq, d = qr.shape
    length, hkv, _ = kr.shape
    g = hq // hkv
    out = np.empty((n, hq, d))
    qpos = first_pos + np.arange(n)
    masked = np.arange(length)[None, :] > qpos[:, None]
    for h in range(hq):
        s = (qr[:, h, :] @ kr[:, h // g, :].T) * scale
        s[masked] = -np.inf
        s -= s.max(axis=1, keepdims=True)
        pr = np.exp(s)
        pr /= pr.sum(axis=1, keepdims=True)
        out[:, h, :] = pr @ vr[:, h // g, :]
    return out
