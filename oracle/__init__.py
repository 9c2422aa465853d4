"""CPU oracle for the paged-KV attention step -- TEST INFRASTRUCTURE ONLY.

Thin ctypes wrappers around ``pa_oracle.c`` (plain C, fp64).  Only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg import this
package; the CUDA library and its Python binding never do.

Parity status of each function (how it is pinned, in ``tests/test_oracle.py``):

* ``prepare_inputs`` -- pinned by the pages' printed worked examples
  (``tests/golden/``), hand-derived exercise answers, invariants and a brute
  force against a separately written pure-Python restatement.
* ``gather_input_ids`` -- pinned by the printed token_indices comment
  ([0, 1, M, M+1, ..., 2M+2] for query positions [0, 1, 0, 1, 2, 3, 4, 0, 1, 2])
  and the Go program's input_ids (token ids 100.., 200.., 300..), plus
  invariants (each id comes from its own request's row at its position).
* ``discard_request_mask`` -- pinned by the printed [False, True, True] of the
  [2, 5, 3] example and the Go program's per-request verdicts.
* ``spec_logits_indices`` -- pinned by the printed no-draft rows [1, 6, 9]
  (drafts all zero reduce to query_start_loc[1:] - 1) and by invariants of the
  draft case (length R + sum(d); each request's rows are consecutive, inside
  its own slice and end on its last row).
* ``copy_blocks`` / ``zero_blocks`` -- pinned by NumPy block slicing (a
  library copy), untouched-block preservation, and the beam-search scenario
  (after a copy and a table remap, the diverging beam attends over exactly
  what it attended over before, and its new token no longer reaches the
  other beam).
* ``e4m3_decode`` / ``e4m3_encode`` -- pinned by PyTorch's float8_e4m3fn
  conversions (every code; random values inside the finite range), closed
  forms (448, 2^-6, 2^-9, 1), round trips of every finite code, ties to even
  and saturation.
* ``cache_write_fp8`` -- pinned by PyTorch's fp32 division and float8 rounding
  of the same elements and untouched-slot preservation.
* ``attention(kv_cache_dtype="fp8_e4m3")`` -- pinned by equality with
  attention over 16-bit pools holding the same values (power-of-two scales
  keep them exact).
* ``cache_write`` -- pinned by bit equality against a direct per-slot copy,
  untouched-slot preservation and write-then-gather round trips.
* ``attention`` -- pinned by closed forms (one visible key, K = 0, constant V,
  one dominant key), a pure-Python ``math.fsum`` brute force on tiny inputs,
  NumPy dense causal attention on the unpaged K/V, and invariances (physical
  block permutation, request order, GQA vs. replicated MHA, chunked vs. full
  prefill).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"bf16": 0, "fp16": 1}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` into ``libpa_oracle.so`` (gcc, strict IEEE)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # PA_ORACLE_LIB points the wrappers at another build of the same
            # source (the mutation tests use it to load deliberately broken
            # copies); by default the library is built next to this file.
            path = os.environ.get("PA_ORACLE_LIB") or build()
            lib = ctypes.CDLL(path)
            i32p = ctypes.POINTER(ctypes.c_int32)
            u16p = ctypes.c_void_p
            lib.oracle_prepare_inputs.restype = ctypes.c_int
            lib.oracle_prepare_inputs.argtypes = [
                i32p, i32p, i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, i32p, i32p, i32p, i32p, ctypes.c_int32,
                i32p, i32p]
            lib.oracle_gather_input_ids.restype = ctypes.c_int
            lib.oracle_gather_input_ids.argtypes = [
                i32p, i32p, ctypes.c_int32, i32p, ctypes.c_int32, ctypes.c_int32,
                ctypes.POINTER(ctypes.c_int64), i32p]
            lib.oracle_discard_request_mask.restype = ctypes.c_int
            lib.oracle_discard_request_mask.argtypes = [
                i32p, i32p, i32p, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint8)]
            lib.oracle_spec_logits_indices.restype = ctypes.c_int
            lib.oracle_spec_logits_indices.argtypes = [
                i32p, i32p, ctypes.c_int32, ctypes.c_int32, i32p, i32p]
            for fn in (lib.oracle_copy_blocks, lib.oracle_zero_blocks):
                fn.restype = ctypes.c_int
            lib.oracle_copy_blocks.argtypes = [u16p, u16p, ctypes.c_int64, ctypes.c_int32, i32p,
                                               i32p, ctypes.c_int32]
            lib.oracle_zero_blocks.argtypes = [u16p, u16p, ctypes.c_int64, ctypes.c_int32, i32p,
                                               ctypes.c_int32]
            lib.oracle_cache_write.restype = ctypes.c_int
            lib.oracle_cache_write.argtypes = [
                u16p, u16p, ctypes.c_int64, u16p, u16p, i32p, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [
                u16p, u16p, u16p, i32p, ctypes.c_int32, i32p, i32p, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_double, ctypes.c_int32,
                ctypes.POINTER(ctypes.c_double), i32p, ctypes.c_int32, ctypes.c_int32]
            lib.oracle_attention_ex.restype = ctypes.c_int
            lib.oracle_attention_ex.argtypes = [
                u16p, u16p, u16p, i32p, ctypes.c_int32, i32p, i32p, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_double, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_double, ctypes.c_double,
                ctypes.POINTER(ctypes.c_double), i32p, ctypes.c_int32, ctypes.c_int32]
            lib.oracle_cache_write_fp8.restype = ctypes.c_int
            lib.oracle_cache_write_fp8.argtypes = [
                u16p, u16p, ctypes.c_int64, u16p, u16p, i32p, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_float, ctypes.c_float]
            lib.oracle_e4m3_decode.restype = ctypes.c_int
            lib.oracle_e4m3_decode.argtypes = [u16p, ctypes.c_int64,
                                               ctypes.POINTER(ctypes.c_double)]
            lib.oracle_e4m3_encode.restype = ctypes.c_int
            lib.oracle_e4m3_encode.argtypes = [u16p, ctypes.c_int64, u16p]
            lib.oracle_num_cpus.restype = ctypes.c_int
            lib.oracle_num_cpus.argtypes = []
            _lib = lib
    return _lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _bits(a) -> np.ndarray:
    """16-bit element patterns of a bf16/fp16 torch tensor or a uint16 array."""
    if isinstance(a, np.ndarray):
        if a.dtype == np.float16:
            return np.ascontiguousarray(a).view(np.uint16)
        return np.ascontiguousarray(a.astype(np.uint16, copy=False))
    import torch  # local: torch only as a carrier of bf16 bit patterns
    t = a.detach().to("cpu").contiguous()
    return t.view(torch.int16).numpy().view(np.uint16)


def _bytes8(a) -> np.ndarray:
    """Byte patterns of an FP8 pool (torch uint8 / float8 tensor or NumPy)."""
    if isinstance(a, np.ndarray):
        return np.ascontiguousarray(a).view(np.uint8)
    import torch  # local: torch only as a carrier of the pool's bytes
    return a.detach().to("cpu").contiguous().view(torch.uint8).numpy()


def e4m3_decode(codes) -> np.ndarray:
    """Exact values (float64) of E4M3 byte codes."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_decode(c.ctypes.data, c.size,
                               out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def e4m3_encode(x) -> np.ndarray:
    """E4M3 byte codes of float32 values (nearest, ties to even, +-448
    saturation)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(f.shape, np.uint8)
    _load().oracle_e4m3_encode(f.ctypes.data, f.size, out.ctypes.data)
    return out


def num_cpus() -> int:
    return int(_load().oracle_num_cpus())


def prepare_inputs(num_scheduled_tokens, num_computed_tokens, block_table, block_size,
                   num_tokens, num_blocks, qsl_capacity=None, check=True):
    """Index tensors of one step.  Returns a dict of int32 arrays:
    req_indices, positions, slot_mapping [T]; query_start_loc [qsl_capacity];
    seq_lens, logits_indices [R]; and ``status`` (0 when the inputs are valid)."""
    lib = _load()
    nst, nct = _i32(num_scheduled_tokens), _i32(num_computed_tokens)
    bt = _i32(block_table)
    r = nst.shape[0]
    bt = bt.reshape(r, -1) if r else bt.reshape(0, max(1, bt.size))
    mb = bt.shape[1]
    cap = r + 1 if qsl_capacity is None else int(qsl_capacity)
    out = {k: np.full(max(num_tokens, 0), -7, np.int32)
           for k in ("req_indices", "positions", "slot_mapping")}
    out["query_start_loc"] = np.full(max(cap, 1), -7, np.int32)
    out["seq_lens"] = np.full(r, -7, np.int32)
    out["logits_indices"] = np.full(r, -7, np.int32)
    rc = lib.oracle_prepare_inputs(
        _p32(nst), _p32(nct), _p32(bt), r, mb, int(block_size), int(num_tokens),
        int(num_blocks), _p32(out["req_indices"]), _p32(out["positions"]),
        _p32(out["slot_mapping"]), _p32(out["query_start_loc"]), cap,
        _p32(out["seq_lens"]), _p32(out["logits_indices"]))
    out["status"] = int(rc)
    if check and rc != 0:
        raise OracleError(f"oracle_prepare_inputs rejected the inputs ({rc})")
    return out


def gather_input_ids(req_indices, positions, token_ids, check=True):
    """token_indices (int64) and input_ids (int32) of every flat token, gathered
    from the ``[max_num_reqs, max_model_len]`` token buffer ``token_ids``.
    Returns (token_indices, input_ids, status)."""
    lib = _load()
    req, pos = _i32(req_indices), _i32(positions)
    ids = _i32(token_ids)
    if ids.ndim != 2:
        raise OracleError("token_ids must be [max_num_reqs, max_model_len]")
    t = req.shape[0]
    tok_idx = np.full(t, -7, np.int64)
    input_ids = np.full(t, -7, np.int32)
    rc = lib.oracle_gather_input_ids(
        _p32(req), _p32(pos), t, _p32(ids), ids.shape[0], ids.shape[1],
        tok_idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _p32(input_ids))
    if check and rc != 0:
        raise OracleError(f"oracle_gather_input_ids rejected the inputs ({rc})")
    return tok_idx, input_ids, int(rc)


def discard_request_mask(num_computed_tokens, num_scheduled_tokens, request_num_tokens):
    """Boolean per request: True when computed + scheduled is still short of
    the request's total token count (its sampled token is thrown away)."""
    lib = _load()
    nct, nst, ntok = (_i32(num_computed_tokens), _i32(num_scheduled_tokens),
                      _i32(request_num_tokens))
    r = nst.shape[0]
    mask = np.full(r, 7, np.uint8)
    rc = lib.oracle_discard_request_mask(_p32(nct), _p32(nst), _p32(ntok), r,
                                         mask.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
    if rc != 0:
        raise OracleError(f"oracle_discard_request_mask rejected the inputs ({rc})")
    return mask.astype(bool)


def spec_logits_indices(query_start_loc, num_draft_tokens=None, num_logits=None, check=True):
    """Sampled rows.  Returns (logits_indices [num_logits], cu_num_logits [R+1],
    status).  ``num_draft_tokens`` None means no drafts (one row per request)."""
    lib = _load()
    qsl = _i32(query_start_loc)
    r = qsl.shape[0] - 1
    d = None if num_draft_tokens is None else _i32(num_draft_tokens)
    n = (r + (int(d.sum()) if d is not None else 0)) if num_logits is None else int(num_logits)
    rows = np.full(max(n, 0), -7, np.int32)
    cu = np.full(r + 1, -7, np.int32)
    rc = lib.oracle_spec_logits_indices(_p32(qsl), None if d is None else _p32(d), r, n,
                                        _p32(rows), _p32(cu))
    if check and rc != 0:
        raise OracleError(f"oracle_spec_logits_indices rejected the inputs ({rc})")
    return rows, cu, int(rc)


def _pool_bytes(pool) -> np.ndarray:
    """A private byte copy of a pool ([NB, ...], any element type; a torch
    tensor or a NumPy array), shaped [NB, block_bytes]."""
    if isinstance(pool, np.ndarray):
        a = np.ascontiguousarray(pool)
    else:
        import torch  # local: torch only as a carrier of the pool's bytes
        t = pool.detach().to("cpu").contiguous()
        a = t.view(torch.uint8).numpy() if t.element_size() == 1 else \
            t.view(torch.int16).numpy()
    nb = a.shape[0]
    return a.view(np.uint8).reshape(nb, -1).copy()


def copy_blocks(key_cache, value_cache, src_blocks, dst_blocks, check=True):
    """Copy-on-write block copy.  Returns (key bytes, value bytes, status): the
    pools as uint8 [NB, block_bytes] after block dst[i] became a copy of
    block src[i] in both pools."""
    lib = _load()
    kb, vb = _pool_bytes(key_cache), _pool_bytes(value_cache)
    src, dst = _i32(src_blocks), _i32(dst_blocks)
    if src.shape != dst.shape or kb.shape != vb.shape:
        raise OracleError("src/dst lengths or pool shapes differ")
    rc = lib.oracle_copy_blocks(kb.ctypes.data, vb.ctypes.data, kb.shape[1], kb.shape[0],
                                _p32(src), _p32(dst), src.shape[0])
    if check and rc != 0:
        raise OracleError(f"oracle_copy_blocks rejected the inputs ({rc})")
    return kb, vb, int(rc)


def zero_blocks(key_cache, value_cache, block_ids, check=True):
    """Zero whole blocks of both pools.  Returns (key bytes, value bytes,
    status) as uint8 [NB, block_bytes]."""
    lib = _load()
    kb, vb = _pool_bytes(key_cache), _pool_bytes(value_cache)
    ids = _i32(block_ids)
    rc = lib.oracle_zero_blocks(kb.ctypes.data, vb.ctypes.data, kb.shape[1], kb.shape[0],
                                _p32(ids), ids.shape[0])
    if check and rc != 0:
        raise OracleError(f"oracle_zero_blocks rejected the inputs ({rc})")
    return kb, vb, int(rc)


def cache_write(key, value, key_cache, value_cache, slot_mapping, num_kv_heads, head_dim,
                block_size, num_blocks, kv_token_stride=None, check=True):
    """Return (key_cache', value_cache', status) as uint16 arrays shaped like the
    input caches: the pools after each token's K/V was copied to its slot."""
    lib = _load()
    kb, vb = _bits(key), _bits(value)
    stride = num_kv_heads * head_dim if kv_token_stride is None else int(kv_token_stride)
    kcb = _bits(key_cache).copy()
    vcb = _bits(value_cache).copy()
    slots = _i32(slot_mapping)
    t = slots.shape[0]
    if kb.size < (t - 1) * stride + num_kv_heads * head_dim if t else False:
        raise OracleError("key buffer too small for the stride")
    rc = lib.oracle_cache_write(kb.ctypes.data, vb.ctypes.data, stride, kcb.ctypes.data,
                                vcb.ctypes.data, _p32(slots), t, int(num_kv_heads),
                                int(head_dim), int(block_size), int(num_blocks))
    if check and rc != 0:
        raise OracleError(f"oracle_cache_write rejected the inputs ({rc})")
    return kcb, vcb, int(rc)


def cache_write_fp8(key, value, key_cache, value_cache, slot_mapping, num_kv_heads, head_dim,
                    block_size, num_blocks, dtype, k_scale, v_scale, kv_token_stride=None,
                    check=True):
    """The write into FP8 pools: returns (key bytes, value bytes, status),
    uint8 arrays shaped like the input pools."""
    lib = _load()
    kb, vb = _bits(key), _bits(value)
    stride = num_kv_heads * head_dim if kv_token_stride is None else int(kv_token_stride)
    kcb = _bytes8(key_cache).copy()
    vcb = _bytes8(value_cache).copy()
    slots = _i32(slot_mapping)
    rc = lib.oracle_cache_write_fp8(kb.ctypes.data, vb.ctypes.data, stride, kcb.ctypes.data,
                                    vcb.ctypes.data, _p32(slots), slots.shape[0],
                                    int(num_kv_heads), int(head_dim), int(block_size),
                                    int(num_blocks), DTYPES[dtype], float(k_scale),
                                    float(v_scale))
    if check and rc != 0:
        raise OracleError(f"oracle_cache_write_fp8 rejected the inputs ({rc})")
    return kcb, vcb, int(rc)


def attention(q, key_cache, value_cache, block_table, query_start_loc, seq_lens,
              num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
              tokens=None, num_threads=0, kv_cache_dtype="auto", k_scale=1.0, v_scale=1.0):
    """fp64 attention output [T, Hq, D].  With ``tokens`` (ascending flat token
    indices) only those rows are computed; the others are NaN.  With
    ``kv_cache_dtype="fp8_e4m3"`` the pools hold E4M3 bytes and the cached
    values are element * k_scale / * v_scale."""
    lib = _load()
    qb = _bits(q)
    fp8 = kv_cache_dtype == "fp8_e4m3"
    if fp8:
        kcb, vcb = _bytes8(key_cache), _bytes8(value_cache)
        cdt = 2
    else:
        kcb, vcb = _bits(key_cache), _bits(value_cache)
        cdt = DTYPES[dtype]
    qsl, sl = _i32(query_start_loc), _i32(seq_lens)
    r = sl.shape[0]
    bt = _i32(block_table).reshape(r, -1) if r else _i32(block_table).reshape(0, 1)
    t = int(qsl[r]) if r else 0
    out = np.full((t, num_q_heads, head_dim), np.nan, np.float64)
    sel = None if tokens is None else _i32(np.sort(np.asarray(tokens)))
    rc = lib.oracle_attention_ex(
        qb.ctypes.data, kcb.ctypes.data, vcb.ctypes.data, _p32(bt), bt.shape[1], _p32(qsl),
        _p32(sl), r, t, int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size),
        int(num_blocks), float(scale), DTYPES[dtype], cdt, float(k_scale), float(v_scale),
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
        None if sel is None else _p32(sel), 0 if sel is None else sel.shape[0],
        int(num_threads))
    if rc != 0:
        raise OracleError(f"oracle_attention rejected the inputs ({rc})")
    return out


def step(w, vals, qsl_capacity=None, tokens=None, num_threads=0):
    """The whole step for a workload from ``workloads``: index build, cache
    write, attention.  Returns (indices dict, key_cache', value_cache', out)."""
    idx = prepare_inputs(w.num_scheduled_tokens, w.num_computed_tokens, w.block_table,
                         w.block_size, w.num_tokens, w.num_blocks, qsl_capacity)
    fp8 = getattr(w, "kv_cache_dtype", "auto") == "fp8_e4m3"
    if fp8:
        kc, vc, _ = cache_write_fp8(vals["key"], vals["value"], vals["key_cache"],
                                    vals["value_cache"], idx["slot_mapping"], w.num_kv_heads,
                                    w.head_dim, w.block_size, w.num_blocks, w.dtype,
                                    w.k_scale, w.v_scale)
    else:
        kc, vc, _ = cache_write(vals["key"], vals["value"], vals["key_cache"],
                                vals["value_cache"], idx["slot_mapping"], w.num_kv_heads,
                                w.head_dim, w.block_size, w.num_blocks)
    out = attention(vals["q"], kc, vc, w.block_table, idx["query_start_loc"][: w.num_reqs + 1],
                    idx["seq_lens"], w.num_q_heads, w.num_kv_heads, w.head_dim,
                    w.block_size, w.num_blocks, w.scale, w.dtype, tokens, num_threads,
                    kv_cache_dtype="fp8_e4m3" if fp8 else "auto",
                    k_scale=getattr(w, "k_scale", 1.0), v_scale=getattr(w, "v_scale", 1.0))
    return idx, kc, vc, out
