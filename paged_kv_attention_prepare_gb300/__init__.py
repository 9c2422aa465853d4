"""Paged-KV attention step for GB300: Python binding of ``libpa.so``.

Argument marshalling only: every function takes torch CUDA tensors, checks
their dtype, device and layout, and passes raw pointers, sizes and the
stream to the C ABI in ``include/pa.h``.  Every step runs in the library's
CUDA kernels; there is no CPU or PyTorch fallback, and using the package
without the built library raises immediately.

Functions carry the C names: ``pa_prepare_inputs``, ``pa_prepare_inputs_ex``,
``pa_cache_write`` (over ``pa_cache_write_ex``), ``pa_prepare_and_write``, ``pa_copy_blocks``, ``pa_zero_blocks``,
``pa_attention_workspace_size``, ``pa_attention`` (over ``pa_attention_ex``),
``pa_attention_noalloc``,
``pa_get_status``, ``pa_launch_count``.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_OK, PA_ERR_INVALID, PA_ERR_CUDA, PA_ERR_UNSUPPORTED = 0, 1, 2, 3
PA_ERR_DEVICE_CHECK, PA_ERR_TIMEOUT, PA_ERR_WORKSPACE = 4, 5, 6
PA_BF16, PA_FP16, PA_FP8_E4M3 = 0, 1, 2
PA_ATTN_SHARED_BLOCKS = 1

CHECK_BITS = {
    "empty_request": 1 << 0, "token_count": 1 << 1, "block_id": 1 << 2,
    "logical_block": 1 << 3, "slot": 1 << 4, "seq_len": 1 << 5, "timeout": 1 << 6,
    "token_index": 1 << 7, "draft_count": 1 << 8,
}

_DTYPES = {torch.bfloat16: PA_BF16, torch.float16: PA_FP16}
# FP8 (E4M3) pools may be held as uint8 or float8_e4m3fn tensors
_FP8_POOL = {torch.uint8, torch.float8_e4m3fn}
_lock = threading.Lock()
_lib = None


class PAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_string(status)} ({status})")


def build(force: bool = False) -> str:
    """Compile ``libpa.so`` (nvcc, sm_103a) next to this file."""
    from .builder import build as _build
    return _build(force=force)


def lib():
    """The loaded ``libpa.so``; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -m paged_kv_attention_prepare_gb300.builder)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            L.pa_prepare_inputs.restype = ctypes.c_int
            L.pa_prepare_inputs.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                            i32, vp, vp, vp]
            L.pa_prepare_inputs_ex.restype = ctypes.c_int
            L.pa_prepare_inputs_ex.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, i32, i32,
                                               vp, vp, i32, vp, vp, vp, vp, i32, vp, vp, vp, vp,
                                               vp, vp, vp]
            L.pa_prepare_and_write.restype = ctypes.c_int
            L.pa_prepare_and_write.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp,
                                               vp, i32, vp, vp, vp, vp, i64, vp, vp, i32, i32,
                                               ctypes.c_int, ctypes.c_int, vp, vp, vp]
            for fn in (L.pa_copy_blocks, L.pa_zero_blocks):
                fn.restype = ctypes.c_int
            L.pa_copy_blocks.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_int, vp]
            L.pa_zero_blocks.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_int, vp]
            L.pa_cache_write.restype = ctypes.c_int
            L.pa_cache_write.argtypes = [vp, vp, i64, vp, vp, vp, i32, i32, i32, i32, i32,
                                         ctypes.c_int, vp]
            L.pa_attention_workspace_size.restype = sz
            L.pa_attention_workspace_size.argtypes = [i32] * 7
            L.pa_attention.restype = ctypes.c_int
            L.pa_attention.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                       i32, i32, i32, ctypes.c_float, ctypes.c_int, vp, vp, sz, vp]
            L.pa_cache_write_ex.restype = ctypes.c_int
            L.pa_cache_write_ex.argtypes = [vp, vp, i64, vp, vp, vp, i32, i32, i32, i32, i32,
                                            ctypes.c_int, ctypes.c_int, vp, vp, vp]
            L.pa_attention_ex.restype = ctypes.c_int
            L.pa_attention_ex.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                          i32, i32, i32, i32, ctypes.c_float, ctypes.c_int,
                                          ctypes.c_int, vp, vp, ctypes.c_uint32, vp, vp, sz, vp]
            L.pa_attention_noalloc.restype = ctypes.c_int
            L.pa_attention_noalloc.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                               i32, i32, i32, i32, i32, ctypes.c_float,
                                               ctypes.c_int, vp, vp]
            L.pa_selftest_wait_timeout.restype = ctypes.c_int
            L.pa_selftest_wait_timeout.argtypes = [vp]
            L.pa_get_status.restype = ctypes.c_int
            L.pa_get_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
            L.pa_status_string.restype = ctypes.c_char_p
            L.pa_status_string.argtypes = [ctypes.c_int]
            L.pa_launch_count.restype = ctypes.c_uint64
            L.pa_launch_count.argtypes = []
            _lib = L
    return _lib


def _status_string(s: int) -> str:
    try:
        return lib().pa_status_string(int(s)).decode()
    except Exception:  # pragma: no cover - only while reporting another error
        return "status"


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, name: str, dtype=None, contiguous=True):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _check(rc: int, what: str):
    if rc != PA_OK:
        raise PAError(rc, what)


def pa_prepare_inputs(num_scheduled_tokens, num_computed_tokens, block_table, block_size,
                      num_tokens, num_blocks, req_indices, positions, slot_mapping,
                      query_start_loc, seq_lens, logits_indices, stream=None):
    """Index tensors of one step into caller-allocated int32 CUDA tensors."""
    i32 = torch.int32
    R = num_scheduled_tokens.shape[0]
    rc = lib().pa_prepare_inputs(
        _dev(num_scheduled_tokens, "num_scheduled_tokens", i32),
        _dev(num_computed_tokens, "num_computed_tokens", i32),
        _dev(block_table, "block_table", i32), R, block_table.shape[1] if R else 0,
        int(block_size), int(num_tokens), int(num_blocks),
        _dev(req_indices, "req_indices", i32), _dev(positions, "positions", i32),
        _dev(slot_mapping, "slot_mapping", i32), _dev(query_start_loc, "query_start_loc", i32),
        query_start_loc.shape[0], _dev(seq_lens, "seq_lens", i32),
        _dev(logits_indices, "logits_indices", i32), _stream(stream))
    _check(rc, "pa_prepare_inputs")


def _opt(t, name, dtype):
    return None if t is None else _dev(t, name, dtype)


def pa_prepare_inputs_ex(num_scheduled_tokens, num_computed_tokens, block_table, block_size,
                         num_tokens, num_blocks, req_indices, positions, slot_mapping,
                         query_start_loc, seq_lens, logits_indices, token_ids=None,
                         token_indices=None, input_ids=None, request_num_tokens=None,
                         discard_request_mask=None, num_draft_tokens=None, cu_num_logits=None,
                         stream=None):
    """``pa_prepare_inputs`` plus the token-id gather (``token_ids`` is the
    [max_num_reqs, max_model_len] int32 buffer, a CUDA tensor or a pinned CPU
    tensor; ``token_indices`` int64 and ``input_ids`` int32 [T] receive the
    result), the discard mask (``request_num_tokens`` int32 [R] in,
    ``discard_request_mask`` bool/uint8 [R] out) and the sampled rows of
    speculative decoding (``num_draft_tokens`` int32 [R]; ``logits_indices``
    then holds R + sum(drafts) rows, ``cu_num_logits`` [R+1] their starts)."""
    i32 = torch.int32
    R = num_scheduled_tokens.shape[0]
    if token_ids is not None:
        if token_ids.dtype != i32 or token_ids.dim() != 2 or not token_ids.is_contiguous():
            raise TypeError("token_ids must be a contiguous int32 [max_num_reqs, max_model_len]")
        if not (token_ids.is_cuda or token_ids.is_pinned()):
            raise TypeError("token_ids must be a CUDA tensor or a pinned CPU tensor")
        tok_ptr = ctypes.c_void_p(token_ids.data_ptr())
        rows, width = token_ids.shape
    else:
        tok_ptr, rows, width = None, 0, 0
    mask_ptr = None
    if discard_request_mask is not None:
        if discard_request_mask.dtype not in (torch.bool, torch.uint8):
            raise TypeError("discard_request_mask must be bool or uint8")
        mask_ptr = _dev(discard_request_mask, "discard_request_mask")
    rc = lib().pa_prepare_inputs_ex(
        _dev(num_scheduled_tokens, "num_scheduled_tokens", i32),
        _dev(num_computed_tokens, "num_computed_tokens", i32),
        _dev(block_table, "block_table", i32), R, block_table.shape[1] if R else 0,
        int(block_size), int(num_tokens), int(num_blocks), tok_ptr, rows, width,
        _opt(request_num_tokens, "request_num_tokens", i32),
        _opt(num_draft_tokens, "num_draft_tokens", i32), logits_indices.shape[0],
        _dev(req_indices, "req_indices", i32), _dev(positions, "positions", i32),
        _dev(slot_mapping, "slot_mapping", i32), _dev(query_start_loc, "query_start_loc", i32),
        query_start_loc.shape[0], _dev(seq_lens, "seq_lens", i32),
        _opt(token_indices, "token_indices", torch.int64), _opt(input_ids, "input_ids", i32),
        mask_ptr, _dev(logits_indices, "logits_indices", i32),
        _opt(cu_num_logits, "cu_num_logits", i32), _stream(stream))
    _check(rc, "pa_prepare_inputs_ex")


def _scale_ptr(t, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 \
            or t.numel() != 1:
        raise TypeError(f"{name} must be a one-element float32 CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _cache_dtype(q_dtype, key_cache, value_cache):
    """The pools' pa_dtype: the q dtype, or PA_FP8_E4M3 for byte pools."""
    if key_cache.dtype in _FP8_POOL and value_cache.dtype in _FP8_POOL:
        return PA_FP8_E4M3
    if key_cache.dtype != q_dtype or value_cache.dtype != q_dtype:
        raise TypeError("caches must have the q/key dtype, or be FP8 (uint8/float8_e4m3fn)")
    return _DTYPES[q_dtype]


def pa_cache_write(key, value, key_cache, value_cache, slot_mapping, num_blocks=None,
                   stream=None, k_scale=None, v_scale=None):
    """Scatter key/value [T, Hkv, D] (token stride may exceed Hkv*D) into the
    [NB, bs, Hkv, D] pools at slot_mapping.  FP8 pools (uint8 or
    float8_e4m3fn) take E4M3(x / scale) with ``k_scale``/``v_scale`` one-element
    float32 CUDA tensors (None = 1.0)."""
    T, hkv, d = key.shape
    if key.stride(1) != d or key.stride(2) != 1 or value.stride() != key.stride():
        raise ValueError("key/value rows must be [Hkv, D]-contiguous with equal strides")
    dt = _DTYPES.get(key.dtype)
    if dt is None or value.dtype != key.dtype:
        raise TypeError("key and value must share a bf16/fp16 dtype")
    cdt = _cache_dtype(key.dtype, key_cache, value_cache)
    nb, bs = key_cache.shape[0], key_cache.shape[1]
    rc = lib().pa_cache_write_ex(
        _dev(key, "key", contiguous=False), _dev(value, "value", contiguous=False),
        int(key.stride(0)) if T else hkv * d, _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(slot_mapping, "slot_mapping", torch.int32), T,
        hkv, d, bs, nb if num_blocks is None else int(num_blocks), dt, cdt,
        _scale_ptr(k_scale, "k_scale"), _scale_ptr(v_scale, "v_scale"), _stream(stream))
    _check(rc, "pa_cache_write")


def pa_prepare_and_write(num_scheduled_tokens, num_computed_tokens, block_table, block_size,
                         num_tokens, num_blocks, req_indices, positions, slot_mapping,
                         query_start_loc, seq_lens, logits_indices, key, value, key_cache,
                         value_cache, k_scale=None, v_scale=None, stream=None):
    """``pa_prepare_inputs`` and ``pa_cache_write`` (same arguments) in one
    launch: the index tensors, then each token's key/value row written to the
    pools at its slot."""
    i32 = torch.int32
    R = num_scheduled_tokens.shape[0]
    T, hkv, d = key.shape
    if key.stride(1) != d or key.stride(2) != 1 or value.stride() != key.stride():
        raise ValueError("key/value rows must be [Hkv, D]-contiguous with equal strides")
    dt = _DTYPES.get(key.dtype)
    if dt is None or value.dtype != key.dtype:
        raise TypeError("key and value must share a bf16/fp16 dtype")
    cdt = _cache_dtype(key.dtype, key_cache, value_cache)
    rc = lib().pa_prepare_and_write(
        _dev(num_scheduled_tokens, "num_scheduled_tokens", i32),
        _dev(num_computed_tokens, "num_computed_tokens", i32),
        _dev(block_table, "block_table", i32), R, block_table.shape[1] if R else 0,
        int(block_size), int(num_tokens), int(num_blocks),
        _dev(req_indices, "req_indices", i32), _dev(positions, "positions", i32),
        _dev(slot_mapping, "slot_mapping", i32), _dev(query_start_loc, "query_start_loc", i32),
        query_start_loc.shape[0], _dev(seq_lens, "seq_lens", i32),
        _dev(logits_indices, "logits_indices", i32),
        _dev(key, "key", contiguous=False), _dev(value, "value", contiguous=False),
        int(key.stride(0)) if T else hkv * d, _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), hkv, d, dt, cdt,
        _scale_ptr(k_scale, "k_scale"), _scale_ptr(v_scale, "v_scale"), _stream(stream))
    _check(rc, "pa_prepare_and_write")


def _pools(key_cache, value_cache):
    if key_cache.shape != value_cache.shape or key_cache.dim() != 4:
        raise ValueError("key/value caches must both be [NB, bs, Hkv, D]")
    if key_cache.dtype in _FP8_POOL and value_cache.dtype in _FP8_POOL:
        dt = PA_FP8_E4M3
    else:
        dt = _DTYPES.get(key_cache.dtype)
        if dt is None or value_cache.dtype != key_cache.dtype:
            raise TypeError("caches must share a bf16/fp16/FP8 dtype")
    nb, bs, hkv, d = key_cache.shape
    return nb, bs, hkv, d, dt


def pa_copy_blocks(key_cache, value_cache, src_blocks, dst_blocks, stream=None):
    """Copy-on-write: block dst_blocks[i] of both pools becomes a copy of
    block src_blocks[i] (int32 CUDA tensors of equal length)."""
    nb, bs, hkv, d, dt = _pools(key_cache, value_cache)
    if src_blocks.shape != dst_blocks.shape or src_blocks.dim() != 1:
        raise ValueError("src_blocks and dst_blocks must be 1-D of equal length")
    rc = lib().pa_copy_blocks(_dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
                              _dev(src_blocks, "src_blocks", torch.int32),
                              _dev(dst_blocks, "dst_blocks", torch.int32), src_blocks.shape[0],
                              bs, hkv, d, nb, dt, _stream(stream))
    _check(rc, "pa_copy_blocks")


def pa_zero_blocks(key_cache, value_cache, block_ids, stream=None):
    """Zero every byte of the listed blocks in both pools."""
    nb, bs, hkv, d, dt = _pools(key_cache, value_cache)
    rc = lib().pa_zero_blocks(_dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
                              _dev(block_ids, "block_ids", torch.int32), block_ids.shape[0], bs,
                              hkv, d, nb, dt, _stream(stream))
    _check(rc, "pa_zero_blocks")


def pa_attention_workspace_size(num_reqs, num_tokens, max_query_len, max_seq_len, num_q_heads,
                                num_kv_heads, head_dim) -> int:
    return int(lib().pa_attention_workspace_size(num_reqs, num_tokens, max_query_len,
                                                 max_seq_len, num_q_heads, num_kv_heads,
                                                 head_dim))


def pa_attention(q, key_cache, value_cache, block_table, query_start_loc, seq_lens,
                 max_query_len, max_seq_len, scale, out, workspace=None, stream=None,
                 k_scale=None, v_scale=None, shared_blocks=False):
    """Paged causal GQA attention: q [T, Hq, D] -> out [T, Hq, D].  FP8 pools
    (uint8 / float8_e4m3fn) read element * k_scale / * v_scale.
    ``shared_blocks``: block tables may share physical blocks across requests
    (PA_ATTN_SHARED_BLOCKS); requests sharing whole partitions are computed
    together."""
    T, hq, d = q.shape
    nb, bs, hkv, _ = key_cache.shape
    R = seq_lens.shape[0]
    dt = _DTYPES.get(q.dtype)
    if dt is None or out.dtype != q.dtype:
        raise TypeError("q and out must share a bf16/fp16 dtype")
    cdt = _cache_dtype(q.dtype, key_cache, value_cache)
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None and workspace.numel() > 0:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().pa_attention_ex(
        _dev(q, "q"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(block_table, "block_table", torch.int32), block_table.shape[1],
        _dev(query_start_loc, "query_start_loc", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), R, T, int(max_query_len), int(max_seq_len),
        hq, hkv, d, bs, nb, float(scale), dt, cdt, _scale_ptr(k_scale, "k_scale"),
        _scale_ptr(v_scale, "v_scale"), PA_ATTN_SHARED_BLOCKS if shared_blocks else 0,
        _dev(out, "out"), ws_ptr, ws_bytes, _stream(stream))
    _check(rc, "pa_attention")


def pa_attention_noalloc(q, key_cache, value_cache, block_table, query_start_loc, seq_lens,
                         max_query_len, max_seq_len, scale, out, stream=None):
    """pa_attention without a caller workspace: for callers that cannot
    allocate device memory at call time.  The library's own fixed device
    array (PA_NOALLOC_SCRATCH_BYTES per GPU) serves as scratch; calls on one
    device must not overlap on the GPU.  Make the first call on a device
    before any stream capture (it looks up the array's address)."""
    T, hq, d = q.shape
    nb, bs, hkv, _ = key_cache.shape
    R = seq_lens.shape[0]
    dt = _DTYPES.get(q.dtype)
    if dt is None or key_cache.dtype != q.dtype or out.dtype != q.dtype:
        raise TypeError("q, caches and out must share a bf16/fp16 dtype")
    rc = lib().pa_attention_noalloc(
        _dev(q, "q"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(block_table, "block_table", torch.int32), block_table.shape[1],
        _dev(query_start_loc, "query_start_loc", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), R, T, int(max_query_len), int(max_seq_len),
        hq, hkv, d, bs, nb, float(scale), dt, _dev(out, "out"), _stream(stream))
    _check(rc, "pa_attention_noalloc")


NOALLOC_SCRATCH_BYTES = 32 << 20
NOALLOC_MAX_REQS = 65536


def pa_get_status(stream=None):
    """(status, detail bits): synchronises the stream, reads and clears the
    device status word."""
    detail = ctypes.c_uint32(0)
    rc = lib().pa_get_status(_stream(stream), ctypes.byref(detail))
    return int(rc), int(detail.value)


def pa_selftest_wait_timeout(stream=None):
    """Diagnostic: run a kernel whose bounded wait cannot succeed (see pa.h)."""
    _check(lib().pa_selftest_wait_timeout(_stream(stream)), "pa_selftest_wait_timeout")


def pa_launch_count() -> int:
    return int(lib().pa_launch_count())


def check_bits(detail: int) -> set:
    return {k for k, b in CHECK_BITS.items() if detail & b}
