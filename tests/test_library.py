"""The C-ABI library without a GPU: it builds, loads, exports every symbol
include/pa.h declares, and its host-side checks reject bad arguments before
any CUDA call."""

import ctypes
import os
import re

import pytest

import paged_kv_attention_prepare_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("pa_prepare_inputs", "pa_cache_write", "pa_attention",
              "pa_attention_workspace_size", "pa_get_status", "pa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(pa.build())
    for n in _declared():
        assert hasattr(lib, n), n


def test_status_strings():
    for s in range(7):
        assert pa.lib().pa_status_string(s)


FAKE = ctypes.c_void_p(0x100000)  # never dereferenced: the checks return first


def test_attention_rejects_unsupported_head_dim():
    L = pa.lib()
    rc = L.pa_attention(FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 2, 2, 1, 16, 4, 2, 96, 16, 8,
                        0.1, pa.PA_BF16, FAKE, None, 0, None)
    assert rc == pa.PA_ERR_UNSUPPORTED


@pytest.mark.parametrize("case", ["block_size", "ratio", "null", "ws_align", "neg"])
def test_attention_rejects_bad_arguments(case):
    L = pa.lib()
    args = dict(bs=16, hq=4, hkv=2, q=FAKE, ws=None, wsb=0, R=2)
    if case == "block_size":
        args["bs"] = 32
    elif case == "ratio":
        args["hq"] = 5
    elif case == "null":
        args["q"] = None
    elif case == "ws_align":
        args["ws"], args["wsb"] = ctypes.c_void_p(0x100004), 64
    elif case == "neg":
        args["R"] = -1
    rc = L.pa_attention(args["q"], FAKE, FAKE, FAKE, 4, FAKE, FAKE, args["R"], 2, 1, 16,
                        args["hq"], args["hkv"], 64, args["bs"], 8, 0.1, pa.PA_BF16, FAKE,
                        args["ws"], args["wsb"], None)
    expect = pa.PA_ERR_UNSUPPORTED if case in ("block_size", "ratio") else pa.PA_ERR_INVALID
    assert rc == expect


@pytest.mark.parametrize("flags", [2, 0x80000000, 3])
def test_attention_ex_rejects_unknown_flags(flags):
    # PA_ATTN_SHARED_BLOCKS is the only flag; any other bit is refused before
    # anything is launched
    L = pa.lib()
    rc = L.pa_attention_ex(FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 2, 2, 1, 16, 4, 2, 64, 16, 8,
                           0.1, pa.PA_BF16, pa.PA_BF16, None, None, flags, FAKE, None, 0, None)
    assert rc == pa.PA_ERR_INVALID


def test_prepare_rejects_small_qsl_capacity_and_huge_pool():
    L = pa.lib()
    assert L.pa_prepare_inputs(FAKE, FAKE, FAKE, 3, 2, 16, 5, 8, FAKE, FAKE, FAKE, FAKE, 3,
                               FAKE, FAKE, None) == pa.PA_ERR_INVALID
    assert L.pa_prepare_inputs(FAKE, FAKE, FAKE, 3, 2, 16, 5, 1 << 28, FAKE, FAKE, FAKE, FAKE,
                               4, FAKE, FAKE, None) == pa.PA_ERR_INVALID


@pytest.mark.parametrize("case", ["gather_without_ids", "ids_without_width", "negative_width",
                                  "rows_below_reqs", "mask_without_counts",
                                  "counts_without_mask", "logits_count_without_drafts",
                                  "negative_logits", "qsl_capacity"])
def test_prepare_ex_rejects_half_given_groups(case):
    L = pa.lib()
    a = dict(tok=None, rows=0, width=0, ntok=None, drafts=None, nlog=3, ti=None, ids=None,
             mask=None, cap=4)
    if case == "gather_without_ids":
        a.update(tok=FAKE, rows=3, width=8, ti=FAKE)             # input_ids missing
    elif case == "ids_without_width":
        a.update(tok=FAKE, rows=3, ti=FAKE, ids=FAKE)            # max_model_len == 0
    elif case == "negative_width":
        a.update(width=-1)
    elif case == "rows_below_reqs":
        a.update(tok=FAKE, rows=2, width=8, ti=FAKE, ids=FAKE)
    elif case == "mask_without_counts":
        a.update(mask=FAKE)
    elif case == "counts_without_mask":
        a.update(ntok=FAKE)
    elif case == "logits_count_without_drafts":
        a.update(nlog=5)
    elif case == "negative_logits":
        a.update(drafts=FAKE, nlog=-1)
    else:
        a.update(cap=3)
    rc = L.pa_prepare_inputs_ex(FAKE, FAKE, FAKE, 3, 2, 16, 5, 8, a["tok"], a["rows"],
                                a["width"], a["ntok"], a["drafts"], a["nlog"], FAKE, FAKE, FAKE,
                                FAKE, a["cap"], FAKE, a["ti"], a["ids"], a["mask"], FAKE, None,
                                None)
    assert rc == pa.PA_ERR_INVALID


@pytest.mark.parametrize("fn", ["copy", "zero"])
def test_block_ops_reject_bad_arguments(fn):
    L = pa.lib()
    unaligned = ctypes.c_void_p(0x100008)

    def call(kc=FAKE, n=3, bs=16, hkv=8, d=128, dtype=pa.PA_BF16, ids=FAKE):
        if fn == "copy":
            return L.pa_copy_blocks(kc, FAKE, ids, FAKE, n, bs, hkv, d, 64, dtype, None)
        return L.pa_zero_blocks(kc, FAKE, ids, n, bs, hkv, d, 64, dtype, None)

    assert call(n=-1) == pa.PA_ERR_INVALID
    assert call(ids=None) == pa.PA_ERR_INVALID
    assert call(kc=unaligned) == pa.PA_ERR_INVALID
    assert call(dtype=9) == pa.PA_ERR_INVALID
    assert call(bs=1, hkv=1, d=3) == pa.PA_ERR_UNSUPPORTED   # 16-byte blocks only
    assert call(n=0, ids=None) == pa.PA_OK                   # nothing to do, nothing launched


def test_cache_write_rejects_short_stride_and_bad_dtype():
    L = pa.lib()
    assert L.pa_cache_write(FAKE, FAKE, 100, FAKE, FAKE, FAKE, 4, 2, 64, 16, 8, pa.PA_BF16,
                            None) == pa.PA_ERR_INVALID
    assert L.pa_cache_write(FAKE, FAKE, 128, FAKE, FAKE, FAKE, 4, 2, 64, 16, 8, 7,
                            None) == pa.PA_ERR_INVALID


def test_workspace_size_grows_with_context():
    small = pa.pa_attention_workspace_size(256, 256, 1, 512, 32, 8, 128)
    big = pa.pa_attention_workspace_size(256, 256, 1, 4096, 32, 8, 128)
    assert 0 < small < big


def test_binding_refuses_host_tensors():
    import torch
    t = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(TypeError):
        pa.pa_prepare_inputs(t, t, t.view(4, 1), 16, 4, 4, t, t, t, t, t, t)


@pytest.mark.parametrize("case", ["short_stride", "bad_dtype", "bad_cache_dtype", "null_key",
                                  "small_qsl"])
def test_prepare_and_write_rejects_bad_arguments(case):
    # host checks of the fused index build + cache write, before any launch
    L = pa.lib()
    a = dict(stride=128, dtype=pa.PA_BF16, cdt=pa.PA_BF16, key=FAKE, cap=4)
    if case == "short_stride":
        a["stride"] = 100
    elif case == "bad_dtype":
        a["dtype"] = 7
    elif case == "bad_cache_dtype":
        a["cdt"] = pa.PA_FP16
    elif case == "null_key":
        a["key"] = None
    else:
        a["cap"] = 2
    rc = L.pa_prepare_and_write(FAKE, FAKE, FAKE, 3, 2, 16, 5, 8, FAKE, FAKE, FAKE, FAKE,
                                a["cap"], FAKE, FAKE, a["key"], FAKE, a["stride"], FAKE, FAKE, 2,
                                64, a["dtype"], a["cdt"], None, None, None)
    assert rc == pa.PA_ERR_INVALID
