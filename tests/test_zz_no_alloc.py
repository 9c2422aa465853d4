"""pa_attention_noalloc: attention for callers that cannot allocate.

Callers such as an engine that has handed nearly all free HBM to its KV
pool, or a decode loop that cannot afford the device synchronisation of
cudaMalloc, use this entry point: it takes no workspace and uses the
library's own fixed device array instead.  Its output must match the
existing pa_attention entry point on the same inputs, call after call (the
array keeps the previous call's contents, which must not leak into the
next result).  This file is collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prepare_gb300 as pa
import workloads
from gpu_step import run_step, to_dev
from helpers import check_attention_close


def _existing_and_noalloc(w, seed):
    vals = workloads.make_values(w, seed, device="cuda")
    res = run_step(w, vals)                     # pa_attention with its default workspace
    assert res["status"] == pa.PA_OK
    q = vals["q"].contiguous()
    bt = to_dev(w.block_table)
    qsl = torch.from_numpy(res["query_start_loc"][: w.num_reqs + 1]).cuda()
    sl = torch.from_numpy(res["seq_lens"]).cuda()
    # the existing entry point given a caller workspace of the same size
    same = torch.full_like(q, float("nan"))
    ws = torch.empty(pa.NOALLOC_SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
    pa.pa_attention(q, res["key_cache"], res["value_cache"], bt, qsl, sl, w.max_query_len,
                    w.max_seq_len, w.scale, same, ws)
    got = torch.full_like(q, float("nan"))
    pa.pa_attention_noalloc(q, res["key_cache"], res["value_cache"], bt, qsl, sl,
                            w.max_query_len, w.max_seq_len, w.scale, got)
    assert pa.pa_get_status() == (pa.PA_OK, 0)
    _, _, _, ref = oracle.step(w, {k: v.cpu() for k, v in vals.items()})
    return same, got, ref


@pytest.mark.gpu
def test_noalloc_matches_existing_entry_point_twice_in_a_row():
    pa.pa_get_status()
    # First call: 256 long-context decodes (the scratch is smaller than the
    # default workspace, so partitions are longer); second call: a smaller,
    # different batch with a 300-token chunk for the tensor-core kernel,
    # which must not see the first call's leftovers.  Both kernels' results
    # depend only on the inputs and the workspace size, so the output must
    # equal, bit for bit, that of pa_attention given a workspace of the
    # array's size -- and lie within the bound of the oracle.
    cases = [workloads.decode_batch(1),
             workloads.random_case(5, max_reqs=6, max_computed=2500, long_prefill=300)]
    for i, w in enumerate(cases):
        same, got, ref = _existing_and_noalloc(w, 10 + i)
        assert torch.equal(got, same), i
        check_attention_close(got.double().cpu().numpy(), ref, got.dtype)


def test_noalloc_rejects_too_many_requests():
    # Rejected on the host before any device work: no GPU needed.
    fake = ctypes.c_void_p(0x100000)
    rc = pa.lib().pa_attention_noalloc(fake, fake, fake, fake, 4, fake, fake,
                                       pa.NOALLOC_MAX_REQS + 1, 10, 1, 16, 4, 2, 64, 16, 8,
                                       0.1, pa.PA_BF16, fake, None)
    assert rc == pa.PA_ERR_WORKSPACE
