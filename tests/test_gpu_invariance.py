"""Invariances of the CUDA path (the same properties the oracle is pinned
to, here on the GPU and to the bit):

- relabelling the pool's physical blocks (contents moved with their ids)
  changes nothing;
- laying every request's context out in consecutive blocks (paged equal to
  contiguous) changes nothing;
- shuffling the order of the requests in the batch only permutes the
  output rows.

Each work item's arithmetic depends only on the values it reads, not on
block ids or on where its request sits in the batch."""

import numpy as np
import pytest
import torch

import paged_kv_attention_prepare_gb300 as pa
import workloads
from gpu_step import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clean_status():
    pa.pa_get_status()
    yield


def _case():
    # decodes with long contexts (split-K and the merge pass), a short chunk
    # (split-K) and a long prompt chunk (the tensor-core kernel)
    rng = np.random.default_rng(12)
    nst = [1, 1, 5, 1, 200, 1, 9, 1]
    nct = [3000, 700, 1200, 40, 900, 2500, 300, 1600]
    w = workloads._make("invariance", nst, nct, rng, 8, 2, 128, "bf16")
    vals = workloads.make_values(w, 21, device="cuda")
    return w, vals


def _attend(w, q, kc, vc, bt):
    qsl = to_dev(np.concatenate([[0], np.cumsum(w.num_scheduled_tokens)]).astype(np.int32))
    sl = to_dev(w.context_lens.astype(np.int32))
    nb = pa.pa_attention_workspace_size(w.num_reqs, w.num_tokens, w.max_query_len,
                                        w.max_seq_len, w.num_q_heads, w.num_kv_heads, w.head_dim)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    out = torch.full_like(q, float("nan"))
    pa.pa_attention(q, kc, vc, to_dev(bt), qsl, sl, w.max_query_len, w.max_seq_len, w.scale,
                    out, ws)
    assert pa.pa_get_status() == (pa.PA_OK, 0)
    return out


def _relabel(w, vals, new_id):
    """Pool and table with block b stored at new_id[b]."""
    kc = torch.empty_like(vals["key_cache"])
    vc = torch.empty_like(vals["value_cache"])
    idx = to_dev(new_id.astype(np.int64))
    kc[idx] = vals["key_cache"]
    vc[idx] = vals["value_cache"]
    bt = w.block_table.copy()
    bt[bt >= 0] = new_id[bt[bt >= 0]]
    return kc, vc, bt


def _same(a, b):
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_physical_block_relabelling():
    w, vals = _case()
    base = _attend(w, vals["q"], vals["key_cache"], vals["value_cache"], w.block_table)
    new_id = np.random.default_rng(5).permutation(w.num_blocks)
    kc, vc, bt = _relabel(w, vals, new_id)
    _same(_attend(w, vals["q"], kc, vc, bt), base)


def test_paged_equals_contiguous():
    w, vals = _case()
    base = _attend(w, vals["q"], vals["key_cache"], vals["value_cache"], w.block_table)
    # every request's blocks in order, request after request, then the rest
    used = [int(b) for row in w.block_table for b in row if b >= 0]
    rest = [b for b in range(w.num_blocks) if b not in set(used)]
    new_id = np.empty(w.num_blocks, np.int64)
    new_id[np.array(used + rest)] = np.arange(w.num_blocks)
    kc, vc, bt = _relabel(w, vals, new_id)
    for r, row in enumerate(bt):   # each context is one run of consecutive blocks
        ids = row[row >= 0]
        assert (np.diff(ids) == 1).all()
    _same(_attend(w, vals["q"], kc, vc, bt), base)


def test_request_order_shuffle():
    w, vals = _case()
    base = _attend(w, vals["q"], vals["key_cache"], vals["value_cache"], w.block_table)
    order = np.random.default_rng(9).permutation(w.num_reqs)
    starts = np.concatenate([[0], np.cumsum(w.num_scheduled_tokens)])
    tok = np.concatenate([np.arange(starts[r], starts[r + 1]) for r in order])
    w2 = workloads.Workload("shuffled", w.num_scheduled_tokens[order],
                            w.num_computed_tokens[order], w.block_table[order], w.num_blocks,
                            w.block_size, w.num_q_heads, w.num_kv_heads, w.head_dim, w.dtype,
                            w.unique_blocks)
    q2 = vals["q"][to_dev(tok.astype(np.int64))].contiguous()
    out2 = _attend(w2, q2, vals["key_cache"], vals["value_cache"], w2.block_table)
    _same(out2, base[to_dev(tok.astype(np.int64))])
