"""bf16 pools: the prefill kernel's V comes from a copy widened to f16 once
per call in the workspace's tail (requests in order while it has room), or
is converted inside the kernel.  The two routes round the same bf16 values to
the same f16 values, so every prefill row must come out bit for bit the same
whatever the workspace holds, and within the bound of the oracle."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prepare_gb300 as pa
import workloads
from gpu_step import run_step
from helpers import check_attention_close

pytestmark = pytest.mark.gpu

# Bytes of the widened copy per 16-token page at 8 kv heads, head_dim 128:
# the f16 rows of every head plus one flag byte per head.
PAGE = 8 * (16 * 128 * 2 + 1)


def _prefill_tokens(w):
    qsl = np.concatenate([[0], np.cumsum(w.num_scheduled_tokens)])
    rows = [np.arange(qsl[r], qsl[r + 1]) for r in range(w.num_reqs)
            if w.num_scheduled_tokens[r] > 16]
    return np.concatenate(rows)


@pytest.mark.parametrize("beyond", [False, True])
def test_widened_v_gives_the_same_bits(beyond):
    rng = np.random.default_rng(31)
    # three prefill requests (400, 1200 and 700 keys) between decodes
    w = workloads._make("widen", [300, 1, 200, 1, 700, 1], [100, 500, 1000, 50, 0, 900], rng,
                        32, 8, 128, "bf16")
    vals = workloads.make_values(w, 3)
    if beyond:
        # a page of the second prefill request with values f16 cannot hold:
        # its tiles come from the pool and keep those halves bf16
        vc = vals["value_cache"]
        for pos in (130, 700):
            blk, off = int(w.block_table[2][pos // 16]), pos % 16
            vc[blk, off, :, 5] = 70000.0
            vc[blk, off, :, 9] = -1e30
    full = pa.pa_attention_workspace_size(w.num_reqs, w.num_tokens, w.max_query_len,
                                          w.max_seq_len, 32, 8, 128)
    ref = run_step(w, vals, workspace_bytes=full)
    assert ref["status"] == pa.PA_OK, pa.check_bits(ref["detail"])
    host = {k: v.cpu() for k, v in vals.items()}
    _, _, _, want = oracle.step(w, host)
    got = ref["out"].float().cpu().numpy().astype(np.float64)
    check_attention_close(got, want, ref["out"].dtype)
    rows = torch.from_numpy(_prefill_tokens(w)).cuda()
    base = ref["out"].index_select(0, rows)
    # Room for all of the copy, for the first request only, for none of it;
    # and a workspace without the decode partials' full share either.
    for cut in (PAGE * 300, PAGE * 400, PAGE * 440, PAGE * 460, full // 2, 0):
        ws = max(full - cut, 0) if cut else 0
        res = run_step(w, vals, workspace_bytes=ws)
        assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
        assert torch.equal(res["out"].index_select(0, rows), base), f"workspace {ws}"
        got = res["out"].float().cpu().numpy().astype(np.float64)
        check_attention_close(got, want, res["out"].dtype)
