"""The step's three calls captured once into a CUDA graph and replayed.

A replay must give exactly what the same calls give when launched one by
one on the same inputs (the same kernels, launch shapes and arguments), and
new input values copied into the captured buffers between replays must show
up in the next replay's results."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prepare_gb300 as pa
import workloads
from gpu_step import to_dev

pytestmark = pytest.mark.gpu


class Step:
    """Static buffers for one workload shape and the calls of one step."""

    def __init__(self, w, seed):
        self.w = w
        R, T = w.num_reqs, w.num_tokens
        i32 = torch.int32
        self.nst, self.nct, self.bt = (to_dev(w.num_scheduled_tokens),
                                       to_dev(w.num_computed_tokens), to_dev(w.block_table))
        self.ids = to_dev(workloads.make_token_buffer(w, seed))
        self.totals = to_dev(workloads.make_request_totals(w, seed))
        self.req, self.pos, self.slot = (torch.empty(T, dtype=i32, device="cuda")
                                         for _ in range(3))
        self.tok = torch.empty(T, dtype=torch.int64, device="cuda")
        self.input_ids = torch.empty(T, dtype=i32, device="cuda")
        self.qsl = torch.empty(R + 1, dtype=i32, device="cuda")
        self.sl, self.li = (torch.empty(R, dtype=i32, device="cuda") for _ in range(2))
        self.discard = torch.empty(R, dtype=torch.uint8, device="cuda")
        vals = workloads.make_values(w, seed, device="cuda")
        self.q, self.key, self.value = vals["q"], vals["key"], vals["value"]
        self.kc0, self.vc0 = vals["key_cache"], vals["value_cache"]
        self.kc, self.vc = self.kc0.clone(), self.vc0.clone()
        self.out = torch.empty_like(self.q)
        nbytes = pa.pa_attention_workspace_size(R, T, w.max_query_len, w.max_seq_len,
                                                w.num_q_heads, w.num_kv_heads, w.head_dim)
        self.ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")

    def reset_pools(self):
        self.kc.copy_(self.kc0)
        self.vc.copy_(self.vc0)

    def __call__(self):
        w = self.w
        pa.pa_prepare_inputs_ex(self.nst, self.nct, self.bt, w.block_size, w.num_tokens,
                                w.num_blocks, self.req, self.pos, self.slot, self.qsl, self.sl,
                                self.li, token_ids=self.ids, token_indices=self.tok,
                                input_ids=self.input_ids, request_num_tokens=self.totals,
                                discard_request_mask=self.discard)
        pa.pa_cache_write(self.key, self.value, self.kc, self.vc, self.slot)
        pa.pa_attention(self.q, self.kc, self.vc, self.bt, self.qsl, self.sl, w.max_query_len,
                        w.max_seq_len, w.scale, self.out, self.ws)

    def results(self):
        return {k: getattr(self, k).clone() for k in
                ("req", "pos", "slot", "tok", "input_ids", "qsl", "sl", "li", "discard", "kc",
                 "vc", "out")}


def _assert_same(a, b):
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("name", ["tiny", "mixed", "decode"])
def test_graph_replay_equals_eager_launches(name):
    w = workloads.named(name)
    s = Step(w, 5)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        s()                                  # eager once: every kernel loaded
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    assert pa.pa_get_status()[0] == pa.PA_OK

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s()
    torch.cuda.synchronize()

    for seed in (11, 12):
        # new values into the captured buffers
        fresh = workloads.make_values(w, seed, device="cuda")
        s.q.copy_(fresh["q"])
        s.key.copy_(fresh["key"])
        s.value.copy_(fresh["value"])
        del fresh
        s.reset_pools()
        g.replay()
        torch.cuda.synchronize()
        replayed = s.results()
        s.reset_pools()
        s()
        torch.cuda.synchronize()
        _assert_same(replayed, s.results())
        assert pa.pa_get_status() == (pa.PA_OK, 0)

    if name == "tiny":
        # and the replay is the step the oracle computes
        host = {"q": s.q.cpu(), "key": s.key.cpu(), "value": s.value.cpu(),
                "key_cache": s.kc0.cpu(), "value_cache": s.vc0.cpu()}
        idx, kc, vc, ref = oracle.step(w, host)
        np.testing.assert_array_equal(replayed["slot"].cpu().numpy(), idx["slot_mapping"])
        err = np.abs(replayed["out"].double().cpu().numpy() - ref).max()
        assert err <= 1e-2


def test_graph_replay_follows_new_indices():
    # Same shapes, new request state: the replay reads the captured index
    # buffers at run time, so new computed counts / block tables take effect.
    w = workloads.named("tiny")
    s = Step(w, 2)
    s()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s()
    # rotate the physical blocks of every request (still inside the pool)
    bt = w.block_table.copy()
    valid = bt >= 0
    bt[valid] = (bt[valid] + 5) % w.num_blocks
    s.bt.copy_(to_dev(bt))
    s.reset_pools()
    g.replay()
    torch.cuda.synchronize()
    replayed = s.results()
    s.reset_pools()
    s()
    torch.cuda.synchronize()
    _assert_same(replayed, s.results())
    w2 = workloads.Workload(w.name, w.num_scheduled_tokens, w.num_computed_tokens, bt,
                            w.num_blocks, w.block_size, w.num_q_heads, w.num_kv_heads,
                            w.head_dim, w.dtype)
    idx = oracle.prepare_inputs(w2.num_scheduled_tokens, w2.num_computed_tokens, bt,
                                w2.block_size, w2.num_tokens, w2.num_blocks)
    np.testing.assert_array_equal(replayed["slot"].cpu().numpy(), idx["slot_mapping"])


@pytest.mark.parametrize("name", ["decode", "mixed", "decode_fp8", "shared_prefix"])
def test_attention_is_deterministic(name):
    # CTAs take work items in whatever order they free up; an item's
    # arithmetic must not depend on that order: repeated calls on the same
    # inputs give the same bits.
    w = workloads.named(name)
    vals = workloads.make_values(w, 3, device="cuda")
    qsl = to_dev(np.concatenate([[0], np.cumsum(w.num_scheduled_tokens)]).astype(np.int32))
    sl, bt = to_dev(w.context_lens.astype(np.int32)), to_dev(w.block_table)
    nbytes = pa.pa_attention_workspace_size(w.num_reqs, w.num_tokens, w.max_query_len,
                                            w.max_seq_len, w.num_q_heads, w.num_kv_heads,
                                            w.head_dim)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    shared = w.shares_blocks    # the shared-prefix step runs its group items
    outs = []
    for _ in range(3):
        out = torch.full_like(vals["q"], float("nan"))
        pa.pa_attention(vals["q"], vals["key_cache"], vals["value_cache"], bt, qsl, sl,
                        w.max_query_len, w.max_seq_len, w.scale, out, ws,
                        k_scale=vals.get("k_scale"), v_scale=vals.get("v_scale"),
                        shared_blocks=shared)
        outs.append(out)
    torch.cuda.synchronize()
    assert pa.pa_get_status() == (pa.PA_OK, 0)
    assert not torch.isnan(outs[0]).any()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    del vals, outs
    torch.cuda.empty_cache()
