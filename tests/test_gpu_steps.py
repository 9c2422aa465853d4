"""Consecutive engine steps on the same pools and the same attention
workspace.

Between steps, requests finish and new ones join with a prompt chunk. The
others decode one token more each step, so their contexts grow by the
tokens the previous step wrote. Every step must match the oracle run on the
pools as the previous steps left them. This covers the per-call state
(the item counters in the workspace's control block, the partition
choice, the merge metadata): nothing may carry over from one call to the
next."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prepare_gb300 as pa
import workloads
from gpu_step import to_dev
from helpers import to_bits

pytestmark = pytest.mark.gpu

BS, HQ, HKV, D = 16, 8, 2, 128
NB = 4000


@pytest.fixture(autouse=True)
def clean_status():
    pa.pa_get_status()
    yield


class Engine:
    """Request state of a small engine: block lists from one free list."""

    def __init__(self, rng, shared):
        self.rng = rng
        self.free = [int(b) for b in rng.permutation(NB)]
        self.reqs = []                      # dicts: blocks, computed, next (tokens to schedule)
        prefix = [self.free.pop() for _ in range(64)] if shared else None
        for i in range(10):
            ctx = int(rng.integers(100, 2500))
            blocks = []
            if prefix is not None and i < 5:   # five requests share a 1024-token prefix
                blocks = list(prefix)
                ctx = 1024 + int(rng.integers(1, 900))
            self.reqs.append({"blocks": blocks, "computed": ctx - 1, "next": 1})
            self._grow(self.reqs[-1])

    def _grow(self, r):
        need = -(-(r["computed"] + r["next"]) // BS)
        while len(r["blocks"]) < need:
            r["blocks"].append(self.free.pop())

    def advance(self):
        """The previous step's tokens are now context; some requests finish,
        new ones join with a prompt chunk, the rest decode one token."""
        for r in self.reqs:
            r["computed"] += r["next"]
            r["next"] = 1
        keep = [r for r in self.reqs if self.rng.random() > 0.15]
        for _ in range(int(self.rng.integers(0, 3))):
            n = int(self.rng.integers(20, 300))
            keep.append({"blocks": [], "computed": int(self.rng.integers(0, 1500)), "next": n})
        self.reqs = keep
        for r in self.reqs:
            self._grow(r)

    def workload(self, name):
        nst = np.array([r["next"] for r in self.reqs], np.int32)
        nct = np.array([r["computed"] for r in self.reqs], np.int32)
        bt = workloads._tables([r["blocks"] for r in self.reqs])
        return workloads.Workload(name, nst, nct, bt, NB, BS, HQ, HKV, D, "bf16",
                                  int(np.unique(bt[bt >= 0]).size))


def _bits_to_pool(bits, like):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).reshape(
        like.shape)


@pytest.mark.parametrize("shared", [False, True])
def test_consecutive_steps_share_pools_and_workspace(shared):
    rng = np.random.default_rng(31 + shared)
    eng = Engine(rng, shared)
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    kc = torch.randn(NB, BS, HKV, D, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(NB, BS, HKV, D, generator=g, device="cuda").to(torch.bfloat16)
    host_k, host_v = kc.cpu(), vc.cpu()
    # one workspace for every step, sized for the largest
    ws = torch.empty(pa.pa_attention_workspace_size(32, 1024, 300, 4096, HQ, HKV, D),
                     dtype=torch.uint8, device="cuda")
    i32 = torch.int32
    for step in range(5):
        if step:
            eng.advance()
        w = eng.workload(f"step-{step}")
        vals = workloads.make_values(w, 100 + step, device="cuda")   # q and the new K/V only
        R, T = w.num_reqs, w.num_tokens
        nst, nct, bt = (to_dev(w.num_scheduled_tokens), to_dev(w.num_computed_tokens),
                        to_dev(w.block_table))
        req, pos, slot = (torch.empty(T, dtype=i32, device="cuda") for _ in range(3))
        qsl = torch.empty(R + 1, dtype=i32, device="cuda")
        sl, li = (torch.empty(R, dtype=i32, device="cuda") for _ in range(2))
        pa.pa_prepare_inputs(nst, nct, bt, BS, T, NB, req, pos, slot, qsl, sl, li)
        pa.pa_cache_write(vals["key"], vals["value"], kc, vc, slot)
        out = torch.full_like(vals["q"], float("nan"))
        pa.pa_attention(vals["q"], kc, vc, bt, qsl, sl, w.max_query_len, w.max_seq_len, w.scale,
                        out, ws, shared_blocks=shared and w.shares_blocks)
        assert pa.pa_get_status() == (pa.PA_OK, 0), step
        host = {"q": vals["q"].cpu(), "key": vals["key"].cpu(), "value": vals["value"].cpu(),
                "key_cache": host_k, "value_cache": host_v}
        idx, kb, vb, ref = oracle.step(w, host)
        np.testing.assert_array_equal(slot.cpu().numpy(), idx["slot_mapping"])
        np.testing.assert_array_equal(to_bits(kc), kb)
        np.testing.assert_array_equal(to_bits(vc), vb)
        err = np.abs(out.double().cpu().numpy() - ref).max()
        assert err <= 1e-2, (step, err)
        host_k, host_v = _bits_to_pool(kb, host_k), _bits_to_pool(vb, host_v)
