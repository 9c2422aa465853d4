"""Copy-on-write block copies and new-block zeroing on the GPU vs. the
oracle, through the C ABI.  Pool contents must match byte for byte."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prepare_gb300 as pa
import workloads
from gpu_step import run_step, to_dev
from helpers import to_bits

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(autouse=True)
def clean_status():
    pa.pa_get_status()
    yield


def _pool(nb, bs, hkv, d, dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    mk = lambda: torch.randn(nb, bs, hkv, d, generator=g, device="cuda").to(DT[dtype])
    return mk(), mk()


def _bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy().reshape(t.shape[0], -1)


def _fresh_pairs(rng, nb, n, fan_out=False):
    blocks = rng.permutation(nb)
    dst = blocks[:n]
    src = np.full(n, blocks[n]) if fan_out else blocks[n:2 * n]
    return src.astype(np.int32), dst.astype(np.int32)


# shapes: block bytes below one 16 KiB chunk, a ragged multiple, exact chunks,
# and the 40-head LLaMA-13B block (10 chunks)
SHAPES = [(16, 1, 64, "bf16"), (16, 3, 64, "fp16"), (16, 8, 128, "bf16"), (16, 40, 128, "fp16"),
          (4, 2, 64, "bf16"), (1, 1, 8, "fp16")]


@pytest.mark.parametrize("bs,hkv,d,dtype", SHAPES)
@pytest.mark.parametrize("fan_out", [False, True])
def test_copy_blocks_vs_oracle(bs, hkv, d, dtype, fan_out):
    nb = 300
    rng = np.random.default_rng(bs * 1000 + hkv * 10 + d)
    kc, vc = _pool(nb, bs, hkv, d, dtype, 1)
    k0, v0 = _bytes(kc), _bytes(vc)
    for n in (1, 37, 149):
        src, dst = _fresh_pairs(rng, nb, n, fan_out)
        pa.pa_copy_blocks(kc, vc, to_dev(src), to_dev(dst))
        kb, vb, st = oracle.copy_blocks(k0, v0, src, dst)
        assert st == 0
        assert pa.pa_get_status() == (pa.PA_OK, 0)
        np.testing.assert_array_equal(_bytes(kc), kb)
        np.testing.assert_array_equal(_bytes(vc), vb)
        k0, v0 = kb, vb


@pytest.mark.parametrize("bs,hkv,d,dtype", SHAPES)
def test_zero_blocks_vs_oracle(bs, hkv, d, dtype):
    nb = 300
    rng = np.random.default_rng(7 + hkv)
    kc, vc = _pool(nb, bs, hkv, d, dtype, 2)
    kc[5] = float("nan")                          # a stale NaN block among the victims
    k0, v0 = _bytes(kc), _bytes(vc)
    ids = np.concatenate([[5], rng.choice(np.arange(6, nb), size=60, replace=False)])
    ids = ids.astype(np.int32)
    pa.pa_zero_blocks(kc, vc, to_dev(ids))
    kb, vb, st = oracle.zero_blocks(k0, v0, ids)
    assert pa.pa_get_status() == (pa.PA_OK, 0)
    np.testing.assert_array_equal(_bytes(kc), kb)
    np.testing.assert_array_equal(_bytes(vc), vb)
    assert (kc[5] == 0).all() and not torch.signbit(kc[5].float()).any()


def test_out_of_pool_ids_are_flagged_and_skipped():
    kc, vc = _pool(40, 16, 2, 64, "bf16", 3)
    k0, v0 = _bytes(kc), _bytes(vc)
    src = np.array([1, 40, -3, 2], np.int32)
    dst = np.array([10, 11, 12, 41], np.int32)
    pa.pa_copy_blocks(kc, vc, to_dev(src), to_dev(dst))
    st, detail = pa.pa_get_status()
    assert st == pa.PA_ERR_DEVICE_CHECK and pa.check_bits(detail) == {"block_id"}
    kb, vb, _ = oracle.copy_blocks(k0, v0, src, dst, check=False)
    np.testing.assert_array_equal(_bytes(kc), kb)
    np.testing.assert_array_equal(_bytes(vc), vb)
    pa.pa_zero_blocks(kc, vc, to_dev(np.array([3, 99], np.int32)))
    st, detail = pa.pa_get_status()
    assert st == pa.PA_ERR_DEVICE_CHECK and pa.check_bits(detail) == {"block_id"}
    assert (kc[3] == 0).all()


def test_empty_lists_are_no_ops():
    kc, vc = _pool(8, 16, 1, 64, "bf16", 4)
    k0 = _bytes(kc)
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(kc, vc, e, e)
    pa.pa_zero_blocks(kc, vc, e)
    assert pa.pa_get_status() == (pa.PA_OK, 0)
    np.testing.assert_array_equal(_bytes(kc), k0)


@pytest.mark.parametrize("name", ["decode", "mha"])
def test_full_size_pools_sampled(name):
    # The workload's own pools (GBs): 4096 copies and 4096 zeroed blocks.
    # The oracle runs on a compact pool holding every block involved plus a
    # sample of untouched ones, ids remapped; that pool's blocks must match.
    w = workloads.named(name)
    vals = workloads.make_values(w, 9, device="cuda")
    kc, vc = vals["key_cache"], vals["value_cache"]
    rng = np.random.default_rng(12)
    n = min(4096, w.num_blocks // 3)
    perm = rng.permutation(w.num_blocks).astype(np.int32)
    src, dst, zero = perm[:n], perm[n:2 * n], perm[2 * n:3 * n]
    others = rng.choice(perm[3 * n:], size=min(64, w.num_blocks - 3 * n), replace=False)
    keep = np.concatenate([src, dst, zero, others]).astype(np.int32)
    remap = {int(b): i for i, b in enumerate(keep)}
    k0, v0 = _bytes(kc[to_dev(keep).long()]), _bytes(vc[to_dev(keep).long()])
    pa.pa_copy_blocks(kc, vc, to_dev(src), to_dev(dst))
    pa.pa_zero_blocks(kc, vc, to_dev(zero))
    assert pa.pa_get_status() == (pa.PA_OK, 0)
    m = np.vectorize(remap.get)
    kb, vb, _ = oracle.copy_blocks(k0, v0, m(src), m(dst))
    kb, vb, _ = oracle.zero_blocks(kb, vb, m(zero))
    np.testing.assert_array_equal(_bytes(kc[to_dev(keep).long()]), kb)
    np.testing.assert_array_equal(_bytes(vc[to_dev(keep).long()]), vb)
    del vals, kc, vc
    torch.cuda.empty_cache()


def test_beam_fork_through_the_whole_step():
    # 8 beams share a 1000-token prefix whose last block holds 8 of its 16
    # slots.  Each beam but the first copies that block, remaps its table,
    # then the step writes each beam's own new token and attends.  Every beam
    # must see the shared prefix plus only its own token.
    bs, hq, hkv, d, dtype = 16, 8, 2, 128, "bf16"
    beams, prefix = 8, 1000
    nfull, tail = divmod(prefix, bs)               # 62 full blocks + 8 tokens
    nb = nfull + 1 + beams + 4
    rng = np.random.default_rng(21)
    blocks = rng.permutation(nb).astype(np.int32)
    shared, last, fresh = blocks[:nfull], blocks[nfull], blocks[nfull + 1:nfull + beams]
    table = np.tile(np.concatenate([shared, [last]]), (beams, 1)).astype(np.int32)
    nct = np.full(beams, prefix, np.int32)
    nst = np.ones(beams, np.int32)
    w = workloads.Workload("beams", nst, nct, table, nb, bs, hq, hkv, d, dtype)
    vals = workloads.make_values(w, 4, device="cuda")
    # copy-on-write: beams 1.. get their own copy of the partial block
    kc, vc = vals["key_cache"].clone(), vals["value_cache"].clone()
    pa.pa_copy_blocks(kc, vc, to_dev(np.full(beams - 1, last, np.int32)), to_dev(fresh))
    table[1:, nfull] = fresh
    w2 = workloads.Workload("beams", nst, nct, table, nb, bs, hq, hkv, d, dtype)
    vals2 = dict(vals, key_cache=kc, value_cache=vc)
    res = run_step(w2, vals2)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    # oracle: the same copy, remap and step on the host
    kb, vb, _ = oracle.copy_blocks(vals["key_cache"], vals["value_cache"],
                                   np.full(beams - 1, last, np.int32), fresh)
    host = {k: v.cpu() for k, v in vals.items()}
    host["key_cache"] = torch.from_numpy(kb.view(np.int16).reshape(
        vals["key_cache"].shape)).view(torch.bfloat16)
    host["value_cache"] = torch.from_numpy(vb.view(np.int16).reshape(
        vals["value_cache"].shape)).view(torch.bfloat16)
    idx, kco, vco, ref = oracle.step(w2, host)
    np.testing.assert_array_equal(res["slot_mapping"], idx["slot_mapping"])
    assert len(set(idx["slot_mapping"].tolist())) == beams      # every beam writes its own slot
    np.testing.assert_array_equal(to_bits(res["key_cache"]), kco)
    np.testing.assert_array_equal(to_bits(res["value_cache"]), vco)
    err = np.abs(res["out"].double().cpu().numpy() - ref).max()
    assert err <= 1e-2
