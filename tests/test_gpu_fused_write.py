"""pa_prepare_and_write: the index build and the cache write in one launch
("How vLLM Works Internally", section "Fused Kernels").  Its outputs must be,
bit for bit, those of pa_prepare_inputs followed by pa_cache_write, and so
the oracle's."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prepare_gb300 as pa
import workloads
from gpu_step import run_step, to_dev
from helpers import to_bits

pytestmark = pytest.mark.gpu

IDX = ("req_indices", "positions", "slot_mapping", "query_start_loc", "seq_lens",
       "logits_indices")


@pytest.fixture(autouse=True)
def clean_status():
    pa.pa_get_status()
    yield


def _bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def _same_as_two_calls_and_oracle(w, vals):
    two = run_step(w, vals)
    one = run_step(w, vals, fused=True)
    assert one["status"] == two["status"] == pa.PA_OK, pa.check_bits(one["detail"])
    for k in IDX:
        np.testing.assert_array_equal(one[k], two[k], err_msg=k)
    for k in ("key_cache", "value_cache"):
        np.testing.assert_array_equal(_bytes(one[k]), _bytes(two[k]), err_msg=k)
    assert torch.equal(one["out"], two["out"])
    host = {k: v.cpu() for k, v in vals.items()}
    idx, kc, vc, _ = oracle.step(w, host, tokens=np.zeros(0, np.int32))
    for k in IDX:
        np.testing.assert_array_equal(one[k], idx[k], err_msg=k)
    for k, want in (("key_cache", kc), ("value_cache", vc)):
        np.testing.assert_array_equal(_bytes(one[k]).reshape(-1),
                                      np.ascontiguousarray(want).view(np.uint8).reshape(-1))


@pytest.mark.parametrize("name", ["tiny", "decode", "mixed", "mha", "shared_prefix"])
def test_fused_matches_two_calls_on_the_workloads(name):
    w = workloads.named(name)
    _same_as_two_calls_and_oracle(w, workloads.make_values(w, 1, device="cuda"))


@pytest.mark.parametrize("seed", range(6))
def test_fused_matches_two_calls_random(seed):
    w = workloads.random_case(400 + seed, max_reqs=8, max_computed=900,
                              long_prefill=40 if seed % 2 else 0)
    _same_as_two_calls_and_oracle(w, workloads.make_values(w, seed, fused_qkv=bool(seed % 3)))


@pytest.mark.parametrize("name", ["decode_fp8", "mixed_fp8"])
def test_fused_matches_two_calls_fp8(name):
    w = workloads.named(name)
    _same_as_two_calls_and_oracle(w, workloads.make_values(w, 1, device="cuda"))


def test_fused_flags_bad_blocks_and_skips_their_rows():
    # a block id past the pool: the token gets slot -1, its row is not
    # written, the same status bit is set as by the two separate calls
    rng = np.random.default_rng(3)
    w = workloads._make("badblock", [3, 1], [30, 10], rng, 4, 2, 64, "bf16")
    w.block_table[0, 1] = w.num_blocks + 5
    vals = workloads.make_values(w, 2)
    res = {}
    for fused in (False, True):
        res[fused] = run_step(w, vals, fused=fused)
        assert res[fused]["status"] == pa.PA_ERR_DEVICE_CHECK
        assert pa.check_bits(res[fused]["detail"]) >= {"block_id"}
    for k in IDX:
        np.testing.assert_array_equal(res[True][k], res[False][k], err_msg=k)
    assert (res[True]["slot_mapping"][:3] == -1).sum() >= 1
    for k in ("key_cache", "value_cache"):
        np.testing.assert_array_equal(to_bits(res[True][k]), to_bits(res[False][k]))


def test_fused_rejects_unaligned_rows():
    # 16-bit rows of an odd number of elements: the fused kernel copies 16-byte
    # vectors only; the two separate calls take any alignment
    nst = to_dev(np.array([2], np.int32))
    nct = to_dev(np.array([0], np.int32))
    bt = to_dev(np.array([[0]], np.int32))
    i = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (2, 2, 2, 2, 1, 1)]
    key = torch.zeros(2, 1, 12, dtype=torch.bfloat16, device="cuda")   # 24-byte rows
    pool = torch.zeros(1, 16, 1, 12, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_prepare_and_write(nst, nct, bt, 16, 2, 1, *i, key, key, pool, pool.clone())
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
