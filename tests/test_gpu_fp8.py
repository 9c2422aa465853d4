"""FP8 (E4M3) KV cache on the GPU vs. the oracle, through the C ABI: the
quantising write must match byte for byte, attention over FP8 pools within
the same bound as 16-bit pools (max |gpu - oracle| <= 1e-2; the oracle reads
the same E4M3 bytes exactly, so the bound covers the kernel's own rounding)."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prepare_gb300 as pa
import workloads
from gpu_step import run_step, to_dev
from helpers import check_attention_close

pytestmark = pytest.mark.gpu

ATOL = 1e-2
DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(autouse=True)
def clean_status():
    pa.pa_get_status()
    yield


def _bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def _scales(ks, vs):
    return (torch.tensor([ks], dtype=torch.float32, device="cuda"),
            torch.tensor([vs], dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("hkv,d", [(1, 64), (8, 128), (3, 64), (40, 128)])
@pytest.mark.parametrize("fused", [False, True])
def test_fp8_write_matches_oracle(dtype, hkv, d, fused):
    rng = np.random.default_rng(hkv * d)
    t, bs, nb = 37, 16, 20
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    hq = hkv * 2
    if fused:
        qkv = (torch.randn(t, (hq + 2 * hkv) * d, generator=g, device="cuda") * 5).to(DT[dtype])
        key = qkv[:, hq * d:(hq + hkv) * d].view(t, hkv, d)
        value = qkv[:, (hq + hkv) * d:].view(t, hkv, d)
    else:
        key = (torch.randn(t, hkv, d, generator=g, device="cuda") * 5).to(DT[dtype])
        value = (torch.randn(t, hkv, d, generator=g, device="cuda") * 300).to(DT[dtype])
    slots = rng.permutation(nb * bs)[:t].astype(np.int32)
    slots[3] = -1
    kc = torch.from_numpy(rng.integers(0, 256, size=(nb, bs, hkv, d)).astype(np.uint8)).cuda()
    vc = torch.from_numpy(rng.integers(0, 256, size=(nb, bs, hkv, d)).astype(np.uint8)).cuda()
    k0, v0 = _bytes(kc), _bytes(vc)
    ks, vs = _scales(0.3, 0.7)     # V / 0.7 passes 448 here: saturation is exercised
    pa.pa_cache_write(key, value, kc, vc, to_dev(slots), k_scale=ks, v_scale=vs)
    assert pa.pa_get_status() == (pa.PA_OK, 0)
    kb, vb, st = oracle.cache_write_fp8(key.contiguous(), value.contiguous(), k0, v0, slots, hkv,
                                        d, bs, nb, dtype, 0.3, 0.7)
    assert st == 0
    np.testing.assert_array_equal(_bytes(kc), kb)
    np.testing.assert_array_equal(_bytes(vc), vb)


def test_fp8_write_without_scales_is_scale_one_and_keeps_nan():
    key = torch.tensor([[[1.0, 500.0, -1e4, float("nan")] * 2]], dtype=torch.bfloat16,
                       device="cuda")
    kc = torch.zeros(1, 16, 1, 8, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    pa.pa_cache_write(key, key, kc, vc, to_dev(np.array([5], np.int32)))
    row = kc.view(-1, 8)[5].cpu().numpy()
    assert row[:3].tolist() == [0x38, 0x7E, 0xFE] and row[3] & 0x7F == 0x7F


def _fp8_case(seed, **kw):
    w = workloads.random_case(seed, **kw)
    return workloads.fp8(w, k_scale=0.25 + 0.05 * (seed % 3), v_scale=0.125)


def _check_step(w, vals, tokens=None):
    res = run_step(w, vals)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    host = {k: v.cpu() for k, v in vals.items()}
    idx, kc, vc, ref = oracle.step(w, host, tokens=tokens)
    np.testing.assert_array_equal(_bytes(res["key_cache"]).reshape(kc.shape), kc)
    np.testing.assert_array_equal(_bytes(res["value_cache"]).reshape(vc.shape), vc)
    got = res["out"].double().cpu().numpy()
    if tokens is not None:
        got, ref = got[tokens], ref[tokens]
    return check_attention_close(got, ref, res["out"].dtype)


@pytest.mark.parametrize("seed", range(10))
def test_fp8_random_steps(seed):
    w = _fp8_case(seed, max_reqs=8, max_new=20, max_computed=900)
    _check_step(w, workloads.make_values(w, seed))


@pytest.mark.parametrize("d,dtype,group", [(64, "bf16", 1), (64, "fp16", 4), (128, "bf16", 8),
                                           (128, "fp16", 2), (128, "bf16", 3)])
def test_fp8_head_shapes(d, dtype, group):
    w = _fp8_case(40 + group, max_reqs=5, max_new=16, max_computed=700, head_dim=d, dtype=dtype,
                  group=group, num_kv_heads=2)
    _check_step(w, workloads.make_values(w, 2))


@pytest.mark.parametrize("d,dtype,group,hkv", [(128, "bf16", 4, 2), (64, "bf16", 4, 2),
                                               (64, "fp16", 1, 3), (64, "bf16", 7, 1),
                                               (64, "fp16", 16, 1)])
def test_fp8_long_chunk(d, dtype, group, hkv):
    # A 200-token prompt chunk over FP8 pools runs on the tensor-core kernel,
    # which widens each landed E4M3 tile to f16 in shared memory (head_dim
    # 128: in place; 64: from a staging area).  Short requests beside it stay
    # on the split-K kernel.
    w = _fp8_case(77 + d + group, max_reqs=3, max_new=8, max_computed=300, long_prefill=200,
                  head_dim=d, dtype=dtype, group=group, num_kv_heads=hkv)
    _check_step(w, workloads.make_values(w, 5))


def test_fp8_head_dim_64_prompt_tiles():
    # Head_dim 64 over FP8 pools, a 600-token chunk at 500 computed: many
    # 128-key tiles and both staging stages of K and V, a ragged last tile.
    rng = np.random.default_rng(64)
    w = workloads._make("fp8-d64", [600, 1, 3], [500, 900, 40], rng, 8, 2, 64, "bf16")
    w = workloads.fp8(w, k_scale=0.25, v_scale=0.125)
    _check_step(w, workloads.make_values(w, 9))


@pytest.mark.parametrize("name", ["decode_fp8", "mixed_fp8", "chunk_fp8_d64"])
def test_fp8_full_size(name):
    # Every byte of both pools and every output element against the oracle.
    w = workloads.named(name)
    vals = workloads.make_values(w, 1, device="cuda")
    _check_step(w, vals)
    del vals
    torch.cuda.empty_cache()


def test_fp8_matches_16_bit_pools_holding_the_same_values():
    # Same cached values two ways: FP8 bytes with power-of-two scales, and
    # bf16 pools holding element * scale exactly.  Both GPU outputs are near
    # each other and the oracle.
    w16 = workloads.random_case(5, max_reqs=6, max_new=12, max_computed=500, head_dim=128,
                                dtype="bf16", group=4, num_kv_heads=2)
    w8 = workloads.fp8(w16, k_scale=0.25, v_scale=0.125)
    v8 = workloads.make_values(w8, 8)
    v16 = dict(v8)
    for k, sc in (("key_cache", 0.25), ("value_cache", 0.125)):
        v16[k] = (v8[k].view(torch.float8_e4m3fn).float() * sc).to(torch.bfloat16)
    del v16["k_scale"], v16["v_scale"]
    # both steps write the same new tokens; compare attention only where the
    # written values agree: quantise the new K/V first so both pools hold them
    ks, vs = 0.25, 0.125
    v16["key"] = ((v8["key"].float() / ks).to(torch.float8_e4m3fn).float() * ks).to(torch.bfloat16)
    v16["value"] = ((v8["value"].float() / vs).to(torch.float8_e4m3fn).float() * vs).to(
        torch.bfloat16)
    r8 = run_step(w8, v8)
    r16 = run_step(w16, v16)
    assert r8["status"] == pa.PA_OK and r16["status"] == pa.PA_OK
    a, b = r8["out"].double(), r16["out"].double()
    assert (a - b).abs().max().item() <= 2 * ATOL


def test_fp8_block_ops():
    kc = torch.randint(0, 256, (64, 16, 8, 128), dtype=torch.uint8, device="cuda")
    vc = torch.randint(0, 256, (64, 16, 8, 128), dtype=torch.uint8, device="cuda")
    k0, v0 = _bytes(kc).reshape(64, -1), _bytes(vc).reshape(64, -1)
    src, dst = np.arange(0, 20, dtype=np.int32), np.arange(30, 50, dtype=np.int32)
    pa.pa_copy_blocks(kc, vc, to_dev(src), to_dev(dst))
    pa.pa_zero_blocks(kc, vc, to_dev(np.array([60, 61], np.int32)))
    assert pa.pa_get_status() == (pa.PA_OK, 0)
    kb, vb, _ = oracle.copy_blocks(k0, v0, src, dst)
    kb, vb, _ = oracle.zero_blocks(kb, vb, [60, 61])
    np.testing.assert_array_equal(_bytes(kc).reshape(64, -1), kb)
    np.testing.assert_array_equal(_bytes(vc).reshape(64, -1), vb)
