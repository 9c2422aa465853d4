"""CUDA path vs. the oracle, through the C ABI.

Indices and cache contents must match bit for bit; attention within the
stated bound: max |gpu - oracle| <= 1e-2 (bf16/fp16 output, fp32
accumulation, oracle in fp64)."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prepare_gb300 as pa
import workloads
from gpu_step import run_step, to_dev
from helpers import ATOL, check_attention_close, golden, to_bits

pytestmark = pytest.mark.gpu

IDX_KEYS = ("req_indices", "positions", "slot_mapping", "query_start_loc", "seq_lens",
            "logits_indices")


@pytest.fixture(autouse=True)
def clean_status():
    pa.pa_get_status()
    yield


def _oracle_step(w, vals, tokens=None, qsl_capacity=None):
    host = {k: v.cpu() for k, v in vals.items()}
    return oracle.step(w, host, qsl_capacity=qsl_capacity, tokens=tokens)


def _check_indices(res, idx):
    for k in IDX_KEYS:
        np.testing.assert_array_equal(res[k], idx[k], err_msg=k)


def _check_attention(res, ref, tokens=None):
    got = res["out"].float().cpu().numpy().astype(np.float64)
    if tokens is not None:
        got, ref = got[tokens], ref[tokens]
    return check_attention_close(got, ref, res["out"].dtype)


# ---------------------------------------------------------------------------
# Small workloads: everything compared in full
# ---------------------------------------------------------------------------

def test_tiny_step_full_parity():
    w = workloads.tiny()
    vals = workloads.make_values(w, 0)
    res = run_step(w, vals, qsl_capacity=8)
    idx, kc, vc, ref = _oracle_step(w, vals, qsl_capacity=8)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    _check_indices(res, idx)
    np.testing.assert_array_equal(to_bits(res["key_cache"]), kc)
    np.testing.assert_array_equal(to_bits(res["value_cache"]), vc)
    _check_attention(res, ref)


@pytest.mark.parametrize("seed", range(12))
def test_random_small_steps(seed):
    kw = dict(max_computed=1500 if seed % 3 else 200)
    if seed % 4 == 1:
        kw["long_prefill"] = 70
    w = workloads.random_case(seed, **kw)
    vals = workloads.make_values(w, seed, fused_qkv=bool(seed % 2))
    res = run_step(w, vals)
    host = {k: v.cpu() for k, v in vals.items()}
    host["key"] = host["key"].contiguous()
    host["value"] = host["value"].contiguous()
    idx, kc, vc, ref = oracle.step(w, host)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    _check_indices(res, idx)
    np.testing.assert_array_equal(to_bits(res["key_cache"]), kc)
    np.testing.assert_array_equal(to_bits(res["value_cache"]), vc)
    _check_attention(res, ref)


@pytest.mark.parametrize("ws", ["none", "tiny", "default"])
def test_partition_choice_does_not_change_result(ws):
    # Long contexts: the kernel picks its partition length from the workspace
    # it is given (no workspace: one partition per request).
    w = workloads.random_case(77, max_reqs=5, max_computed=3000, head_dim=128, dtype="bf16",
                              group=4, num_kv_heads=2)
    vals = workloads.make_values(w, 77)
    nbytes = {"none": 0, "tiny": 64 * 1024, "default": None}[ws]
    res = run_step(w, vals, workspace_bytes=nbytes)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK
    _check_attention(res, ref)


@pytest.mark.parametrize("longest,hq,hkv", [(10_000, 6, 2), (20_000, 5, 1), (40_000, 6, 2),
                                             (90_000, 3, 3)])
def test_many_partitions_merge(longest, hq, hkv):
    # Long contexts split into 20-176 partitions: the merge pass spreads one
    # head's partitions over 2-8 warps and combines them; head counts that
    # leave a CTA's last heads unused, and short multi-token requests beside.
    rng = np.random.default_rng(longest)
    w = workloads._make("many-splits", [1, 3, 1, 2], [longest - 1, longest // 3, 300, 1000], rng,
                        hq, hkv, 128, "bf16")
    vals = workloads.make_values(w, 3)
    res = run_step(w, vals)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    _check_attention(res, ref)


def _shared_runs_case(seed, group, hkv, dtype, nreq=14):
    """Decode requests whose block tables share 80 blocks (1280 tokens: two
    whole 512-key partitions and a quarter of a third), each with its own
    tail; request 5 diverges inside the second partition, request 7 is a
    3-token chunk, and the last two requests share nothing."""
    rng = np.random.default_rng(seed)
    bs, shared_n = 16, 80
    tails = rng.integers(2, 40, size=nreq)          # private blocks after the prefix
    need = shared_n + int(tails.sum()) + 1 + 2 * 120
    nb = int(need * 1.1) + 8
    perm = [int(b) for b in rng.permutation(nb)]
    shared, k = perm[:shared_n], shared_n
    rows, nst, nct = [], [], []
    for r in range(nreq):
        if r >= nreq - 2:                            # unrelated requests
            own = perm[k:k + 120]
            k += 120
            rows.append(own)
            ctx = 120 * bs - int(rng.integers(0, 15))
        else:
            own = perm[k:k + int(tails[r])]
            k += int(tails[r])
            row = list(shared) + own
            if r == 5:                               # one block of the second partition differs
                row[40] = perm[k]
                k += 1
            rows.append(row)
            ctx = len(row) * bs - int(rng.integers(0, 15))
        n = 3 if r == 7 else 1
        nst.append(n)
        nct.append(ctx - n)
    bt = workloads._tables(rows)
    uniq = np.unique(bt[bt >= 0]).size
    return workloads.Workload(f"shared-runs-{seed}", np.array(nst, np.int32),
                              np.array(nct, np.int32), bt, nb, bs, hkv * group, hkv, 128, dtype,
                              uniq)


@pytest.mark.parametrize("group,hkv,dtype,fp8", [(4, 2, "bf16", False), (1, 2, "fp16", False),
                                                 (8, 1, "bf16", False), (2, 3, "bf16", False),
                                                 (3, 2, "fp16", False), (4, 2, "bf16", True)])
def test_shared_partition_groups(group, hkv, dtype, fp8):
    # Requests reading the same blocks over whole partitions are computed as
    # one group item (up to 32 rows); the rest as usual.  Same results as
    # the oracle, which reads every request's blocks on its own.
    w = _shared_runs_case(group * 10 + hkv, group, hkv, dtype)
    if fp8:
        w = workloads.fp8(w, k_scale=0.3, v_scale=0.2)
    assert w.shares_blocks
    vals = workloads.make_values(w, 5)
    _, _, _, ref = _oracle_step(w, vals)
    for shared in (True, False):   # with and without the group kernel
        res = run_step(w, vals, shared_blocks=shared)
        assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
        _check_attention(res, ref)


def _random_sharing_case(seed):
    """Random requests over a pool where runs of requests share a prefix of
    random length (0-3 partitions and a bit), some diverging at a random
    block, some holding several query tokens; random head shapes."""
    rng = np.random.default_rng(1000 + seed)
    bs = 16
    group = int(rng.choice([1, 2, 3, 4, 8]))
    hkv = int(rng.choice([1, 2, 4]))
    d = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["bf16", "fp16"]))
    nreq = int(rng.integers(2, 40))
    rows, nst, nct, k = [], [], [], 0
    nb = 60_000
    perm = [int(b) for b in rng.permutation(nb)]
    r = 0
    while r < nreq:
        run = int(rng.integers(1, 12))
        shared = perm[k:k + int(rng.integers(0, 110))]
        k += len(shared)
        for _ in range(min(run, nreq - r)):
            row = list(shared)
            if row and rng.random() < 0.2:            # diverge at a random block
                row[int(rng.integers(0, len(row)))] = perm[k]
                k += 1
            tail = int(rng.integers(1, 30))
            row += perm[k:k + tail]
            k += tail
            n = 1 if rng.random() < 0.85 else int(rng.integers(2, 6))
            ctx = len(row) * bs - int(rng.integers(0, bs - n + 1))
            rows.append(row)
            nst.append(n)
            nct.append(ctx - n)
            r += 1
    bt = workloads._tables(rows)
    used = np.unique(bt[bt >= 0])
    # compact the pool to the blocks in use (ids remapped), plus a few spares
    remap = {int(b): i for i, b in enumerate(used)}
    bt = np.vectorize(lambda b: remap.get(int(b), -1))(bt).astype(np.int32)
    w = workloads.Workload(f"rand-share-{seed}", np.array(nst, np.int32), np.array(nct, np.int32),
                           bt, len(used) + 4, bs, hkv * group, hkv, d, dtype, len(used))
    if rng.random() < 0.25:
        w = workloads.fp8(w, k_scale=0.3, v_scale=0.2)
    return w, float(rng.choice([1, 1, 2, 8]))


@pytest.mark.parametrize("seed", range(24))
def test_random_sharing_patterns(seed):
    w, shrink = _random_sharing_case(seed)
    vals = workloads.make_values(w, seed)
    full = pa.pa_attention_workspace_size(w.num_reqs, w.num_tokens, w.max_query_len,
                                          w.max_seq_len, w.num_q_heads, w.num_kv_heads,
                                          w.head_dim)
    _, _, _, ref = _oracle_step(w, vals)
    res = run_step(w, vals, workspace_bytes=max(int(full / shrink), 4096), shared_blocks=True)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    _check_attention(res, ref)


@pytest.mark.parametrize("shrink", [2, 4, 16])
def test_shared_partition_groups_with_longer_partitions(shrink):
    # A smaller workspace makes the kernel pick longer partitions (1024+
    # keys: 64+ pages compared per group check); groups then cover fewer,
    # longer partitions and the last partial one stays per request.
    w = _shared_runs_case(99 + shrink, 4, 2, "bf16", nreq=20)
    vals = workloads.make_values(w, 7)
    full = pa.pa_attention_workspace_size(w.num_reqs, w.num_tokens, w.max_query_len,
                                          w.max_seq_len, w.num_q_heads, w.num_kv_heads,
                                          w.head_dim)
    _, _, _, ref = _oracle_step(w, vals)
    res = run_step(w, vals, workspace_bytes=max(full // shrink, 4096), shared_blocks=True)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    _check_attention(res, ref)


@pytest.mark.parametrize("group,ws", [(4, None), (8, None), (1, 0)])
def test_prompt_chunk_longer_than_a_partition(group, ws):
    # A 600-token chunk at 300 computed spans two 512-key partitions: its first
    # row chunks see nothing of the second partition (empty work items).
    rng = np.random.default_rng(group)
    w = workloads._make("long-chunk", [600, 1, 3], [300, 700, 40], rng, 2 * group, 2, 128,
                        "bf16")
    vals = workloads.make_values(w, group)
    res = run_step(w, vals, workspace_bytes=ws)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK
    _check_attention(res, ref)


@pytest.mark.parametrize("d,dtype,group,hkv", [(128, "bf16", 4, 2), (128, "fp16", 8, 1),
                                               (64, "bf16", 2, 2), (64, "fp16", 1, 3),
                                               (128, "bf16", 16, 1)])
def test_tensor_core_prefill_chunks(d, dtype, group, hkv):
    # Chunks longer than 16 tokens run on the tensor-core kernel: several row
    # tiles, several key tiles, ragged tails, next to short requests that stay
    # on the split-K kernel.
    rng = np.random.default_rng(d + group)
    nst = [300, 1, 17, 5, 129]
    nct = [0, 400, 250, 33, 700]
    w = workloads._make("prefill-mix", nst, nct, rng, hkv * group, hkv, d, dtype)
    vals = workloads.make_values(w, 11)
    res = run_step(w, vals)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    _check_attention(res, ref)


@pytest.mark.parametrize("dtype,fp8,d", [("bf16", False, 128), ("fp16", False, 128),
                                        ("bf16", True, 128), ("fp16", False, 64), ("bf16", True, 64)])
def test_prefill_score_jumps_inside_and_across_tiles(dtype, fp8, d):
    # Keys whose K rows are scaled up make some scores far larger than the
    # rest: inside a 128-key tile the second half's maximum passes the
    # first's by far more than 2^8 (the first half's P, already written, is
    # scaled down), and later tiles move the reference again (O and the row
    # sum are scaled down).  Many rows end near one-hot on a scaled key, with
    # V as drawn (N(0,1)).  Same results as the oracle.
    rng = np.random.default_rng(17)
    w = workloads._make("jumps", [300, 1], [500, 900], rng, 8, 2, d, dtype)
    if fp8:
        w = workloads.fp8(w, k_scale=0.25, v_scale=0.125)
    vals = workloads.make_values(w, 4)
    kc = vals["key_cache"]
    bt = w.block_table[0]
    for lo, hi, f in ((64, 128, 6.0), (600, 640, 9.0), (700, 720, 12.0)):
        for pos in range(lo, hi):
            blk, off = int(bt[pos // 16]), pos % 16
            if fp8:   # E4M3 bytes: scale the decoded value, re-encode
                row = kc[blk, off].view(torch.float8_e4m3fn).float() * f
                kc[blk, off] = row.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            else:
                kc[blk, off] = (kc[blk, off].float() * f).to(kc.dtype)
    res = run_step(w, vals)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    _check_attention(res, ref)


@pytest.mark.parametrize("d,dtype,group,hkv,fp8", [
    (128, "bf16", 3, 2, False), (64, "fp16", 5, 2, False), (128, "bf16", 7, 4, False),
    (128, "fp16", 6, 1, False), (64, "bf16", 48, 1, False), (64, "fp16", 65, 1, False),
    (128, "bf16", 7, 4, True)])
def test_tensor_core_prefill_head_ratios_not_dividing_128(d, dtype, group, hkv, fp8):
    # A 128-row tile holds floor(128/G) whole tokens; the rows left over are
    # zero and never written.  Several tile pairs, a last pair with only its
    # first tile, a tile with a single token (G = 65), next to short requests
    # on the split-K kernel.
    rng = np.random.default_rng(group + d)
    nst = [300, 1, 17, 5, 129]
    nct = [0, 400, 250, 33, 700]
    w = workloads._make("ratio", nst, nct, rng, hkv * group, hkv, d, dtype)
    if fp8:
        w = workloads.fp8(w, k_scale=0.5, v_scale=0.25)
    vals = workloads.make_values(w, group)
    res = run_step(w, vals)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    _check_attention(res, ref)


# (q heads per kv head, kv heads, head_dim, dtype, FP8 pools): ratios that do
# and do not divide 128, up to a single token per tensor-core tile, on both
# kernels (8-row split-K items combine their warps in two passes at D 128)
RATIO_SWEEP = [
    (1, 2, 64, "bf16", False), (2, 2, 128, "fp16", False), (3, 1, 64, "fp16", False),
    (5, 1, 128, "bf16", False), (6, 2, 64, "bf16", False), (9, 1, 128, "fp16", False),
    (10, 1, 64, "fp16", False), (11, 2, 128, "bf16", False), (12, 1, 128, "bf16", False),
    (13, 1, 64, "bf16", False), (14, 1, 128, "fp16", False), (15, 2, 64, "fp16", False),
    (20, 1, 128, "bf16", False), (24, 1, 64, "bf16", False), (32, 1, 128, "fp16", False),
    (40, 1, 128, "bf16", False), (64, 1, 64, "fp16", False), (96, 1, 128, "bf16", False),
    (127, 1, 64, "bf16", False), (128, 1, 128, "fp16", False),
    (3, 2, 128, "bf16", True), (5, 1, 128, "fp16", True), (6, 1, 128, "bf16", True),
    (12, 1, 128, "bf16", True), (16, 1, 64, "bf16", True), (24, 1, 128, "fp16", True),
]


@pytest.mark.parametrize("group,hkv,d,dtype,fp8", RATIO_SWEEP)
def test_head_ratio_sweep(group, hkv, d, dtype, fp8):
    # Random decodes, short chunks (split-K) and chunks of 17..150 tokens
    # (tensor-core kernel), contexts up to ~850 keys (two partitions and the
    # merge pass).  The first request starts from nothing, so its first rows
    # see one to a few keys; the others start anywhere in 0..700.
    rng = np.random.default_rng(1000 * group + d + (7 if fp8 else 0))
    r = int(rng.integers(2, 6, endpoint=True))
    nst = np.where(rng.random(r) < 0.5, 1, rng.integers(2, 25, size=r))
    nst[0] = int(rng.integers(17, 151))
    nct = rng.integers(0, 701, size=r)
    nct[0] = 0
    w = workloads._make("ratio-sweep", nst, nct, rng, hkv * group, hkv, d, dtype)
    if fp8:
        w = workloads.fp8(w, k_scale=0.25, v_scale=0.125)
    vals = workloads.make_values(w, group)
    res = run_step(w, vals)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    _check_attention(res, ref)


def test_head_ratio_above_128_stays_on_split_k():
    # More than 128 q heads per kv head: a token no longer fits a tile, so
    # long requests run on the split-K kernel too.  The third request starts
    # from nothing: 160 rows per token that see one to a few keys each.
    rng = np.random.default_rng(160)
    w = workloads._make("g160", [40, 1, 20], [10, 300, 0], rng, 160, 1, 64, "bf16")
    vals = workloads.make_values(w, 3)
    res = run_step(w, vals)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK
    _check_attention(res, ref)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("fp16", 128)])
def test_attention_sink_rows(dtype, d):
    # Near one-hot rows whose winning weight is not exactly 1.  Key 0 of
    # every request is a sink (K = 30 N(0,1) per element, V = 0), so rows
    # whose q leans its way (a third) take their softmax reference from it;
    # key 130 holds 1.08 times the same K and V = +-3.96875, so on those rows
    # it scores 1 to 5 units higher and carries 77-99% of the weight without
    # moving the reference.  Its weight is then some P in (2.5, 256), the
    # rows come out at 3 < |o| < 3.97 (bf16's [2, 4) binade, half a spacing
    # 0.0078), and rounding P to one bf16 term would add up to
    # 2^-9 * 3.97 = 0.0078 more (a CPU model of that puts the worst element
    # at 0.020).  Key 130 lies in a later unit of the same split-K warp as
    # key 0 at either head_dim, and in the tensor-core kernel's second tile.
    rng = np.random.default_rng(40 + d)
    nst = [200, 1, 1, 7, 1, 33]
    nct = [140, 700, 150, 190, 1500, 260]
    w = workloads._make("sink", nst, nct, rng, 16, 4, d, dtype)
    vals = workloads.make_values(w, 21)
    kc, vc = vals["key_cache"], vals["value_cache"]
    g = torch.Generator().manual_seed(5)
    for r in range(w.num_reqs):
        a, b = int(w.block_table[r][0]), int(w.block_table[r][130 // 16])
        ka = 30.0 * torch.randn(w.num_kv_heads, d, generator=g)
        kc[a, 0] = ka.to(kc.dtype)
        kc[b, 130 % 16] = (1.08 * ka).to(kc.dtype)
        vc[a, 0] = 0
        sign = torch.where(torch.rand(w.num_kv_heads, d, generator=g) < 0.5, -1.0, 1.0)
        vc[b, 130 % 16] = (3.96875 * sign).to(vc.dtype)
    res = run_step(w, vals)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    # the case does what it says: a quarter or more of the outputs past 3 and
    # every one inside the binade where the bound is 1e-2
    assert (np.abs(ref) > 3.0).mean() > 0.25 and np.abs(ref).max() < 4.0
    assert _check_attention(res, ref) <= ATOL


@pytest.mark.parametrize("d", [128, 64])
def test_bf16_values_beyond_f16_range(d):
    # bf16 V values f16 cannot hold (70,000 and 1e30) in a few 64-key halves
    # of the long chunk's context: those halves keep bf16 V on the tensor-core
    # kernel (P split into two bf16 terms), the rest run as f16; decodes read
    # the same keys on the split-K kernel.  Outputs that lean on the large
    # values are large, and are compared at the bf16 output's own spacing.
    rng = np.random.default_rng(70 + d)
    w = workloads._make("big-v", [260, 1, 1, 20], [300, 900, 400, 500], rng, 8, 2, d, "bf16")
    vals = workloads.make_values(w, 6)
    vc = vals["value_cache"]
    g = torch.Generator().manual_seed(1)
    for r in range(w.num_reqs):
        for pos in (70, 200, 333):            # three halves of the first tiles
            blk, off = int(w.block_table[r][pos // 16]), pos % 16
            dims = torch.randperm(d, generator=g)[:3]
            vc[blk, off, :, dims[0]] = 70000.0
            vc[blk, off, :, dims[1]] = -1e30
            vc[blk, off, :, dims[2]] = 65536.0
    res = run_step(w, vals)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    assert np.abs(ref).max() > 1e20            # some rows do lean on the large values
    _check_attention(res, ref)


@pytest.mark.parametrize("long_chunk", [False, True])
def test_stale_slots_past_the_context_are_never_used(long_chunk):
    # Slots of a request's last block past its context hold NaN: neither
    # kernel may let them reach the output.
    rng = np.random.default_rng(9)
    nst = [200, 1, 3] if long_chunk else [1, 1, 3]
    nct = [37, 50, 61]
    w = workloads._make("nan-tail", nst, nct, rng, 8, 2, 128, "bf16")
    vals = workloads.make_values(w, 9)
    kc, vc = vals["key_cache"], vals["value_cache"]
    for r in range(w.num_reqs):
        L = int(w.context_lens[r])
        last = int(w.block_table[r][(L - 1) // 16])
        kc[last, L % 16 or 16:] = float("nan")
        vc[last, L % 16 or 16:] = float("nan")
    res = run_step(w, vals)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK
    _check_attention(res, ref)


@pytest.mark.parametrize("d,dtype,group", [(64, "bf16", 1), (64, "fp16", 8), (128, "fp16", 2),
                                           (128, "bf16", 8), (128, "bf16", 3)])
def test_head_shapes(d, dtype, group):
    w = workloads.random_case(300 + d + group, max_reqs=4, max_computed=700, head_dim=d,
                              dtype=dtype, group=group, num_kv_heads=2, long_prefill=21)
    vals = workloads.make_values(w, 5)
    res = run_step(w, vals)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK
    _check_attention(res, ref)


def test_golden_examples_on_gpu():
    # The pages' worked index examples, block size 4, through the CUDA kernel.
    for name in ("prep_go_program_bs4.json", "block_table_nano_vllm_bs4.json"):
        g = golden(name)["inputs"]
        nst = np.asarray(g["num_scheduled_tokens"], np.int32)
        nct = np.asarray(g["num_computed_tokens"], np.int32)
        bt = np.asarray(g["block_table"], np.int32)
        t = int(nst.sum())
        want = oracle.prepare_inputs(nst, nct, bt, g["block_size"], t, g["num_blocks"])
        outs = [torch.empty(n, dtype=torch.int32, device="cuda")
                for n in (t, t, t, len(nst) + 1, len(nst), len(nst))]
        pa.pa_prepare_inputs(to_dev(nst), to_dev(nct), to_dev(bt), g["block_size"], t,
                             g["num_blocks"], *outs)
        for k, o in zip(IDX_KEYS, outs):
            np.testing.assert_array_equal(o.cpu().numpy(), want[k], err_msg=f"{name}:{k}")
    for c in golden("prep_exercises.json")["cases"]:
        nst = np.asarray(c["num_scheduled_tokens"], np.int32)
        t = int(nst.sum())
        outs = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (t, t, t, 2, 1, 1)]
        pa.pa_prepare_inputs(to_dev(nst), to_dev(np.asarray(c["num_computed_tokens"], np.int32)),
                             to_dev(np.asarray(c["block_table"], np.int32)), c["block_size"], t,
                             c["num_blocks"], *outs)
        assert outs[2].cpu().tolist() == c["slot_mapping_by_hand"]


# ---------------------------------------------------------------------------
# Full-size workloads: indices, pools and attention compared in full
# ---------------------------------------------------------------------------

def _sample_tokens(w, k, seed):
    rng = np.random.default_rng(seed)
    starts = np.concatenate([[0], np.cumsum(w.num_scheduled_tokens)])
    picks = {int(starts[0]), int(starts[-1] - 1)}
    picks |= set(rng.choice(w.num_tokens, size=min(k, w.num_tokens), replace=False).tolist())
    # every request boundary kind: longest context, shortest, multi-token chunk ends
    ctx = w.context_lens
    for r in (int(np.argmax(ctx)), int(np.argmin(ctx)), int(np.argmax(w.num_scheduled_tokens))):
        picks.add(int(starts[r + 1] - 1))
        picks.add(int(starts[r]))
    return np.array(sorted(picks), np.int32)


@pytest.mark.parametrize("name", ["tiny", "decode", "mixed", "mha", "shared_prefix",
                                  "mixed_gqa28_4"])
def test_full_size_workloads(name):
    # The configurations at full size, in the bench's launch configuration:
    # every index, every byte of both pools and every output element against
    # the oracle.
    w = workloads.named(name)
    vals = workloads.make_values(w, 1, device="cuda")
    res = run_step(w, vals)
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    idx, kc, vc, ref = _oracle_step(w, vals)
    _check_indices(res, idx)
    np.testing.assert_array_equal(to_bits(res["key_cache"]), kc)
    np.testing.assert_array_equal(to_bits(res["value_cache"]), vc)
    _check_attention(res, ref)
    del vals, res
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# Edge cases and device-side checks (host-made bad inputs; every access stays
# in bounds because the kernels check before they read)
# ---------------------------------------------------------------------------

def test_empty_step_is_a_no_op():
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    qsl = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    pa.pa_prepare_inputs(e, e, torch.empty(0, 1, dtype=torch.int32, device="cuda"), 16, 0, 4,
                         e, e, e, qsl, e, e)
    assert qsl.cpu().tolist() == [0, 0, 0, 0]
    q = torch.empty(0, 4, 64, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    kv = torch.empty(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    pa.pa_cache_write(kv, kv, pool, pool.clone(), e)
    pa.pa_attention(q, pool, pool, torch.zeros(0, 1, dtype=torch.int32, device="cuda"), qsl[:1],
                    e, 0, 0, 0.125, q)
    assert pa.pa_get_status() == (pa.PA_OK, 0)


def test_negative_slot_skips_and_out_of_pool_slot_is_flagged():
    pool = torch.zeros(2, 16, 1, 64, dtype=torch.float16, device="cuda")
    key = torch.ones(3, 1, 64, dtype=torch.float16, device="cuda")
    slots = torch.tensor([-1, 5, 32], dtype=torch.int32, device="cuda")
    kc, vc = pool.clone(), pool.clone()
    pa.pa_cache_write(key, key, kc, vc, slots)
    st, detail = pa.pa_get_status()
    assert st == pa.PA_ERR_DEVICE_CHECK and pa.check_bits(detail) == {"slot"}
    flat = kc.view(-1, 64)
    assert (flat[5] == 1).all() and (flat[:5] == 0).all() and (flat[6:] == 0).all()


@pytest.mark.parametrize("bad", ["block_id", "empty_request", "token_count", "logical_block"])
def test_prep_device_checks(bad):
    nst = np.array([2, 3], np.int32)
    nct = np.array([5, 0], np.int32)
    bt = np.array([[0, 1], [2, -1]], np.int32)
    t = 5
    if bad == "block_id":
        bt[1, 0] = 9
    elif bad == "empty_request":
        nst[0], t = 0, 3
    elif bad == "token_count":
        t = 7
    elif bad == "logical_block":
        nct[0] = 40
    outs = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (t, t, t, 3, 2, 2)]
    pa.pa_prepare_inputs(to_dev(nst), to_dev(nct), to_dev(bt), 16, t, 4, *outs)
    st, detail = pa.pa_get_status()
    assert st == pa.PA_ERR_DEVICE_CHECK
    assert bad in pa.check_bits(detail)


def test_attention_flags_bad_block_and_bad_lengths():
    w = workloads.random_case(3, max_reqs=3, max_computed=100, head_dim=64)
    vals = workloads.make_values(w, 3)
    res = run_step(w, vals)
    assert res["status"] == pa.PA_OK
    q = vals["q"].cuda()
    bt = to_dev(w.block_table.copy())
    bt[0, 0] = w.num_blocks + 5                      # outside the pool
    o = torch.empty_like(q)
    qsl = torch.from_numpy(res["query_start_loc"]).cuda()
    sl = torch.from_numpy(res["seq_lens"]).cuda()
    pa.pa_attention(q, res["key_cache"], res["value_cache"], bt, qsl, sl, w.max_query_len,
                    w.max_seq_len, w.scale, o)
    st, detail = pa.pa_get_status()
    assert st == pa.PA_ERR_DEVICE_CHECK and "block_id" in pa.check_bits(detail)
    sl_bad = sl.clone()
    sl_bad[0] = w.max_blocks_per_req * 16 + 1          # wider than its table
    pa.pa_attention(q, res["key_cache"], res["value_cache"], to_dev(w.block_table), qsl, sl_bad,
                    w.max_query_len, w.max_seq_len + 32, w.scale, o)
    st, detail = pa.pa_get_status()
    assert st == pa.PA_ERR_DEVICE_CHECK and "seq_len" in pa.check_bits(detail)


def test_seq_len_above_max_seq_len_is_flagged_and_skipped():
    # max_seq_len is the caller's bound on seq_lens: a longer request is
    # flagged and left out; every other request is computed as usual.
    rng = np.random.default_rng(8)
    w = workloads._make("bound", [1, 1, 1, 3], [2900, 1200, 700, 2000], rng, 8, 2, 128, "bf16")
    vals = workloads.make_values(w, 8)
    res = run_step(w, vals)
    assert res["status"] == pa.PA_OK
    _, _, _, ref = _oracle_step(w, vals)
    q = vals["q"].cuda()
    qsl = torch.from_numpy(res["query_start_loc"]).cuda()
    sl = torch.from_numpy(res["seq_lens"]).cuda()
    bound = 2500                                       # request 0 (2901 keys) is past it
    nbytes = pa.pa_attention_workspace_size(w.num_reqs, w.num_tokens, w.max_query_len, bound,
                                            w.num_q_heads, w.num_kv_heads, w.head_dim)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    o = torch.full_like(q, float("nan"))
    pa.pa_attention(q, res["key_cache"], res["value_cache"], to_dev(w.block_table), qsl, sl,
                    w.max_query_len, bound, w.scale, o, ws)
    st, detail = pa.pa_get_status()
    assert st == pa.PA_ERR_DEVICE_CHECK and pa.check_bits(detail) == {"seq_len"}
    got = o.float().cpu().numpy().astype(np.float64)
    assert np.abs(got[1:] - ref[1:]).max() <= ATOL


def test_host_side_rejections():
    q = torch.zeros(2, 4, 96, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(4, 16, 2, 96, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_attention(q, pool, pool, torch.zeros(2, 1, dtype=torch.int32, device="cuda"),
                        torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda"), i, 1, 1,
                        0.1, q)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    with pytest.raises(TypeError):
        pa.pa_attention(q.cpu(), pool, pool, i, i, i, 1, 1, 0.1, q)


def test_launch_count():
    w = workloads.tiny()
    vals = workloads.make_values(w, 0)
    pa.pa_launch_count()
    run_step(w, vals)
    assert pa.pa_launch_count() >= 3


def test_bounded_wait_times_out_and_context_survives():
    # A wait on a barrier nothing completes ends with a timeout status, not a
    # hang, and the next step on the same context is still correct.
    pa.pa_selftest_wait_timeout()
    st, detail = pa.pa_get_status()
    assert st == pa.PA_ERR_TIMEOUT and pa.check_bits(detail) == {"timeout"}
    w = workloads.tiny()
    vals = workloads.make_values(w, 0)
    res = run_step(w, vals)
    _, _, _, ref = _oracle_step(w, vals)
    assert res["status"] == pa.PA_OK
    _check_attention(res, ref)
