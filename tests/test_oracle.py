"""Pins for the CPU oracle: printed worked examples, hand-derived answers,
closed forms, brute force and invariances.  None of these compares the
oracle with itself or with the CUDA path."""

import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import (brute_attention, brute_prepare, dense_causal_numpy, from_bits,
                     golden, scatter_to_pool, to_bits)


# ---------------------------------------------------------------------------
# Index build: worked examples printed on the pages
# ---------------------------------------------------------------------------

def _table_for(nst, nct, bs, nb, rng):
    need = [-(-(int(c) + int(n)) // bs) for n, c in zip(nst, nct)]
    perm = rng.permutation(nb)
    bt = np.full((len(nst), max(need)), -1, np.int32)
    k = 0
    for r, m in enumerate(need):
        bt[r, :m] = perm[k:k + m]
        k += m
    return bt


def test_prep_worked_example_2_5_3():
    g = golden("prep_worked_example_2_5_3.json")
    nst = g["inputs"]["num_scheduled_tokens"]
    nct = g["inputs"]["num_computed_tokens"]
    bs = g["inputs"]["block_size"]
    bt = _table_for(nst, nct, bs, 64, np.random.default_rng(0))
    out = oracle.prepare_inputs(nst, nct, bt, bs, sum(nst), 64)
    p = g["printed"]
    assert out["req_indices"].tolist() == p["req_indices"]
    assert out["query_start_loc"].tolist() == p["query_start_loc"]
    assert out["query_start_loc"][1:].tolist() == p["cu_num_tokens"]
    assert out["logits_indices"].tolist() == p["logits_indices"]
    qpos = out["positions"] - np.asarray(nct)[out["req_indices"]]
    assert qpos.tolist() == p["query_pos"]
    # R1 reaches 102, R2 5 of 600, R3 43 of 60 (the page's request state)
    assert out["seq_lens"].tolist() == [102, 5, 43]


def test_prep_packed_abc():
    g = golden("prep_packed_abc.json")
    i = g["inputs"]
    bt = _table_for(i["num_scheduled_tokens"], i["num_computed_tokens"], 16, 32,
                    np.random.default_rng(1))
    out = oracle.prepare_inputs(i["num_scheduled_tokens"], i["num_computed_tokens"], bt, 16,
                                6, 32)
    assert out["positions"].tolist() == g["printed"]["positions"]
    assert out["query_start_loc"].tolist() == g["printed"]["query_start_loc"]


def test_prep_go_program_printed_and_hand_derived():
    g = golden("prep_go_program_bs4.json")
    i = g["inputs"]
    out = oracle.prepare_inputs(i["num_scheduled_tokens"], i["num_computed_tokens"],
                                i["block_table"], i["block_size"], 9, i["num_blocks"])
    p = g["printed"]
    assert out["positions"][1:6].tolist() == p["positions_of_B"]
    assert out["positions"][0] == p["position_of_A"]
    assert out["slot_mapping"][1:5].tolist() == p["slots_of_B_positions_4_to_7"]
    assert out["slot_mapping"][5] == p["slot_of_B_position_8"]
    h = g["derived_by_hand"]
    for k in ("slot_mapping", "query_start_loc", "seq_lens", "logits_indices",
              "req_indices", "positions"):
        assert out[k].tolist() == h[k], k


def test_prep_exercises_by_hand():
    for c in golden("prep_exercises.json")["cases"]:
        out = oracle.prepare_inputs(c["num_scheduled_tokens"], c["num_computed_tokens"],
                                    c["block_table"], c["block_size"],
                                    sum(c["num_scheduled_tokens"]), c["num_blocks"])
        assert out["slot_mapping"].tolist() == c["slot_mapping_by_hand"], c["name"]


def test_prep_nano_vllm_block_table():
    g = golden("block_table_nano_vllm_bs4.json")
    i = g["inputs"]
    out = oracle.prepare_inputs(i["num_scheduled_tokens"], i["num_computed_tokens"],
                                i["block_table"], i["block_size"], 10, i["num_blocks"])
    assert out["slot_mapping"].tolist() == g["derived_by_hand"]["slot_mapping"]
    for lb, phys in g["printed"]["logical_to_physical"].items():
        toks = g["printed"]["tokens_per_logical_block"][int(lb)]
        assert all(out["slot_mapping"][t] // 4 == phys for t in toks)


def test_prep_query_start_loc_tail_padding():
    # "Building the Batch": the unused tail is filled with the total.
    out = oracle.prepare_inputs([2, 5, 3], [0, 0, 0], [[0], [1], [2]], 16, 10, 4,
                                qsl_capacity=8)
    assert out["query_start_loc"].tolist() == [0, 2, 7, 10, 10, 10, 10, 10]


# ---------------------------------------------------------------------------
# Index build: brute force and invariants
# ---------------------------------------------------------------------------

def _check_invariants(nst, nct, bt, bs, out):
    qsl = out["query_start_loc"]
    assert np.all(np.diff(qsl) >= 0) and qsl[0] == 0 and qsl[-1] == sum(nst)
    assert np.array_equal(out["logits_indices"], qsl[1:] - 1)
    for r in range(len(nst)):
        s = out["slot_mapping"][qsl[r]:qsl[r + 1]]
        assert len(set(s.tolist())) == len(s)               # distinct within a request
        assert set((s // bs).tolist()) <= set(bt[r].tolist())  # inside its own blocks


def test_prep_brute_force_exhaustive_small():
    rng = np.random.default_rng(7)
    count = 0
    for bs in (4, 16):
        for r in (1, 2, 3):
            for nst in itertools.product(range(1, 6), repeat=r):
                nct = rng.integers(0, 41, size=r)
                bt = _table_for(nst, nct, bs, 64, rng)
                out = oracle.prepare_inputs(nst, nct, bt, bs, sum(nst), 64)
                ref = brute_prepare(nst, nct, bt, bs)
                for k, v in ref.items():
                    assert out[k].tolist() == v, (k, nst, nct)
                _check_invariants(nst, nct, bt, bs, out)
                count += 1
    assert count > 300


def test_prep_brute_force_random():
    rng = np.random.default_rng(11)
    for _ in range(300):
        r = int(rng.integers(1, 9))
        nst = rng.integers(1, 40, size=r)
        nct = rng.integers(0, 500, size=r)
        bs = int(rng.choice([1, 2, 4, 8, 16, 32]))
        nb = sum(-(-(int(a) + int(b)) // bs) for a, b in zip(nst, nct)) + 3
        bt = _table_for(nst, nct, bs, nb, rng)
        out = oracle.prepare_inputs(nst, nct, bt, bs, int(nst.sum()), nb)
        ref = brute_prepare(nst, nct, bt, bs)
        for k, v in ref.items():
            assert out[k].tolist() == v, k
        _check_invariants(nst, nct, bt, bs, out)


@pytest.mark.parametrize("bad", ["zero_tokens", "total_mismatch", "block_oob",
                                 "logical_oob", "negative_block"])
def test_prep_rejects_bad_inputs(bad):
    nst, nct, bt, t, nb = [2, 3], [5, 0], [[0, 1], [2, -1]], 5, 4
    if bad == "zero_tokens":
        nst, t = [0, 3], 3
    elif bad == "total_mismatch":
        t = 6
    elif bad == "block_oob":
        bt = [[0, 1], [4, -1]]
    elif bad == "logical_oob":
        nct = [40, 0]           # position 40 is logical block 2 of a 2-wide table
    elif bad == "negative_block":
        bt = [[0, 1], [-1, -1]]
    out = oracle.prepare_inputs(nst, nct, bt, 16, t, nb, check=False)
    assert out["status"] != 0


# ---------------------------------------------------------------------------
# Input ids, discard mask, sampled rows
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("m", [8, 16, 1000, 131072])
def test_token_indices_printed_comment(m):
    g = golden("prep_token_indices_comment.json")
    i = g["inputs"]
    # Every entry of the buffer holds its own flat offset, so the gathered
    # id equals the offset the page prints.
    ids = np.arange(3 * m, dtype=np.int64).astype(np.int32).reshape(3, m)
    tok, inp, st = oracle.gather_input_ids(i["req_indices"], i["positions"], ids)
    want = [a * m + b for a, b in g["printed"]["token_indices_as_multiple_of_M_plus_offset"]]
    assert st == 0
    assert tok.tolist() == want
    assert inp.tolist() == want


def test_token_indices_from_oracle_prep_positions():
    # The same comment, with req_indices / positions produced by the index build.
    g = golden("prep_token_indices_comment.json")
    i = g["inputs"]
    out = oracle.prepare_inputs(i["num_scheduled_tokens"], i["num_computed_tokens"],
                                [[0], [1], [2]], 16, 10, 3)
    assert out["positions"].tolist() == i["positions"]
    assert out["req_indices"].tolist() == i["req_indices"]


def _go_token_buffer(width):
    g = golden("prep_go_program_bs4.json")
    rows = np.full((4, width), -5, np.int32)      # a spare fourth row, unused
    for r, name in enumerate("ABC"):
        base, n = g["inputs"]["token_ids_rows"][name]
        rows[r, :n] = np.arange(base, base + n)
    return g, rows


@pytest.mark.parametrize("width", [20, 64])
def test_input_ids_go_program(width):
    g, rows = _go_token_buffer(width)
    i = g["inputs"]
    out = oracle.prepare_inputs(i["num_scheduled_tokens"], i["num_computed_tokens"],
                                i["block_table"], i["block_size"], 9, i["num_blocks"])
    tok, inp, st = oracle.gather_input_ids(out["req_indices"], out["positions"], rows)
    assert st == 0
    assert inp.tolist() == g["derived_by_hand"]["input_ids"]
    assert np.array_equal(tok // width, out["req_indices"])
    assert np.array_equal(tok % width, out["positions"])


def test_input_ids_brute_force_two_dimensional_lookup():
    rng = np.random.default_rng(21)
    for _ in range(200):
        rows_n = int(rng.integers(1, 7))
        width = int(rng.integers(1, 50))
        ids = rng.integers(0, 2**31 - 1, size=(rows_n, width)).astype(np.int32)
        t = int(rng.integers(0, 40))
        req = rng.integers(0, rows_n, size=t)
        pos = rng.integers(0, width, size=t)
        tok, inp, st = oracle.gather_input_ids(req, pos, ids)
        assert st == 0
        assert inp.tolist() == [int(ids[a][b]) for a, b in zip(req, pos)]
        assert tok.tolist() == [int(a) * width + int(b) for a, b in zip(req, pos)]


@pytest.mark.parametrize("bad", ["position_past_row", "row_past_buffer", "negative"])
def test_input_ids_rejects_offsets_outside_own_row(bad):
    ids = np.arange(12, dtype=np.int32).reshape(3, 4)
    req, pos = [0, 1, 2], [1, 2, 3]
    if bad == "position_past_row":
        pos = [1, 4, 3]          # would read row 2's first id
    elif bad == "row_past_buffer":
        req = [0, 3, 2]
    else:
        pos = [1, -1, 3]
    tok, inp, st = oracle.gather_input_ids(req, pos, ids, check=False)
    assert st != 0
    assert tok[1] == -1 and inp[1] == -1
    assert inp[0] == 1 and inp[2] == 11


def test_discard_mask_printed_2_5_3():
    g = golden("prep_worked_example_2_5_3.json")
    i = g["inputs"]
    m = oracle.discard_request_mask(i["num_computed_tokens"], i["num_scheduled_tokens"],
                                    i["request_num_tokens"])
    assert m.tolist() == g["printed"]["discard_request_mask"]


def test_discard_mask_go_program():
    g = golden("prep_go_program_bs4.json")
    i, h = g["inputs"], g["derived_by_hand"]
    m = oracle.discard_request_mask(i["num_computed_tokens"], i["num_scheduled_tokens"],
                                    h["request_num_tokens"])
    assert m.tolist() == h["discard_request_mask"]


def test_discard_mask_boundaries():
    # caught up exactly -> sampled; one short -> discarded; decode (1 token,
    # total already known) -> sampled
    m = oracle.discard_request_mask([9, 9, 41, 0], [1, 1, 1, 16], [10, 11, 42, 17])
    assert m.tolist() == [False, True, False, True]


def test_spec_logits_no_drafts_is_printed_rows():
    g = golden("prep_worked_example_2_5_3.json")
    qsl = g["printed"]["query_start_loc"]
    for drafts in (None, [0, 0, 0]):
        rows, cu, st = oracle.spec_logits_indices(qsl, drafts)
        assert st == 0
        assert rows.tolist() == g["printed"]["logits_indices"]
        assert cu.tolist() == [0, 1, 2, 3]


def test_spec_logits_draft_invariants():
    rng = np.random.default_rng(5)
    for _ in range(300):
        r = int(rng.integers(1, 10))
        nst = rng.integers(1, 9, size=r)
        d = np.array([int(rng.integers(0, n)) for n in nst])
        qsl = np.concatenate([[0], np.cumsum(nst)])
        rows, cu, st = oracle.spec_logits_indices(qsl, d)
        assert st == 0
        assert len(rows) == r + d.sum()                    # one per draft plus one
        assert cu[0] == 0 and np.array_equal(np.diff(cu), d + 1)
        for q in range(r):
            mine = rows[cu[q]:cu[q + 1]]
            assert np.array_equal(np.diff(mine), np.ones(d[q], np.int32))  # consecutive
            assert mine[-1] == qsl[q + 1] - 1                # ends on the slice's last row
            assert mine[0] >= qsl[q]                         # stays in its own slice


def test_spec_logits_decode_with_drafts_example():
    # Two decoding requests verifying 2 and 0 drafts, one prefill chunk:
    # scheduled [3, 1, 4] -> slices [0,3) [3,4) [4,8); rows: 0,1,2 | 3 | 7.
    rows, cu, st = oracle.spec_logits_indices([0, 3, 4, 8], [2, 0, 0])
    assert st == 0 and rows.tolist() == [0, 1, 2, 3, 7] and cu.tolist() == [0, 3, 4, 5]


@pytest.mark.parametrize("bad", ["too_many_drafts", "negative", "count_mismatch"])
def test_spec_logits_rejects(bad):
    qsl, d, n = [0, 3, 4], [2, 0], None
    if bad == "too_many_drafts":
        d = [3, 0]              # 4 rows from a 3-token slice
    elif bad == "negative":
        d = [-1, 0]
    else:
        n = 3
    rows, cu, st = oracle.spec_logits_indices(qsl, d, n, check=False)
    assert st != 0


# ---------------------------------------------------------------------------
# Whole-block operations: copy-on-write copy and zeroing
# ---------------------------------------------------------------------------

def _pools(seed, nb=12, bs=4, hkv=2, d=8, dtype=np.uint16):
    rng = np.random.default_rng(seed)
    k = rng.integers(0, 2**16, size=(nb, bs, hkv, d)).astype(dtype)
    v = rng.integers(0, 2**16, size=(nb, bs, hkv, d)).astype(dtype)
    return k, v


@pytest.mark.parametrize("dtype", [np.uint16, np.uint8])
def test_copy_blocks_equals_numpy_block_slicing(dtype):
    for seed in range(20):
        k, v = _pools(seed, dtype=dtype)
        rng = np.random.default_rng(100 + seed)
        n = int(rng.integers(0, 6))
        blocks = rng.permutation(k.shape[0])
        src, dst = blocks[:n], blocks[n:2 * n]          # fresh destinations
        kb, vb, st = oracle.copy_blocks(k, v, src, dst)
        assert st == 0
        ke, ve = k.copy(), v.copy()
        ke[dst] = k[src]
        ve[dst] = v[src]
        np.testing.assert_array_equal(kb.view(dtype).reshape(k.shape), ke)
        np.testing.assert_array_equal(vb.view(dtype).reshape(v.shape), ve)


def test_copy_blocks_one_source_many_beams():
    # four beams fork from one shared block: each gets its own copy
    k, v = _pools(3)
    kb, vb, st = oracle.copy_blocks(k, v, [5, 5, 5, 5], [0, 1, 2, 3])
    assert st == 0
    kb = kb.view(np.uint16).reshape(k.shape)
    vb = vb.view(np.uint16).reshape(v.shape)
    for b in range(4):
        np.testing.assert_array_equal(kb[b], k[5])
        np.testing.assert_array_equal(vb[b], v[5])
    np.testing.assert_array_equal(kb[4:], k[4:])


def test_copy_blocks_skips_pairs_outside_the_pool():
    k, v = _pools(4)
    kb, vb, st = oracle.copy_blocks(k, v, [1, 12, -1, 2], [3, 4, 5, 6], check=False)
    assert st != 0
    kb = kb.view(np.uint16).reshape(k.shape)
    np.testing.assert_array_equal(kb[3], k[1])
    np.testing.assert_array_equal(kb[6], k[2])
    np.testing.assert_array_equal(kb[4], k[4])          # skipped pairs leave dst alone
    np.testing.assert_array_equal(kb[5], k[5])


def test_zero_blocks_clears_exactly_those_blocks():
    for dtype in (np.uint16, np.uint8):
        k, v = _pools(5, dtype=dtype)
        ids = [7, 0, 11]
        kb, vb, st = oracle.zero_blocks(k, v, ids)
        assert st == 0
        kb, vb = kb.view(dtype).reshape(k.shape), vb.view(dtype).reshape(v.shape)
        keep = [b for b in range(k.shape[0]) if b not in ids]
        assert not kb[ids].any() and not vb[ids].any()
        np.testing.assert_array_equal(kb[keep], k[keep])
        np.testing.assert_array_equal(vb[keep], v[keep])
    # zero bytes decode as +0.0 in bf16 and fp16
    z = np.zeros(4, np.uint16)
    assert (from_bits(z, torch.bfloat16) == 0).all() and (z.view(np.float16) == 0).all()
    k, v = _pools(6)
    _, _, st = oracle.zero_blocks(k, v, [3, 12], check=False)
    assert st != 0


def test_beam_fork_copy_on_write_scenario():
    # Two beams share blocks [a, b]; b holds 2 of its 4 slots.  Beam 1 writes
    # its next token: b is shared, so b is copied to a new block c, beam 1's
    # table is remapped to [a, c], and the token goes to c ("How vLLM Works
    # Internally", Copy-on-Write for Beam Search, steps 1-5).
    rng = np.random.default_rng(8)
    bs, hkv, hq, d, nb = 4, 1, 2, 8, 6
    k = from_bits(rng.integers(0, 2**16, size=(nb, bs, hkv, d)).astype(np.uint16) & 0x3FFF,
                  torch.bfloat16)
    v = from_bits(rng.integers(0, 2**16, size=(nb, bs, hkv, d)).astype(np.uint16) & 0x3FFF,
                  torch.bfloat16)
    a, b, c = 2, 4, 1
    shared = np.array([[a, b], [a, b]], np.int32)
    q = torch.randn(1, hq, d).to(torch.bfloat16).repeat(2, 1, 1)   # both beams ask the same
    # before the fork both beams see the same 6 tokens
    before = oracle.attention(q, k, v, shared, [0, 1, 2], [6, 6], hq, hkv, d, bs, nb, 0.3,
                              "bf16")
    np.testing.assert_array_equal(before[0], before[1])
    kb, vb, st = oracle.copy_blocks(k, v, [b], [c])
    assert st == 0
    kc = from_bits(kb.view(np.uint16).reshape(k.shape), torch.bfloat16)
    vc = from_bits(vb.view(np.uint16).reshape(v.shape), torch.bfloat16)
    forked = np.array([[a, b], [a, c]], np.int32)
    # the copy changes nothing either beam sees
    after = oracle.attention(q, kc, vc, forked, [0, 1, 2], [6, 6], hq, hkv, d, bs, nb, 0.3,
                             "bf16")
    np.testing.assert_array_equal(after, before)
    # beam 1's new token lands in c (slot c*bs + 2) and beam 0 does not see it
    newk = torch.randn(1, hkv, d).to(torch.bfloat16) * 4
    newv = torch.randn(1, hkv, d).to(torch.bfloat16) * 4
    k2, v2, _ = oracle.cache_write(newk, newv, kc, vc, [c * bs + 2], hkv, d, bs, nb)
    k2, v2 = from_bits(k2, torch.bfloat16), from_bits(v2, torch.bfloat16)
    grown = oracle.attention(q, k2, v2, forked, [0, 1, 2], [6, 7], hq, hkv, d, bs, nb, 0.3,
                             "bf16")
    np.testing.assert_array_equal(grown[0], before[0])
    assert not np.array_equal(grown[1], before[1])
    # and beam 1 over [a, c] equals dense attention over its 7 tokens
    keys = torch.cat([k2[a], k2[c][:3]]).double().numpy()
    vals = torch.cat([v2[a], v2[c][:3]]).double().numpy()
    for h in range(hq):
        sc = 0.3 * keys[:, 0, :] @ q[1, h].double().numpy()
        w = np.exp(sc - sc.max())
        np.testing.assert_allclose(grown[1, h], (w / w.sum()) @ vals[:, 0, :], atol=1e-12)


# ---------------------------------------------------------------------------
# FP8 (E4M3) cache
# ---------------------------------------------------------------------------

def _torch_e4m3(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn)


def test_e4m3_decode_every_code_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    want = _torch_e4m3(codes).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert nan.tolist() == np.isnan(got).tolist() and nan.sum() == 2     # 0x7f, 0xff
    np.testing.assert_array_equal(got[~nan], want[~nan])
    np.testing.assert_array_equal(np.signbit(got[~nan]), codes[~nan] >= 0x80)


def test_e4m3_closed_forms():
    got = oracle.e4m3_decode([0x7E, 0x08, 0x07, 0x01, 0x38, 0xC0, 0x00, 0x77])
    assert got.tolist() == [448.0, 2.0 ** -6, 7 * 2.0 ** -9, 2.0 ** -9, 1.0, -2.0, 0.0, 240.0]


def test_e4m3_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(vals), codes)


def test_e4m3_encode_matches_torch_inside_the_finite_range():
    rng = np.random.default_rng(13)
    mag = np.exp2(rng.uniform(-14, np.log2(463.9), size=200_000)).astype(np.float32)
    x = np.where(rng.random(mag.size) < 0.5, -mag, mag).astype(np.float32)
    # and every midpoint between neighbouring finite codes (the ties)
    pos = np.sort(oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, [0.0, -0.0]]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(x), want)


def test_e4m3_ties_go_to_the_even_code():
    pos = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    got = oracle.e4m3_encode(mids)
    assert np.all(got % 2 == 0)                     # even mantissa
    assert np.all((got == np.arange(0, 0x7E)) | (got == np.arange(1, 0x7F)))


def test_e4m3_encode_saturates_and_keeps_nan():
    got = oracle.e4m3_encode([448.0, 463.99, 464.0, 1e30, np.inf, -500.0, -np.inf, np.nan])
    assert got[:7].tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert got[7] & 0x7F == 0x7F


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_cache_write_fp8_matches_torch_division_and_rounding(dtype):
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    rng = np.random.default_rng(3)
    t, hkv, d, bs, nb = 9, 2, 16, 4, 6
    key = torch.randn(t, hkv, d).to(tdt)
    value = (torch.randn(t, hkv, d) * 3).to(tdt)
    slots = rng.permutation(nb * bs)[:t].astype(np.int32)
    slots[4] = -1                                     # a padding row: no write
    kc0 = rng.integers(0, 256, size=(nb, bs, hkv, d)).astype(np.uint8)
    vc0 = rng.integers(0, 256, size=(nb, bs, hkv, d)).astype(np.uint8)
    ks, vs = 0.0625, 0.3
    kc, vc, st = oracle.cache_write_fp8(key, value, kc0, vc0, slots, hkv, d, bs, nb, dtype, ks,
                                        vs)
    assert st == 0
    kq = (key.float() / torch.tensor(ks, dtype=torch.float32)).to(torch.float8_e4m3fn)
    vq = (value.float() / torch.tensor(vs, dtype=torch.float32)).to(torch.float8_e4m3fn)
    flat_k = kc.reshape(nb * bs, hkv, d)
    flat_v = vc.reshape(nb * bs, hkv, d)
    written = slots >= 0
    np.testing.assert_array_equal(flat_k[slots[written]], kq.view(torch.uint8).numpy()[written])
    np.testing.assert_array_equal(flat_v[slots[written]], vq.view(torch.uint8).numpy()[written])
    untouched = np.setdiff1d(np.arange(nb * bs), slots[written])
    np.testing.assert_array_equal(flat_k[untouched], kc0.reshape(nb * bs, hkv, d)[untouched])


def test_attention_over_fp8_pools_equals_16_bit_pools_of_the_same_values():
    rng = np.random.default_rng(17)
    nb, bs, hkv, hq, d = 12, 4, 2, 4, 16
    def pool():
        x = torch.randn(nb, bs, hkv, d) * 12
        return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    k8, v8 = pool(), pool()
    ks, vs = 2.0 ** -4, 2.0 ** -3                     # powers of two: exact in bf16
    kb = (_torch_e4m3(k8).float() * ks).to(torch.bfloat16)
    vb = (_torch_e4m3(v8).float() * vs).to(torch.bfloat16)
    assert torch.equal(kb.double(), torch.from_numpy(oracle.e4m3_decode(k8) * ks))
    bt = rng.permutation(nb)[:9].astype(np.int32).reshape(3, 3)
    nst, sl = [3, 1, 2], [9, 12, 5]
    qsl = np.concatenate([[0], np.cumsum(nst)]).astype(np.int32)
    q = torch.randn(6, hq, d).to(torch.bfloat16)
    got = oracle.attention(q, k8, v8, bt, qsl, sl, hq, hkv, d, bs, nb, 0.25, "bf16",
                           kv_cache_dtype="fp8_e4m3", k_scale=ks, v_scale=vs)
    want = oracle.attention(q, kb, vb, bt, qsl, sl, hq, hkv, d, bs, nb, 0.25, "bf16")
    np.testing.assert_array_equal(got, want)
    # a scale on V scales the output; a scale on K acts like a softmax scale
    got2 = oracle.attention(q, k8, v8, bt, qsl, sl, hq, hkv, d, bs, nb, 0.25 * ks, "bf16",
                            kv_cache_dtype="fp8_e4m3", k_scale=1.0, v_scale=1.0)
    np.testing.assert_allclose(got2 * vs, want, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# Cache write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_cache_write_bit_exact_and_untouched(dtype):
    rng = np.random.default_rng(3)
    nb, bs, hkv, d, t = 12, 16, 3, 8, 20
    slots = rng.choice(nb * bs, size=t, replace=False).astype(np.int32)
    slots[4] = -1                                   # a padding row writes nothing
    key = torch.randn(t, hkv, d).to(dtype)
    value = torch.randn(t, hkv, d).to(dtype)
    sentinel = np.full((nb, bs, hkv, d), 0x7FC1, np.uint16)     # a NaN pattern
    kc, vc, rc = oracle.cache_write(key, value, sentinel, sentinel.copy(), slots, hkv, d, bs, nb)
    assert rc == 0
    kb, vb = to_bits(key), to_bits(value)
    kflat, vflat = kc.reshape(nb * bs, hkv, d), vc.reshape(nb * bs, hkv, d)
    written = set()
    for i, s in enumerate(slots):
        if s < 0:
            continue
        written.add(int(s))
        assert np.array_equal(kflat[s], kb[i]) and np.array_equal(vflat[s], vb[i])
    for s in range(nb * bs):
        if s not in written:
            assert np.all(kflat[s] == 0x7FC1) and np.all(vflat[s] == 0x7FC1)


def test_cache_write_strided_source_and_roundtrip():
    rng = np.random.default_rng(5)
    nb, bs, hkv, d, t, hq = 8, 16, 2, 16, 30, 6
    qkv = torch.randn(t, (hq + 2 * hkv) * d).to(torch.bfloat16)
    stride = (hq + 2 * hkv) * d
    kbits = to_bits(qkv).reshape(-1)[hq * d:]
    vbits = to_bits(qkv).reshape(-1)[(hq + hkv) * d:]
    slots = rng.choice(nb * bs, size=t, replace=False).astype(np.int32)
    pool = np.zeros((nb, bs, hkv, d), np.uint16)
    kc, vc, rc = oracle.cache_write(kbits, vbits, pool, pool.copy(), slots, hkv, d, bs, nb,
                                    kv_token_stride=stride)
    assert rc == 0
    # gather back by slot_mapping == the K/V slices of the fused rows
    full = to_bits(qkv)
    kflat, vflat = kc.reshape(-1, hkv, d), vc.reshape(-1, hkv, d)
    for i, s in enumerate(slots):
        assert np.array_equal(kflat[s].reshape(-1), full[i, hq * d:(hq + hkv) * d])
        assert np.array_equal(vflat[s].reshape(-1), full[i, (hq + hkv) * d:])


def test_cache_write_rejects_slot_out_of_pool():
    key = torch.zeros(2, 1, 8, dtype=torch.bfloat16)
    pool = np.zeros((2, 4, 1, 8), np.uint16)
    _, _, rc = oracle.cache_write(key, key, pool, pool.copy(), [0, 8], 1, 8, 4, 2, check=False)
    assert rc != 0


# ---------------------------------------------------------------------------
# Attention: closed forms
# ---------------------------------------------------------------------------

def _run_attn(q, kc, vc, bt, nst, nct, bs, scale, dtype="bf16"):
    qsl = np.concatenate([[0], np.cumsum(nst)]).astype(np.int32)
    sl = (np.asarray(nct) + np.asarray(nst)).astype(np.int32)
    hq, d = q.shape[1], q.shape[2]
    hkv = kc.shape[2]
    return oracle.attention(q, kc, vc, bt, qsl, sl, hq, hkv, d, bs, kc.shape[0], scale, dtype)


def _rand_case(seed, nst, nct, hq=4, hkv=2, d=16, bs=4, dtype=torch.bfloat16):
    rng = np.random.default_rng(seed)
    torch.manual_seed(seed)
    ctx = [int(a) + int(b) for a, b in zip(nst, nct)]
    ks = [torch.randn(l, hkv, d).to(dtype) for l in ctx]
    vs = [torch.randn(l, hkv, d).to(dtype) for l in ctx]
    nb = sum(-(-l // bs) for l in ctx) + 5
    kc, vc, bt = scatter_to_pool(ks, vs, ctx, bs, nb, rng, dtype)
    q = torch.randn(sum(nst), hq, d).to(dtype)
    return q, kc, vc, bt, ks, vs


def test_attention_single_visible_key_is_v():
    # A fresh request's first token (position 0) sees only key 0: o = v_0.
    q, kc, vc, bt, ks, vs = _rand_case(1, [3, 1], [0, 0])
    out = _run_attn(q, kc, vc, bt, [3, 1], [0, 0], 4, 0.25)
    for t, r in ((0, 0), (3, 1)):
        for h in range(4):
            np.testing.assert_array_equal(out[t, h], vs[r][0, h // 2].double().numpy())


def test_attention_zero_keys_average_values():
    q, kc, vc, bt, ks, vs = _rand_case(2, [4, 1], [6, 20])
    kc.zero_()
    out = _run_attn(q, kc, vc, bt, [4, 1], [6, 20], 4, 0.25)
    for r, (t0, n, c) in enumerate(((0, 4, 6), (4, 1, 20))):
        for i in range(n):
            p = c + i
            mean = vs[r][: p + 1].double().mean(0).numpy()
            for h in range(4):
                np.testing.assert_allclose(out[t0 + i, h], mean[h // 2], rtol=0, atol=1e-14)


def test_attention_constant_values():
    q, kc, vc, bt, ks, vs = _rand_case(3, [5, 2], [9, 33])
    vc.fill_(-1.5)
    out = _run_attn(q, kc, vc, bt, [5, 2], [9, 33], 4, 0.25)
    np.testing.assert_allclose(out, -1.5, rtol=0, atol=1e-14)


def test_attention_one_dominant_key():
    # Key 5 of request 0 is 40 * q (per head group): its score dwarfs the rest,
    # so o is v_5 to within exp(-large).
    q, kc, vc, bt, ks, vs = _rand_case(4, [1], [11], hq=2, hkv=2, d=16)
    for g in range(2):
        kc[bt[0][5 // 4], 5 % 4, g] = (q[0, g].float() * 40).to(torch.bfloat16)
    out = _run_attn(q, kc, vc, bt, [1], [11], 4, 1.0)
    for h in range(2):
        np.testing.assert_allclose(out[0, h], vs[0][5, h].double().numpy(), atol=1e-9)


def test_attention_fp16_decoding_every_pattern():
    # One visible key: o must equal v exactly, for every finite fp16 pattern.
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = pats[((pats >> 10) & 0x1F) != 0x1F]
    d = 64
    n = finite.size // d
    v = finite[: n * d].reshape(n, 1, 1, d)
    vc = np.zeros((n, 1, 1, d), np.uint16)
    vc[:, 0] = v[:, 0]
    kc = np.zeros_like(vc)
    q = np.zeros((n, 1, d), np.uint16)
    bt = np.arange(n, dtype=np.int32).reshape(n, 1)
    qsl = np.arange(n + 1, dtype=np.int32)
    sl = np.ones(n, np.int32)
    out = oracle.attention(q, kc, vc, bt, qsl, sl, 1, 1, d, 1, n, 1.0, "fp16")
    ref = torch.from_numpy(v.reshape(n, d).view(np.float16).astype(np.float64))
    np.testing.assert_array_equal(out[:, 0, :], ref.numpy())


def test_attention_bf16_decoding_sample():
    rng = np.random.default_rng(9)
    pats = rng.integers(0, 65536, size=64 * 200).astype(np.uint16)
    pats = pats[((pats >> 7) & 0xFF) != 0xFF][: 64 * 150]
    n, d = 150, 64
    vc = pats.reshape(n, 1, 1, d)
    out = oracle.attention(np.zeros((n, 1, d), np.uint16), np.zeros_like(vc), vc,
                           np.arange(n, dtype=np.int32).reshape(n, 1),
                           np.arange(n + 1, dtype=np.int32), np.ones(n, np.int32),
                           1, 1, d, 1, n, 1.0, "bf16")
    ref = from_bits(pats.reshape(n, d), torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(out[:, 0, :], ref)


# ---------------------------------------------------------------------------
# Attention: brute force, dense reference, invariances
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_attention_brute_force_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    r = int(rng.integers(1, 4))
    nst = [int(x) for x in rng.integers(1, 5, size=r)]
    nct = [int(x) for x in rng.integers(0, 10, size=r)]
    hkv = int(rng.choice([1, 2]))
    hq = hkv * int(rng.choice([1, 2, 3]))
    dt = torch.bfloat16 if seed % 2 else torch.float16
    q, kc, vc, bt, _, _ = _rand_case(seed, nst, nct, hq=hq, hkv=hkv, d=8, bs=4, dtype=dt)
    out = _run_attn(q, kc, vc, bt, nst, nct, 4, 0.3, "bf16" if seed % 2 else "fp16")
    qsl = [0] + list(np.cumsum(nst))
    ref = brute_attention(q.double().numpy(), kc.double().numpy(), vc.double().numpy(), bt,
                          qsl, [a + b for a, b in zip(nst, nct)], 4, 0.3)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_attention_paged_equals_dense_contiguous(seed):
    nst, nct = [7, 1, 12, 1], [0, 40, 19, 63]
    q, kc, vc, bt, ks, vs = _rand_case(20 + seed, nst, nct, hq=8, hkv=2, d=32, bs=16)
    out = _run_attn(q, kc, vc, bt, nst, nct, 16, 1 / math.sqrt(32))
    t0 = 0
    for r, (n, c) in enumerate(zip(nst, nct)):
        ref = dense_causal_numpy(q[t0:t0 + n].double().numpy(), ks[r].double().numpy(),
                                 vs[r].double().numpy(), c, 1 / math.sqrt(32))
        np.testing.assert_allclose(out[t0:t0 + n], ref, rtol=0, atol=1e-12)
        t0 += n


def test_attention_physical_block_permutation_invariant():
    w = workloads.random_case(5, max_reqs=4, head_dim=64)
    v = workloads.make_values(w, 5)
    idx, kc, vc, out = oracle.step(w, v)
    rng = np.random.default_rng(6)
    perm = rng.permutation(w.num_blocks)          # new id of old block b is perm[b]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1)
    out2 = oracle.attention(v["q"], kc2, vc2, bt2, idx["query_start_loc"], idx["seq_lens"],
                            w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                            w.num_blocks, w.scale, w.dtype)
    np.testing.assert_array_equal(out, out2)


def test_attention_request_order_shuffle_invariant():
    nst, nct = [3, 1, 6], [5, 30, 0]
    q, kc, vc, bt, _, _ = _rand_case(31, nst, nct, hq=4, hkv=2, d=16, bs=16)
    out = _run_attn(q, kc, vc, bt, nst, nct, 16, 0.25)
    order = [2, 0, 1]
    qsl = [0, 3, 4, 10]
    q2 = torch.cat([q[qsl[r]:qsl[r + 1]] for r in order])
    out2 = _run_attn(q2, kc, vc, bt[order], [nst[r] for r in order], [nct[r] for r in order],
                     16, 0.25)
    back = np.concatenate([out[qsl[r]:qsl[r + 1]] for r in order])
    np.testing.assert_array_equal(out2, back)


def test_attention_gqa_equals_replicated_mha():
    nst, nct = [4, 1], [3, 17]
    q, kc, vc, bt, _, _ = _rand_case(41, nst, nct, hq=6, hkv=2, d=16, bs=4)
    out = _run_attn(q, kc, vc, bt, nst, nct, 4, 0.25)
    kc6 = kc.repeat_interleave(3, dim=2)
    vc6 = vc.repeat_interleave(3, dim=2)
    out6 = _run_attn(q, kc6, vc6, bt, nst, nct, 4, 0.25)
    np.testing.assert_array_equal(out, out6)


def test_attention_chunk_equals_tail_of_full_prefill():
    # A chunk at num_computed = c with n tokens is the last n rows of a full
    # prefill of c + n tokens over the same keys and values.
    c, n = 37, 11
    q, kc, vc, bt, _, _ = _rand_case(51, [c + n], [0], hq=4, hkv=1, d=16, bs=16)
    full = _run_attn(q, kc, vc, bt, [c + n], [0], 16, 0.25)
    chunk = _run_attn(q[c:], kc, vc, bt, [n], [c], 16, 0.25)
    np.testing.assert_array_equal(chunk, full[c:])


def test_attention_token_subset_matches_full():
    w = workloads.random_case(8, max_reqs=5)
    v = workloads.make_values(w, 8)
    idx, kc, vc, full = oracle.step(w, v)
    sel = np.arange(0, w.num_tokens, 3)
    part = oracle.attention(v["q"], kc, vc, w.block_table, idx["query_start_loc"],
                            idx["seq_lens"], w.num_q_heads, w.num_kv_heads, w.head_dim,
                            w.block_size, w.num_blocks, w.scale, w.dtype, tokens=sel)
    np.testing.assert_array_equal(part[sel], full[sel])
    rest = np.setdiff1d(np.arange(w.num_tokens), sel)
    assert np.isnan(part[rest]).all()


def test_attention_threads_do_not_change_result():
    w = workloads.random_case(9, max_reqs=6, long_prefill=70)
    v = workloads.make_values(w, 9)
    _, _, _, a = oracle.step(w, v, num_threads=1)
    _, _, _, b = oracle.step(w, v, num_threads=4)
    np.testing.assert_array_equal(a, b)


def test_step_write_then_read_sees_new_tokens():
    # Write-before-read: each token's own key is visible to it.  Make the new
    # tokens' values constant 2.0 and every older value 0: a token at position
    # p of a request with c computed sees (p - c + 1) new values out of p + 1.
    w = workloads.random_case(12, max_reqs=4, head_dim=64, dtype="fp16")
    v = workloads.make_values(w, 12)
    v["value"].fill_(2.0)
    v["value_cache"].zero_()
    v["key"].zero_()
    v["key_cache"].zero_()
    idx, _, _, out = oracle.step(w, v)
    for t in range(w.num_tokens):
        r = idx["req_indices"][t]
        p = idx["positions"][t]
        c = w.num_computed_tokens[r]
        np.testing.assert_allclose(out[t], 2.0 * (p - c + 1) / (p + 1), atol=1e-14)
