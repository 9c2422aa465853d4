"""The rest of input preparation on the GPU (token-id gather, discard mask,
sampled rows with drafts) vs. the oracle, through the C ABI.  Every output
is integer work and must match bit for bit."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prepare_gb300 as pa
import workloads
from gpu_step import to_dev
from helpers import golden

pytestmark = pytest.mark.gpu

BASE_KEYS = ("req_indices", "positions", "slot_mapping", "query_start_loc", "seq_lens")


@pytest.fixture(autouse=True)
def clean_status():
    pa.pa_get_status()
    yield


def _run_ex(nst, nct, bt, bs, t, nb, *, ids=None, totals=None, drafts=None, qsl_cap=None,
            pinned=False, with_cu=True):
    """One pa_prepare_inputs_ex call; returns host copies and the status."""
    i32 = torch.int32
    r = len(nst)
    cap = r + 1 if qsl_cap is None else qsl_cap
    n_log = r + (int(np.sum(drafts)) if drafts is not None else 0)
    out = {k: torch.full((t,), -7, dtype=i32, device="cuda")
           for k in ("req_indices", "positions", "slot_mapping")}
    out["query_start_loc"] = torch.full((cap,), -7, dtype=i32, device="cuda")
    out["seq_lens"] = torch.full((r,), -7, dtype=i32, device="cuda")
    out["logits_indices"] = torch.full((n_log,), -7, dtype=i32, device="cuda")
    out["cu_num_logits"] = torch.full((r + 1,), -7, dtype=i32, device="cuda") if with_cu else None
    tok = None
    if ids is not None:
        tok = torch.from_numpy(np.ascontiguousarray(ids))
        tok = tok.pin_memory() if pinned else tok.cuda()
        out["token_indices"] = torch.full((t,), -7, dtype=torch.int64, device="cuda")
        out["input_ids"] = torch.full((t,), -7, dtype=i32, device="cuda")
    if totals is not None:
        out["discard_request_mask"] = torch.full((r,), 7, dtype=torch.uint8, device="cuda")
    bt = np.asarray(bt, np.int32).reshape(r, -1) if r else np.zeros((0, 1), np.int32)
    pa.pa_prepare_inputs_ex(
        to_dev(np.asarray(nst, np.int32)), to_dev(np.asarray(nct, np.int32)), to_dev(bt), bs, t,
        nb, out["req_indices"], out["positions"], out["slot_mapping"], out["query_start_loc"],
        out["seq_lens"], out["logits_indices"], token_ids=tok,
        token_indices=out.get("token_indices"), input_ids=out.get("input_ids"),
        request_num_tokens=None if totals is None else to_dev(np.asarray(totals, np.int32)),
        discard_request_mask=out.get("discard_request_mask"),
        num_draft_tokens=None if drafts is None else to_dev(np.asarray(drafts, np.int32)),
        cu_num_logits=out["cu_num_logits"])
    status, detail = pa.pa_get_status()
    res = {k: v.cpu().numpy() for k, v in out.items() if v is not None}
    res.update(status=status, detail=detail)
    return res


def _oracle_ex(nst, nct, bt, bs, t, nb, *, ids=None, totals=None, drafts=None, qsl_cap=None):
    r = len(nst)
    want = oracle.prepare_inputs(nst, nct, bt, bs, t, nb, qsl_cap)
    if ids is not None:
        want["token_indices"], want["input_ids"], _ = oracle.gather_input_ids(
            want["req_indices"], want["positions"], ids)
    if totals is not None:
        want["discard_request_mask"] = oracle.discard_request_mask(nct, nst, totals).astype(
            np.uint8)
    rows, cu, _ = oracle.spec_logits_indices(want["query_start_loc"][: r + 1], drafts)
    want["logits_indices"], want["cu_num_logits"] = rows, cu
    return want


def _compare(res, want):
    assert res["status"] == pa.PA_OK, pa.check_bits(res["detail"])
    for k, v in want.items():
        if k == "status":
            continue
        np.testing.assert_array_equal(res[k], v, err_msg=k)


# ---------------------------------------------------------------------------
# The pages' worked examples
# ---------------------------------------------------------------------------

def test_discard_mask_and_rows_of_the_2_5_3_example():
    g = golden("prep_worked_example_2_5_3.json")
    i = g["inputs"]
    bt = np.arange(3 * 8, dtype=np.int32).reshape(3, 8)
    res = _run_ex(i["num_scheduled_tokens"], i["num_computed_tokens"], bt, 16, 10, 64,
                  totals=i["request_num_tokens"])
    assert res["status"] == pa.PA_OK
    assert res["discard_request_mask"].astype(bool).tolist() == \
        g["printed"]["discard_request_mask"]
    assert res["logits_indices"].tolist() == g["printed"]["logits_indices"]
    assert res["cu_num_logits"].tolist() == [0, 1, 2, 3]


@pytest.mark.parametrize("pinned", [False, True])
def test_go_program_input_ids_and_verdicts(pinned):
    g = golden("prep_go_program_bs4.json")
    i, h = g["inputs"], g["derived_by_hand"]
    ids = np.full((4, 20), -5, np.int32)
    for r, name in enumerate("ABC"):
        base, n = i["token_ids_rows"][name]
        ids[r, :n] = np.arange(base, base + n)
    res = _run_ex(i["num_scheduled_tokens"], i["num_computed_tokens"], i["block_table"],
                  i["block_size"], 9, i["num_blocks"], ids=ids,
                  totals=h["request_num_tokens"], pinned=pinned)
    assert res["status"] == pa.PA_OK
    assert res["input_ids"].tolist() == h["input_ids"]
    assert res["discard_request_mask"].astype(bool).tolist() == h["discard_request_mask"]
    for k in ("slot_mapping", "positions", "logits_indices"):
        assert res[k].tolist() == h[k], k


@pytest.mark.parametrize("m", [8, 131072])
def test_token_indices_comment(m):
    g = golden("prep_token_indices_comment.json")
    i = g["inputs"]
    ids = np.arange(3 * m, dtype=np.int64).astype(np.int32).reshape(3, m)
    bt = np.arange(3 * ((m + 15) // 16), dtype=np.int32).reshape(3, -1)
    res = _run_ex(i["num_scheduled_tokens"], i["num_computed_tokens"], bt, 16, 10, bt.size,
                  ids=ids)
    want = [a * m + b for a, b in g["printed"]["token_indices_as_multiple_of_M_plus_offset"]]
    assert res["token_indices"].tolist() == want
    assert res["input_ids"].tolist() == want


# ---------------------------------------------------------------------------
# Random batches: several CTAs, thread-owned request runs, ragged tails
# ---------------------------------------------------------------------------

def _random_batch(seed, r, max_new, max_ctx, bs=16):
    rng = np.random.default_rng(seed)
    nst = np.where(rng.random(r) < 0.6, 1, rng.integers(2, max_new + 1, size=r)).astype(np.int32)
    nct = rng.integers(0, max_ctx, size=r).astype(np.int32)
    need = -(-(nct + nst) // bs)
    nb = int(need.sum()) + 5
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((r, int(need.max())), -1, np.int32)
    k = 0
    for q in range(r):
        bt[q, : need[q]] = perm[k:k + need[q]]
        k += need[q]
    return nst, nct, bt, bs, int(nst.sum()), nb


@pytest.mark.parametrize("seed,r", [(0, 1), (1, 3), (2, 31), (3, 200), (4, 1023), (5, 1025),
                                    (6, 2049), (7, 4500)])
@pytest.mark.parametrize("drafted", [False, True])
def test_random_batches_vs_oracle(seed, r, drafted):
    nst, nct, bt, bs, t, nb = _random_batch(seed, r, 24, 3000)
    w = workloads.Workload("rand", nst, nct, bt, nb, bs, 8, 8, 64, "bf16")
    ids = workloads.make_token_buffer(w, seed)
    totals = workloads.make_request_totals(w, seed)
    drafts = workloads.make_draft_counts(w, seed) if drafted else None
    kw = dict(ids=ids, totals=totals, drafts=drafts, qsl_cap=r + 1 + seed)
    _compare(_run_ex(nst, nct, bt, bs, t, nb, **kw), _oracle_ex(nst, nct, bt, bs, t, nb, **kw))


@pytest.mark.parametrize("r", [12_289, 50_000])
def test_many_requests(r):
    # The request starts of every CTA sit in shared memory (up to 200 KB);
    # 50,000 requests is the documented maximum.
    nst, nct, bt, bs, t, nb = _random_batch(r, r, 4, 120)
    kw = dict(totals=workloads.make_request_totals(
        workloads.Workload("many", nst, nct, bt, nb, bs, 8, 8, 64, "bf16"), 3))
    _compare(_run_ex(nst, nct, bt, bs, t, nb, **kw), _oracle_ex(nst, nct, bt, bs, t, nb, **kw))


def test_extended_call_matches_the_plain_call():
    nst, nct, bt, bs, t, nb = _random_batch(9, 700, 30, 2000)
    res = _run_ex(nst, nct, bt, bs, t, nb, with_cu=False)
    outs = [torch.full((n,), -7, dtype=torch.int32, device="cuda")
            for n in (t, t, t, len(nst) + 1, len(nst), len(nst))]
    pa.pa_prepare_inputs(to_dev(nst), to_dev(nct), to_dev(bt), bs, t, nb, *outs)
    for k, o in zip(BASE_KEYS + ("logits_indices",), outs):
        np.testing.assert_array_equal(res[k], o.cpu().numpy(), err_msg=k)


@pytest.mark.parametrize("name", ["decode", "mixed", "shared_prefix"])
@pytest.mark.parametrize("pinned", [False, True])
def test_full_size_workloads(name, pinned):
    w = workloads.named(name)
    ids = workloads.make_token_buffer(w, 1)
    totals = workloads.make_request_totals(w, 1)
    drafts = workloads.make_draft_counts(w, 1)
    args = (w.num_scheduled_tokens, w.num_computed_tokens, w.block_table, w.block_size,
            w.num_tokens, w.num_blocks)
    kw = dict(ids=ids, totals=totals, drafts=drafts)
    _compare(_run_ex(*args, pinned=pinned, **kw), _oracle_ex(*args, **kw))


# ---------------------------------------------------------------------------
# Edge cases and device-side checks
# ---------------------------------------------------------------------------

def test_empty_step():
    res = _run_ex([], [], np.zeros((0, 1), np.int32), 16, 0, 4,
                  ids=np.zeros((2, 16), np.int32), totals=[], drafts=[], qsl_cap=3)
    assert res["status"] == pa.PA_OK
    assert res["query_start_loc"].tolist() == [0, 0, 0]
    assert res["cu_num_logits"].tolist() == [0]


def test_every_request_drafts_its_maximum():
    nst = np.array([1, 2, 5, 8], np.int32)
    nct = np.array([10, 0, 7, 3], np.int32)
    bt = np.arange(4, dtype=np.int32).reshape(4, 1)
    drafts = nst - 1
    res = _run_ex(nst, nct, bt, 16, 16, 4, drafts=drafts)
    assert res["status"] == pa.PA_OK
    assert res["logits_indices"].tolist() == list(range(16))   # every row is sampled
    assert res["cu_num_logits"].tolist() == [0, 1, 3, 8, 16]


def test_position_past_the_token_row_is_flagged():
    nst = np.array([3, 2], np.int32)
    nct = np.array([0, 7], np.int32)           # positions 7, 8 of request 1
    bt = np.array([[0], [1]], np.int32)
    ids = np.arange(16, dtype=np.int32).reshape(2, 8)   # width 8: position 8 is outside
    res = _run_ex(nst, nct, bt, 16, 5, 2, ids=ids)
    assert res["status"] == pa.PA_ERR_DEVICE_CHECK
    assert pa.check_bits(res["detail"]) == {"token_index"}
    assert res["input_ids"].tolist() == [0, 1, 2, 15, -1]
    assert res["token_indices"].tolist() == [0, 1, 2, 15, -1]


@pytest.mark.parametrize("bad", ["too_many", "negative", "count_mismatch"])
def test_draft_counts_are_checked(bad):
    nst = np.array([3, 1], np.int32)
    nct = np.array([0, 4], np.int32)
    bt = np.array([[0], [1]], np.int32)
    drafts = {"too_many": [3, 0], "negative": [-1, 0], "count_mismatch": [1, 0]}[bad]
    r, t = 2, 4
    n_log = 5 if bad == "count_mismatch" else 2 + max(0, sum(drafts))
    out = [torch.full((n,), -7, dtype=torch.int32, device="cuda") for n in (t, t, t, 3, 2)]
    logits = torch.full((n_log,), -7, dtype=torch.int32, device="cuda")
    pa.pa_prepare_inputs_ex(to_dev(nst), to_dev(nct), to_dev(bt), 16, t, 2, *out, logits,
                            num_draft_tokens=to_dev(np.asarray(drafts, np.int32)))
    st, detail = pa.pa_get_status()
    assert st == pa.PA_ERR_DEVICE_CHECK
    assert pa.check_bits(detail) == {"draft_count"}
    assert (logits.cpu().numpy() < t).all()       # nothing past the batch, nothing past n_log
