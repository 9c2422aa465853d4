"""Seeded synthetic workloads for one paged-KV attention step.

This module builds inputs only: how many tokens each request schedules and
has already computed, where each request's cache blocks sit in the pool, and
random Q/K/V values.  It holds none of the step's own arithmetic (the index
build, the cache write, the attention); the CUDA path's tests, the benchmark
and the oracle all take their inputs from here.

Recipe (the same for every named workload):

* Request lengths come from a NumPy PCG64 generator seeded with ``seed``.
  A decode request has one scheduled token and ``num_computed_tokens =
  context - 1``, so its context length includes the new token.
* Physical blocks: a seeded random permutation of the pool; requests take
  their blocks in order from the shuffled list (shared blocks are taken
  once and referenced by several tables).  Table entries past a request's
  last block are -1, so a stray read of one is detectable.
* The pool holds ``ceil(1.1 * blocks needed)`` blocks (the tiny workload:
  exactly 16).
* Values: every element of q, the new tokens' key/value and the whole cache
  pool is N(0, 1) drawn by a seeded ``torch.Generator`` on the requested
  device, rounded to bf16 / fp16 (round to nearest even).
* FP8 pools (the ``*_fp8`` workloads, scales 0.25 for K and 0.125 for V):
  N(0,1) / scale rounded by PyTorch's float8_e4m3fn conversion, so the cached
  values (element * scale) are about N(0,1).
* Request state for the rest of input preparation: a token buffer of random
  ids (vocabulary 128,256), each request's total known token count (caught
  up or mid-prompt, half each) and draft counts for speculative decoding
  (uniform up to 7, never more than scheduled - 1).
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

BLOCK_SIZE = 16

_TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclasses.dataclass
class Workload:
    """One step's shapes and index inputs (host arrays)."""

    name: str
    num_scheduled_tokens: np.ndarray  # int32 [R], tokens each request runs this step
    num_computed_tokens: np.ndarray   # int32 [R], tokens already in the cache
    block_table: np.ndarray           # int32 [R, MB] physical block ids, -1 padded
    num_blocks: int                   # physical blocks in the pool
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                        # "bf16" | "fp16"
    unique_blocks: int = 0            # distinct physical blocks referenced by the tables
    kv_cache_dtype: str = "auto"      # "auto" (the q dtype) | "fp8_e4m3"
    k_scale: float = 1.0              # FP8 pools: cached value = element * scale
    v_scale: float = 1.0

    @property
    def num_reqs(self) -> int:
        return int(self.num_scheduled_tokens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.num_scheduled_tokens.sum())

    @property
    def max_blocks_per_req(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def context_lens(self) -> np.ndarray:
        """Context length each request was drawn with (history + this step)."""
        return (self.num_computed_tokens.astype(np.int64)
                + self.num_scheduled_tokens.astype(np.int64))

    @property
    def max_query_len(self) -> int:
        return int(self.num_scheduled_tokens.max()) if self.num_reqs else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.context_lens.max()) if self.num_reqs else 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPES[self.dtype]

    def kv_read_bytes(self) -> int:
        """Bytes of K and V context every request's attention reads (logical)."""
        elt = 1 if self.kv_cache_dtype == "fp8_e4m3" else 2
        return int(self.context_lens.sum()) * 2 * self.num_kv_heads * self.head_dim * elt

    @property
    def shares_blocks(self) -> bool:
        """Some physical block is referenced by more than one request's
        context (copy-on-write or prefix sharing)."""
        nblk = -(-self.context_lens // self.block_size)
        ids = self.block_table[np.arange(self.block_table.shape[1])[None, :] < nblk[:, None]]
        return np.unique(ids).size < ids.size

    def kv_unique_bytes(self) -> int:
        """Bytes of K and V in the distinct blocks the tables reference."""
        elt = 1 if self.kv_cache_dtype == "fp8_e4m3" else 2
        return (self.unique_blocks * self.block_size * 2 * self.num_kv_heads
                * self.head_dim * elt)


def _blocks_for(context_len: int, block_size: int) -> int:
    return -(-int(context_len) // block_size)


def _pool_size(needed: int) -> int:
    return int(math.ceil(needed * 1.1))


def _tables(rows: list[list[int]], width: int | None = None) -> np.ndarray:
    width = max(len(r) for r in rows) if width is None else width
    bt = np.full((len(rows), max(width, 1)), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        bt[i, : len(r)] = r
    return bt


def _private_tables(rng: np.random.Generator, ctx: np.ndarray, block_size: int,
                    num_blocks: int | None = None):
    need = [_blocks_for(c, block_size) for c in ctx]
    nb = _pool_size(sum(need)) if num_blocks is None else num_blocks
    perm = rng.permutation(nb)
    rows, k = [], 0
    for n in need:
        rows.append([int(b) for b in perm[k : k + n]])
        k += n
    return _tables(rows), nb, sum(need)


def _make(name, nst, nct, rng, hq, hkv, d, dtype, num_blocks=None) -> Workload:
    nst = np.asarray(nst, dtype=np.int32)
    nct = np.asarray(nct, dtype=np.int32)
    bt, nb, uniq = _private_tables(rng, nct.astype(np.int64) + nst, BLOCK_SIZE, num_blocks)
    return Workload(name, nst, nct, bt, nb, BLOCK_SIZE, hq, hkv, d, dtype, uniq)


# ---------------------------------------------------------------------------
# The five named workloads
# ---------------------------------------------------------------------------

def tiny(seed: int = 0) -> Workload:
    """3 requests, [2,5,3] scheduled at [17,0,40] computed; 4 q / 2 kv heads,
    head_dim 64, a 16-block pool."""
    rng = np.random.default_rng(seed)
    return _make("tiny-3req-[2,5,3]", [2, 5, 3], [17, 0, 40], rng, 4, 2, 64, "bf16",
                 num_blocks=16)


def decode_batch(seed: int = 1) -> Workload:
    """256 single-token decodes, context ~ U[128, 4096]; 32 q / 8 kv heads, D 128."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(128, 4096, size=256, endpoint=True)
    return _make("decode-256x[128,4096]-gqa32/8-d128", np.ones(256, np.int32), ctx - 1,
                 rng, 32, 8, 128, "bf16")


def mixed_step(seed: int = 2, hq: int = 32, hkv: int = 8) -> Workload:
    """One 5000-token prompt chunk at 2048 computed, then 200 single-token decodes
    with context ~ U[256, 8192]; 32 q / 8 kv heads (or hq / hkv), D 128."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(256, 8192, size=200, endpoint=True)
    nst = np.concatenate([[5000], np.ones(200, np.int64)])
    nct = np.concatenate([[2048], ctx - 1])
    return _make(f"mixed-5000@2048+200x[256,8192]-gqa{hq}/{hkv}-d128", nst, nct, rng,
                 hq, hkv, 128, "bf16")


def chunk(seed: int = 5) -> Workload:
    """The mixed step's prompt chunk alone: one 5000-token chunk at 2048
    computed; 32 q / 8 kv heads, D 128, bf16 (a batch of the tensor-core
    kernel only: one grid over every SM)."""
    rng = np.random.default_rng(seed)
    return _make("chunk-5000@2048-gqa32/8-d128", [5000], [2048], rng, 32, 8, 128, "bf16")


def chunk_fp8_d64(seed: int = 5) -> Workload:
    """One 5000-token prompt chunk at 2048 computed over FP8 (E4M3) pools at
    head_dim 64; 32 q / 8 kv heads, bf16 q."""
    rng = np.random.default_rng(seed)
    return fp8(_make("chunk-5000@2048-gqa32/8-d64", [5000], [2048], rng, 32, 8, 64, "bf16"))


def mha_decode(seed: int = 3) -> Workload:
    """30 single-token decodes at context 2048; 40 q = 40 kv heads, D 128, fp16."""
    rng = np.random.default_rng(seed)
    return _make("mha-30x2048-h40-d128-fp16", np.ones(30, np.int32),
                 np.full(30, 2047, np.int32), rng, 40, 40, 128, "fp16")


def shared_prefix(seed: int = 4) -> Workload:
    """64 sequences sharing the physical blocks of a 1024-token prefix, each
    followed by P ~ U[0,31] full private blocks and u ~ U[0,15] more context
    tokens, with the new token at position 1024 + 16P + u in its own private
    block; plus 4 requests at context 32768.  32 q / 8 kv heads, D 128."""
    rng = np.random.default_rng(seed)
    bs = BLOCK_SIZE
    prefix_blocks = 1024 // bs
    p = rng.integers(0, 31, size=64, endpoint=True)
    u = rng.integers(0, 15, size=64, endpoint=True)
    nct_short = 1024 + bs * p + u
    long_ctx = np.full(4, 32768)
    private_need = [int(pi) + 1 for pi in p] + [_blocks_for(c, bs) for c in long_ctx]
    needed = prefix_blocks + sum(private_need)
    nb = _pool_size(needed)
    perm = rng.permutation(nb)
    shared = [int(b) for b in perm[:prefix_blocks]]
    k = prefix_blocks
    rows = []
    for i, n in enumerate(private_need):
        own = [int(b) for b in perm[k : k + n]]
        k += n
        rows.append(shared + own if i < 64 else own)
    nst = np.ones(68, np.int32)
    nct = np.concatenate([nct_short, long_ctx - 1]).astype(np.int32)
    return Workload("shared-prefix-64x(1024+priv)+4x32768-gqa32/8-d128", nst, nct,
                    _tables(rows), nb, bs, 32, 8, 128, "bf16", needed)


def fp8(w: Workload, k_scale: float = 0.25, v_scale: float = 0.125) -> Workload:
    """The same step over FP8 (E4M3) pools with per-pool scales."""
    return dataclasses.replace(w, name=w.name + "_fp8", kv_cache_dtype="fp8_e4m3",
                               k_scale=k_scale, v_scale=v_scale)


NAMED = {
    "tiny": tiny,
    "decode": decode_batch,
    "mixed": mixed_step,
    "mha": mha_decode,
    "shared_prefix": shared_prefix,
    "decode_fp8": lambda seed=1: fp8(decode_batch(seed)),
    "mixed_fp8": lambda seed=2: fp8(mixed_step(seed)),
    # 7 q heads per kv head (28 / 4): the tensor-core kernel's tiles hold 18
    # tokens (126 of 128 rows)
    "mixed_gqa28_4": lambda seed=2: mixed_step(seed, 28, 4),
    "chunk_fp8_d64": lambda seed=5: chunk_fp8_d64(seed),
    "chunk": lambda seed=5: chunk(seed),
}


def named(name: str, seed: int | None = None) -> Workload:
    fn = NAMED[name]
    return fn() if seed is None else fn(seed)


# ---------------------------------------------------------------------------
# Small random workloads for parity sweeps
# ---------------------------------------------------------------------------

def random_case(seed: int, *, max_reqs: int = 6, max_new: int = 40,
                max_computed: int = 300, head_dim: int | None = None,
                dtype: str | None = None, group: int | None = None,
                num_kv_heads: int | None = None, long_prefill: int = 0) -> Workload:
    """A random small step: 1..max_reqs requests mixing decodes (1 token) and
    chunks (2..max_new tokens) at random computed offsets.  ``long_prefill``
    adds one request of that many scheduled tokens."""
    rng = np.random.default_rng(seed)
    r = int(rng.integers(1, max_reqs, endpoint=True))
    kinds = rng.random(r) < 0.5
    nst = np.where(kinds, 1, rng.integers(2, max(3, max_new + 1), size=r))
    nct = rng.integers(0, max_computed, size=r, endpoint=True)
    if long_prefill:
        nst = np.concatenate([nst, [long_prefill]])
        nct = np.concatenate([nct, [int(rng.integers(0, max_computed + 1))]])
    hkv = int(num_kv_heads or rng.choice([1, 2, 4]))
    g = int(group or rng.choice([1, 2, 4, 8]))
    d = int(head_dim or rng.choice([64, 128]))
    dt = dtype or str(rng.choice(["bf16", "fp16"]))
    return _make(f"random-{seed}", nst, nct, rng, hkv * g, hkv, d, dt)


# ---------------------------------------------------------------------------
# Request state around the step: token lists, known totals, draft counts
# ---------------------------------------------------------------------------

VOCAB = 128_256


def make_token_buffer(w: Workload, seed: int = 0, max_num_reqs: int | None = None,
                      max_model_len: int | None = None) -> np.ndarray:
    """The per-request token buffer: int32 ``[max_num_reqs, max_model_len]``
    of random ids in [0, VOCAB).  Row r stands for batch row r's prompt plus
    output so far; every row is filled to the full width (a real buffer
    leaves its tail stale, and the step never reads past a request's
    positions).  Defaults: ``max_num_reqs = R + 3`` (spare rows) and
    ``max_model_len`` = the longest context rounded up to 16."""
    rng = np.random.default_rng(seed + 7_001)
    rows = w.num_reqs + 3 if max_num_reqs is None else int(max_num_reqs)
    width = max_model_len
    if width is None:
        width = max(16, -(-int(w.context_lens.max(initial=1)) // 16) * 16)
    return rng.integers(0, VOCAB, size=(rows, int(width)), dtype=np.int32)


def make_request_totals(w: Workload, seed: int = 0, p_caught_up: float = 0.5) -> np.ndarray:
    """Each request's total known token count (prompt plus output so far).
    With probability ``p_caught_up`` it equals computed + scheduled (the
    step reaches it: a decode, or a prompt's last chunk); otherwise the
    prompt continues for 1..2000 more tokens (a prefill chunk mid-prompt)."""
    rng = np.random.default_rng(seed + 7_002)
    reach = w.num_computed_tokens.astype(np.int64) + w.num_scheduled_tokens
    more = rng.integers(1, 2001, size=w.num_reqs)
    caught = rng.random(w.num_reqs) < p_caught_up
    return np.where(caught, reach, reach + more).astype(np.int32)


def make_draft_counts(w: Workload, seed: int = 0, max_drafts: int = 7) -> np.ndarray:
    """Draft tokens each request verifies this step: uniform in
    [0, min(max_drafts, scheduled - 1)] (the drafts are among the request's
    scheduled tokens, so a one-token request has none)."""
    rng = np.random.default_rng(seed + 7_003)
    hi = np.minimum(max_drafts, w.num_scheduled_tokens - 1)
    return (rng.random(w.num_reqs) * (hi + 1)).astype(np.int32).clip(0, hi)


# ---------------------------------------------------------------------------
# Values
# ---------------------------------------------------------------------------

def _randn(shape, gen: torch.Generator, device, dtype, chunk_elems: int = 1 << 27):
    """N(0,1) in fp32 rounded to ``dtype``; generated in chunks along dim 0 so
    the fp32 temporary stays bounded."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(shape[0], -1)
    row = flat.shape[1] if flat.dim() == 2 else 1
    step = max(1, chunk_elems // max(row, 1))
    for i in range(0, shape[0], step):
        j = min(shape[0], i + step)
        flat[i:j] = torch.randn((j - i, row), generator=gen, device=device,
                                dtype=torch.float32).to(dtype)
    return out


def make_values(w: Workload, seed: int = 0, device="cpu", fused_qkv: bool = False):
    """Q, the new tokens' K/V and a filled cache pool for workload ``w``.

    Returns a dict of tensors on ``device``: ``q [T,Hq,D]``, ``key``/``value``
    ``[T,Hkv,D]`` and ``key_cache``/``value_cache`` ``[NB,bs,Hkv,D]``.  With
    ``fused_qkv`` the three projections are views of one ``[T,(Hq+2Hkv)*D]``
    tensor, so ``key``/``value`` have token stride ``(Hq+2Hkv)*D``."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    dt = w.torch_dtype
    t, hq, hkv, d = w.num_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    out = {}
    if fused_qkv:
        qkv = _randn((max(t, 1), (hq + 2 * hkv) * d), gen, dev, dt)[:t]
        out["q"] = qkv[:, : hq * d].view(t, hq, d)
        out["key"] = qkv[:, hq * d : (hq + hkv) * d].view(t, hkv, d)
        out["value"] = qkv[:, (hq + hkv) * d :].view(t, hkv, d)
        out["qkv"] = qkv
    else:
        out["q"] = _randn((max(t, 1), hq, d), gen, dev, dt)[:t]
        out["key"] = _randn((max(t, 1), hkv, d), gen, dev, dt)[:t]
        out["value"] = _randn((max(t, 1), hkv, d), gen, dev, dt)[:t]
    shape = (w.num_blocks, w.block_size, hkv, d)
    if w.kv_cache_dtype == "fp8_e4m3":
        out["key_cache"] = _randn_fp8(shape, gen, dev, w.k_scale)
        out["value_cache"] = _randn_fp8(shape, gen, dev, w.v_scale)
        out["k_scale"] = torch.tensor([w.k_scale], dtype=torch.float32, device=dev)
        out["v_scale"] = torch.tensor([w.v_scale], dtype=torch.float32, device=dev)
    else:
        out["key_cache"] = _randn(shape, gen, dev, dt)
        out["value_cache"] = _randn(shape, gen, dev, dt)
    return out


def _randn_fp8(shape, gen: torch.Generator, device, scale: float, chunk_elems: int = 1 << 27):
    """Bytes of an FP8 (E4M3) pool whose cached values (element * scale) are
    about N(0, 1): N(0,1) / scale converted by PyTorch's float8_e4m3fn."""
    out = torch.empty(shape, dtype=torch.uint8, device=device)
    flat = out.view(shape[0], -1)
    row = flat.shape[1]
    step = max(1, chunk_elems // max(row, 1))
    for i in range(0, shape[0], step):
        j = min(shape[0], i + step)
        x = torch.randn((j - i, row), generator=gen, device=device, dtype=torch.float32)
        flat[i:j] = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return out
