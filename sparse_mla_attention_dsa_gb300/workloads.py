"""Seeded synthetic inputs for the DeepSeek Sparse Attention (MLA) forward.

This module only draws inputs: query vectors, the latent KV cache (bf16 rows or
FP8-e4m3 rows with per-group scales) and the top-k index lists.  It performs
none of the attention arithmetic.  Both the CUDA library's tests and the CPU
oracle's tests take their inputs from here, so the two sides see identical
bytes.

Shapes follow "Ascend Sparse Attention Forward: algorithm and optimisations",
section "数学建模" (problem statement): per query token Q[h_q, d_qk], a KV cache
KV[s_kv, d_qk] with d_qk = 576 (512 latent + 64 rope), an index list
indices[topk] into the KV rows, and d_v = 512 (the first 512 KV columns serve
as V).  The value -1 marks an unused index slot.

Randomness: numpy ``Generator(PCG64(seed))``, drawn in a fixed order (Q, then
KV, then indices).  Normal draws are float32 and are rounded to bf16 with
round-to-nearest-even by torch's dtype conversion.

FP8 KV row layout (656 bytes per KV token, data and scale adjacent as the
page's "Decoding KV Cache Layout 优化" section asks):

    bytes [0, 512)    512 x e4m3 latent codes
    bytes [512, 528)  4 x float32 scale, one per group of 128 latent channels
    bytes [528, 656)  64 x bf16 rope channels

The quantiser here produces those bytes from float32 latents: per (token,
group) scale = max|x| / 448 (1.0 for an all-zero group) and code = e4m3 of
x / scale, saturated to +-448, rounded to nearest even by torch's float8
conversion.  This is how the synthetic cache is made, not part of the method.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

D_QK = 576
D_V = 512
D_ROPE = D_QK - D_V
FP8_GROUP = 128
FP8_ROW_BYTES = D_V + 4 * (D_V // FP8_GROUP) + 2 * D_ROPE  # 656
E4M3_MAX = 448.0


@dataclass
class Workload:
    """One set of inputs for the forward (host tensors)."""

    name: str
    q: torch.Tensor  # bf16 [s_q, h_q, 576]
    kv: torch.Tensor  # bf16 [s_kv, 576]  or  uint8 [s_kv, 656] (fp8 rows)  or  uint8 [s_kv, 448] (fp4 rows)
    indices: torch.Tensor  # int32 [s_q, topk]
    sm_scale: float
    kv_format: str  # "bf16", "fp8" or "fp4"
    meta: dict = field(default_factory=dict)

    @property
    def s_q(self) -> int:
        return self.q.shape[0]

    @property
    def h_q(self) -> int:
        return self.q.shape[1]

    @property
    def s_kv(self) -> int:
        return self.kv.shape[0]

    @property
    def topk(self) -> int:
        return self.indices.shape[1]


def _normal_bf16(rng: np.random.Generator, shape, sigma: float = 1.0, chunk_rows: int = 1 << 18) -> torch.Tensor:
    """float32 N(0, sigma) draws rounded to bf16 (RNE), generated in row chunks."""
    shape = tuple(shape)
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(shape[0], -1) if len(shape) > 1 else out.view(-1, 1)
    row = flat.shape[1]
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(flat.shape[0], r0 + chunk_rows)
        x = rng.standard_normal((r1 - r0, row), dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        flat[r0:r1] = torch.from_numpy(x).to(torch.bfloat16)
    return out


def quantize_fp8_rows(latent: torch.Tensor, rope_bf16: torch.Tensor) -> torch.Tensor:
    """Pack float32 latents [n, 512] and bf16 rope [n, 64] into 656-byte FP8 rows."""
    n = latent.shape[0]
    g = latent.float().view(n, D_V // FP8_GROUP, FP8_GROUP)
    amax = g.abs().amax(dim=2)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    y = (g / scale.unsqueeze(2)).clamp_(-E4M3_MAX, E4M3_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).view(n, D_V)
    rows = torch.empty((n, FP8_ROW_BYTES), dtype=torch.uint8)
    rows[:, :D_V] = codes
    rows[:, D_V:D_V + 16] = scale.to(torch.float32).contiguous().view(torch.uint8).view(n, 16)
    rows[:, D_V + 16:] = rope_bf16.contiguous().view(torch.uint8).view(n, 2 * D_ROPE)
    return rows


def _fp8_kv(rng: np.random.Generator, s_kv: int, chunk_rows: int = 1 << 18) -> torch.Tensor:
    rows = torch.empty((s_kv, FP8_ROW_BYTES), dtype=torch.uint8)
    for r0 in range(0, s_kv, chunk_rows):
        r1 = min(s_kv, r0 + chunk_rows)
        lat = torch.from_numpy(rng.standard_normal((r1 - r0, D_V), dtype=np.float32))
        rope = torch.from_numpy(rng.standard_normal((r1 - r0, D_ROPE), dtype=np.float32)).to(torch.bfloat16)
        rows[r0:r1] = quantize_fp8_rows(lat, rope)
    return rows


FP4_GROUP = 32
FP4_ROW_BYTES = 448
_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)


def quantize_fp4_rows(latent: np.ndarray, rope_bf16: torch.Tensor) -> torch.Tensor:
    """Pack float32 latents [n, 512] and bf16 rope [n, 64] into 448-byte FP4 rows: 512 e2m1 codes two per
    byte (low nibble = even channel), 16 float32 scales (max |x| / 6 per 32 channels, 1 for an all-zero
    group), 64 bf16 rope values.  Codes are the nearest e2m1 magnitude, ties to the even code."""
    n = latent.shape[0]
    g = latent.astype(np.float32).reshape(n, D_V // FP4_GROUP, FP4_GROUP)
    amax = np.abs(g).max(axis=2)
    scale = np.where(amax > 0, amax / np.float32(6.0), np.float32(1.0)).astype(np.float32)
    y = np.abs(g) / scale[:, :, None]
    mids = (_E2M1_GRID[1:] + _E2M1_GRID[:-1]) / 2  # y between mids[i-1] and mids[i] -> code i
    lo = np.searchsorted(mids, y, side="left")
    hi = np.searchsorted(mids, y, side="right")
    mag = np.where((lo != hi) & (lo % 2 == 1), hi, lo).astype(np.uint8)  # a tie goes to the even code
    codes = (mag | np.where(g < 0, 8, 0).astype(np.uint8)).reshape(n, D_V)
    rows = np.empty((n, FP4_ROW_BYTES), dtype=np.uint8)
    rows[:, :D_V // 2] = codes[:, 0::2] | (codes[:, 1::2] << 4)
    rows[:, D_V // 2:D_V // 2 + 64] = scale.view(np.uint8).reshape(n, 64)
    rows[:, D_V // 2 + 64:] = rope_bf16.contiguous().view(torch.uint8).view(n, 2 * D_ROPE).numpy()
    return torch.from_numpy(rows)


def _fp4_kv(rng: np.random.Generator, s_kv: int, chunk_rows: int = 1 << 17) -> torch.Tensor:
    rows = torch.empty((s_kv, FP4_ROW_BYTES), dtype=torch.uint8)
    for r0 in range(0, s_kv, chunk_rows):
        r1 = min(s_kv, r0 + chunk_rows)
        lat = rng.standard_normal((r1 - r0, D_V), dtype=np.float32)
        rope = torch.from_numpy(rng.standard_normal((r1 - r0, D_ROPE), dtype=np.float32)).to(torch.bfloat16)
        rows[r0:r1] = quantize_fp4_rows(lat, rope)
    return rows


def _distinct(rng: np.random.Generator, lo: int, hi: int, k: int) -> np.ndarray:
    """k distinct integers drawn uniformly from [lo, hi)."""
    return rng.choice(hi - lo, size=k, replace=False).astype(np.int64) + lo


# ---------------------------------------------------------------------------
# The five workload shapes.  Their recipes are stated in the docstrings; the
# pages' own workload ("DeepSeek v4.1 典型工况") is unpublished, these stand in
# for it.
# ---------------------------------------------------------------------------

def tiny(seed: int = 0, s_q: int = 4, h_q: int = 16, s_kv: int = 256, topk: int = 64) -> Workload:
    """4 tokens, h_q=16, s_kv=256, topk=64 distinct uniform indices, N(0,1) bf16."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal_bf16(rng, (s_q, h_q, D_QK))
    kv = _normal_bf16(rng, (s_kv, D_QK))
    idx = np.stack([_distinct(rng, 0, s_kv, topk) for _ in range(s_q)])
    return Workload("tiny", q, kv, torch.from_numpy(idx.astype(np.int32)), 1.0 / math.sqrt(D_QK), "bf16")


def decode_bf16(seed: int = 1, n_seq: int = 64, h_q: int = 64, s_kv_per_seq: int = 32768, topk: int = 2048) -> Workload:
    """n_seq sequences x 1 query token over one flattened bf16 cache.

    Token b attends to `topk` distinct uniform positions of its own sequence,
    i.e. rows [b * s_kv_per_seq, (b + 1) * s_kv_per_seq) of the flattened cache.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal_bf16(rng, (n_seq, h_q, D_QK))
    kv = _normal_bf16(rng, (n_seq * s_kv_per_seq, D_QK))
    idx = np.stack([_distinct(rng, 0, s_kv_per_seq, topk) + b * s_kv_per_seq for b in range(n_seq)])
    return Workload("decode_bf16", q, kv, torch.from_numpy(idx.astype(np.int32)), 1.0 / math.sqrt(D_QK), "bf16",
                    meta={"n_seq": n_seq, "s_kv_per_seq": s_kv_per_seq})


def prefill_causal(seed: int = 2, s_q: int = 4096, h_q: int = 128, s_kv: int = 8192, topk: int = 2048,
                   invalid_frac: float = 0.05) -> Workload:
    """Causal prefill: query t sits at KV position s_kv - s_q + t.

    Each token draws `topk` distinct indices uniformly from [0, pos_t] and then
    round(invalid_frac * topk) slots, at uniformly chosen positions, are set to -1.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal_bf16(rng, (s_q, h_q, D_QK))
    kv = _normal_bf16(rng, (s_kv, D_QK))
    n_bad = int(round(invalid_frac * topk))
    idx = np.empty((s_q, topk), dtype=np.int64)
    base = s_kv - s_q
    for t in range(s_q):
        pos = base + t
        row = _distinct(rng, 0, pos + 1, topk)
        if n_bad:
            row[rng.choice(topk, size=n_bad, replace=False)] = -1
        idx[t] = row
    return Workload("prefill_causal", q, kv, torch.from_numpy(idx.astype(np.int32)), 1.0 / math.sqrt(D_QK), "bf16",
                    meta={"query_pos0": base, "n_invalid_per_token": n_bad})


def decode_fp8(seed: int = 3, n_seq: int = 128, h_q: int = 128, s_kv_per_seq: int = 65536, topk: int = 2048,
               q_sigma: float = 2.0) -> Workload:
    """n_seq sequences x 1 token over a flattened FP8 cache (656-byte rows).

    Q ~ N(0, sigma=2) so that logits spread and the online rescale fires.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal_bf16(rng, (n_seq, h_q, D_QK), sigma=q_sigma)
    kv = _fp8_kv(rng, n_seq * s_kv_per_seq)
    idx = np.stack([_distinct(rng, 0, s_kv_per_seq, topk) + b * s_kv_per_seq for b in range(n_seq)])
    return Workload("decode_fp8", q, kv, torch.from_numpy(idx.astype(np.int32)), 1.0 / math.sqrt(D_QK), "fp8",
                    meta={"n_seq": n_seq, "s_kv_per_seq": s_kv_per_seq, "q_sigma": q_sigma})


def long_prefill(seed: int = 4, s_q: int = 16384, h_q: int = 128, s_kv: int = 65536, topk: int = 2048,
                 nvalid_lo: int = 256, window: int = 512, local_frac: float = 0.7,
                 heavy_frac: float = 0.01, heavy_mult: float = 8.0) -> Workload:
    """Long prefill with ragged valid counts and clustered indices.

    Query t sits at position s_kv - s_q + t.  n_valid ~ U{nvalid_lo..topk};
    c = round(local_frac * n_valid) distinct indices come from the ceil(c/window)
    most recent windows of `window` positions ending at the query, the rest are
    distinct uniform from [0, start of those windows).  Valid slots are shuffled
    and slots [n_valid, topk) hold -1.  1% of (token, head) query rows are
    multiplied by 8 (heavy tails).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal_bf16(rng, (s_q, h_q, D_QK))
    kv = _normal_bf16(rng, (s_kv, D_QK))
    heavy = rng.random((s_q, h_q)) < heavy_frac
    if heavy.any():
        qf = q.float()
        qf[torch.from_numpy(heavy)] *= heavy_mult
        q = qf.to(torch.bfloat16)
    base = s_kv - s_q
    idx = np.full((s_q, topk), -1, dtype=np.int64)
    nvalid = rng.integers(nvalid_lo, topk + 1, size=s_q)
    for t in range(s_q):
        pos = base + t
        n = int(nvalid[t])
        c = int(round(local_frac * n))
        nwin = -(-c // window)
        lo = max(0, pos + 1 - nwin * window)
        local = _distinct(rng, lo, pos + 1, min(c, pos + 1 - lo))
        far_n = n - local.size
        far = _distinct(rng, 0, lo, min(far_n, lo)) if far_n > 0 and lo > 0 else np.empty(0, np.int64)
        row = np.concatenate([local, far])
        rng.shuffle(row)
        idx[t, :row.size] = row
    return Workload("long_prefill", q, kv, torch.from_numpy(idx.astype(np.int32)), 1.0 / math.sqrt(D_QK), "bf16",
                    meta={"query_pos0": base, "heavy_rows": int(heavy.sum())})


WORKLOADS = {
    "tiny": tiny,
    "decode_bf16": decode_bf16,
    "prefill_causal": prefill_causal,
    "decode_fp8": decode_fp8,
    "long_prefill": long_prefill,
}


def small_random(seed: int, s_q: int, h_q: int, s_kv: int, topk: int, kv_format: str = "bf16",
                 invalid_frac: float = 0.0, q_sigma: float = 1.0, distinct: bool = True) -> Workload:
    """A generic small case for parity tests (any shape, optional -1 slots)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal_bf16(rng, (s_q, h_q, D_QK), sigma=q_sigma)
    kv = {"bf16": lambda: _normal_bf16(rng, (s_kv, D_QK)), "fp8": lambda: _fp8_kv(rng, s_kv),
          "fp4": lambda: _fp4_kv(rng, s_kv)}[kv_format]()
    rows = []
    for _ in range(s_q):
        if distinct and topk <= s_kv:
            row = _distinct(rng, 0, s_kv, topk)
        else:
            row = rng.integers(0, max(s_kv, 1), size=topk).astype(np.int64)
        if invalid_frac > 0:
            row[rng.random(topk) < invalid_frac] = -1
        rows.append(row)
    idx = np.stack(rows) if rows else np.zeros((0, topk), np.int64)
    return Workload(f"small_{s_q}x{h_q}x{s_kv}x{topk}", q, kv, torch.from_numpy(idx.astype(np.int32)),
                    1.0 / math.sqrt(D_QK), kv_format)


def _paged(name: str, q: torch.Tensor, kv_pool: torch.Tensor, indices: np.ndarray, seq_of_token: np.ndarray,
           block_table: np.ndarray, page_size: int, kv_format: str, **meta) -> Workload:
    return Workload(name, q, kv_pool, torch.from_numpy(indices.astype(np.int32)), 1.0 / math.sqrt(D_QK), kv_format,
                    meta={"paged": True, "seq_of_token": torch.from_numpy(seq_of_token.astype(np.int32)),
                          "block_table": torch.from_numpy(block_table.astype(np.int32)), "page_size": page_size,
                          **meta})


def small_paged(seed: int, s_q: int, h_q: int, n_seq: int, max_pages: int, page_size: int, topk: int,
                kv_format: str = "bf16", spare_pages: int = 3, unmapped_frac: float = 0.0, invalid_frac: float = 0.0,
                past_end: int = 0) -> Workload:
    """A paged-cache case for parity tests.

    The pool holds n_seq * max_pages + spare_pages pages in random order; sequence s's table lists a random
    set of them, with round(unmapped_frac * max_pages) entries per sequence set to -1 (unmapped).  Each token
    belongs to a uniform random sequence and draws `topk` distinct logical positions from [0, max_pages *
    page_size); then round(invalid_frac * topk) slots become -1 and `past_end` slots point past the table.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    n_pages = n_seq * max_pages + spare_pages
    q = _normal_bf16(rng, (s_q, h_q, D_QK))
    kv = _normal_bf16(rng, (n_pages * page_size, D_QK)) if kv_format == "bf16" else _fp8_kv(rng, n_pages * page_size)
    table = rng.permutation(n_pages)[: n_seq * max_pages].reshape(n_seq, max_pages).astype(np.int64)
    n_unmapped = int(round(unmapped_frac * max_pages))
    for s in range(n_seq):
        if n_unmapped:
            table[s, rng.choice(max_pages, size=n_unmapped, replace=False)] = -1
    seq = rng.integers(0, n_seq, size=s_q)
    span = max_pages * page_size
    rows = []
    for _ in range(s_q):
        row = _distinct(rng, 0, span, topk) if topk <= span else rng.integers(0, span, size=topk).astype(np.int64)
        if invalid_frac > 0:
            row[rng.choice(topk, size=int(round(invalid_frac * topk)), replace=False)] = -1
        if past_end > 0:
            row[rng.choice(topk, size=past_end, replace=False)] = span + rng.integers(0, 4 * page_size, size=past_end)
        rows.append(row)
    return _paged(f"paged_{s_q}x{h_q}x{n_seq}x{max_pages}x{page_size}", q, kv, np.stack(rows), seq, table, page_size,
                  kv_format)


def decode_paged(seed: int = 5, n_seq: int = 64, h_q: int = 64, s_kv_per_seq: int = 32768, topk: int = 2048,
                 page_size: int = 64) -> Workload:
    """decode_bf16's shape over a paged pool: n_seq sequences x 1 query token, each sequence's s_kv_per_seq
    rows in pages of `page_size` rows scattered over the pool by a random permutation; token b attends to
    `topk` distinct uniform logical positions of sequence b."""
    rng = np.random.Generator(np.random.PCG64(seed))
    max_pages = s_kv_per_seq // page_size
    q = _normal_bf16(rng, (n_seq, h_q, D_QK))
    kv = _normal_bf16(rng, (n_seq * s_kv_per_seq, D_QK))
    table = rng.permutation(n_seq * max_pages).reshape(n_seq, max_pages)
    idx = np.stack([_distinct(rng, 0, s_kv_per_seq, topk) for _ in range(n_seq)])
    return _paged("decode_paged", q, kv, idx, np.arange(n_seq), table, page_size, "bf16", n_seq=n_seq,
                  s_kv_per_seq=s_kv_per_seq)


def decode_fp4(seed: int = 6, n_seq: int = 128, h_q: int = 128, s_kv_per_seq: int = 65536, topk: int = 2048,
               q_sigma: float = 2.0) -> Workload:
    """decode_fp8's shape over an FP4 cache (448-byte rows): n_seq sequences x 1 token, Q ~ N(0, sigma=2)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal_bf16(rng, (n_seq, h_q, D_QK), sigma=q_sigma)
    kv = _fp4_kv(rng, n_seq * s_kv_per_seq)
    idx = np.stack([_distinct(rng, 0, s_kv_per_seq, topk) + b * s_kv_per_seq for b in range(n_seq)])
    return Workload("decode_fp4", q, kv, torch.from_numpy(idx.astype(np.int32)), 1.0 / math.sqrt(D_QK), "fp4",
                    meta={"n_seq": n_seq, "s_kv_per_seq": s_kv_per_seq, "q_sigma": q_sigma})


WORKLOADS["decode_paged"] = decode_paged
WORKLOADS["decode_fp4"] = decode_fp4


# ---------------------------------------------------------------- output projection inputs
D_MODEL = 7168  # hidden size of the model the projection writes into (DeepSeek-V3's)


def oproj_inputs(seed: int, s_q: int, h_q: int, d_model: int = D_MODEL, out_sigma: float = 0.05):
    """Synthetic weights and residual for y = O . W_o + x: W_o bf16 [h_q * 512, d_model] ~ N(0, 1/sqrt(h_q * 512))
    (so that y has the scale of one attention output value), x bf16 [s_q, d_model] ~ N(0, 1), and a stand-alone
    attention output O bf16 [s_q, h_q, 512] ~ N(0, out_sigma) for tests of the projection alone."""
    rng = np.random.Generator(np.random.PCG64(seed))
    k = h_q * D_V
    w_o = _normal_bf16(rng, (k, d_model), sigma=1.0 / math.sqrt(k))
    x = _normal_bf16(rng, (s_q, d_model))
    o = _normal_bf16(rng, (s_q, h_q, D_V), sigma=out_sigma)
    return w_o, x, o


def prefill_oproj(seed: int = 7, d_model: int = D_MODEL) -> Workload:
    """The causal prefill followed by the output projection with residual into a d_model-wide hidden state."""
    wl = prefill_causal()
    rng = np.random.Generator(np.random.PCG64(seed))
    k = wl.h_q * D_V
    w_o = _normal_bf16(rng, (k, d_model), sigma=1.0 / math.sqrt(k))
    x = _normal_bf16(rng, (wl.s_q, d_model))
    wl.name = "prefill_oproj"
    wl.meta.update({"w_o": w_o, "x": x, "d_model": d_model})
    return wl


WORKLOADS["prefill_oproj"] = prefill_oproj
