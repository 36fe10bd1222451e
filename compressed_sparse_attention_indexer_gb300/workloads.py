"""Seeded synthetic inputs for the CSA decode step.

This module only draws random numbers and lays them out in the caller-owned
pools the library reads.  It holds none of the method's arithmetic: no score,
no selection, no softmax, no rotary math.  Both the CUDA path and the CPU
oracle are fed from here, so the two always see identical stored values.

Shapes follow the decode workloads of the hw-native-sys/pypto-lib pages
("Perf: skip redundant CSA scoring and fuse gather unpack": TP4 CSA at 16x256;
"Perf: fuse HCA merge, inverse RoPE, and packing": B=16, S=8) extended to long
ragged contexts.  No dataset or trained weight is involved.

Pool layout (the storage contract of the library):
  * compressed pool ``cmp_kv`` and indexer-key pool ``idx_k``: request b owns
    floor(L_b / ratio) consecutive rows starting at ``cmp_off[b]`` /
    ``idx_off[b]``;
  * heavy-compression pool ``hca_kv``: floor(L_b / hca_ratio) rows;
  * raw (sliding-window) pool ``raw_kv``: an SWA cache keeps only the last
    ``raw_keep`` raw tokens of each request, so row r of request b lives at
    ``raw_off[b] + r`` for r in [L_b - raw_keep, L_b) and is absent otherwise
    (``raw_off[b]`` may therefore be negative).
  ``gap_rows`` rows filled with NaN separate requests in every pool, so a read
  of a row a query may not use poisons its output.

With ``idx_dtype="fp8"`` the indexer-key pool is stored as FP8 E4M3 codes
(uint8) with one fp32 scale per row (``idx_scale``): each row is drawn like
the bf16 rows (the same fp32 normal draws), its scale is max|row| / 448 and
its codes are row / scale rounded to E4M3 by torch's float8_e4m3fn cast.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class CsaConfig:
    """Static shape of one CSA attention layer."""
    H: int = 64            # attention heads
    D: int = 576           # KV row width: V value dims + R rope dims
    V: int = 512           # value / output dims
    Hi: int = 64           # indexer heads
    Di: int = 128          # indexer dim
    ratio: int = 4         # CSA compression ratio
    topk: int = 512        # K
    win: int = 128         # sliding window WIN
    hca_ratio: int = 0     # heavy-compression ratio (0 = no third stream)
    dtype: str = "bf16"    # "bf16" or "f32"
    idx_dtype: str = "same"  # indexer-key pool: "same" (the layer dtype) or "fp8" (E4M3 + row scale)
    rope_base: float = 10000.0
    scale: float | None = None  # softmax scale; None -> 1/sqrt(D)

    @property
    def R(self) -> int:
        return self.D - self.V

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def esize(self) -> int:
        return 2 if self.dtype == "bf16" else 4


@dataclass(frozen=True)
class Dists:
    """Standard deviations of the normal draws (w is U(0, w_hi))."""
    q: float = 1.0
    q_idx: float = 1.0
    k_idx: float = 1.0
    raw: float = 1.0
    cmp: float = 0.5
    hca: float = 0.5
    w_hi: float = 1.0


@dataclass(frozen=True)
class Workload:
    name: str
    cfg: CsaConfig
    B: int
    S: int
    L: int | None = None            # fixed context length, or
    L_range: tuple | None = None    # (lo, hi) inclusive, uniform per request
    seed: int = 1000
    dists: Dists = field(default_factory=Dists)
    description: str = ""


TINY_CFG = CsaConfig(H=4, D=80, V=64, Hi=2, Di=32, ratio=4, topk=8, win=8, dtype="f32")
BF16_CFG = CsaConfig()

WORKLOADS = {
    "tiny_f32": Workload(
        "tiny_f32", TINY_CFG, B=1, S=1, L=64, seed=1000,
        dists=Dists(cmp=1.0, hca=1.0),
        description="B=1 S=1 L=64 (16 compressed rows > K=8), WIN=8, H=4, D=80 (V=64 + rope 16), "
                    "indexer 2x32, fp32, all N(0,1), w~U(0,1)"),
    "bypass_b16_l256": Workload(
        "bypass_b16_l256", BF16_CFG, B=16, S=1, L=256, seed=1001,
        description="B=16 S=1 L=256: 64 compressed rows <= K=512 so scoring is skipped; WIN=128, "
                    "H=64, D=576, bf16; activations N(0,1), compressed rows N(0,0.5^2)"),
    "topk_b16_l8192": Workload(
        "topk_b16_l8192", BF16_CFG, B=16, S=1, L=8192, seed=1002,
        description="B=16 S=1 L=8192: 2048 compressed rows, K=512, WIN=128, H=64, D=576, bf16; "
                    "q_idx, k_idx N(0,1) so the Top-K boundary is dense with near-ties"),
    "long_ragged_b64": Workload(
        "long_ragged_b64", BF16_CFG, B=64, S=1, L_range=(1024, 65536), seed=1003,
        description="B=64 S=1, L_b ~ U{1024..65536}: 256..16384 compressed rows per request, "
                    "K=512, WIN=128, H=64, D=576, indexer 64x128, bf16"),
    "long_ragged_b64_fp8idx": Workload(
        "long_ragged_b64_fp8idx", replace(BF16_CFG, idx_dtype="fp8"), B=64, S=1,
        L_range=(1024, 65536), seed=1003,
        description="long_ragged_b64 (same lengths and draws) with the indexer keys stored as "
                    "FP8 E4M3 codes and one fp32 scale per row"),
    "prefill_b2_t512": Workload(
        "prefill_b2_t512", BF16_CFG, B=2, S=512, L=4096, seed=1006,
        description="a prefill chunk: B=2 requests, 512 new tokens each at the end of a 4096-token "
                    "context (positions 3584..4095, vis 896..1024 > K), each token scoring its "
                    "visible compressed rows and taking its own Top-K; H=64, D=576, bf16"),
    "multitoken_hca_b16_s8": Workload(
        "multitoken_hca_b16_s8", replace(BF16_CFG, hca_ratio=128), B=16, S=8, L=32768, seed=1004,
        description="B=16 S=8 L=32768 with per-query causal visibility; CSA (ratio 4, K=512, "
                    "WIN=128) plus all ratio-128 rows as a third stream; H=64, D=576, bf16"),
}


def context_lengths(wl: Workload, gen: torch.Generator) -> torch.Tensor:
    if wl.L is not None:
        return torch.full((wl.B,), wl.L, dtype=torch.int32)
    lo, hi = wl.L_range
    return torch.randint(lo, hi + 1, (wl.B,), generator=gen, dtype=torch.int64).to(torch.int32)


def _normal(gen, shape, std, dtype):
    t = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _pool(gen, counts, width, std, dtype, gap_rows, first=None):
    """Concatenates per-request row blocks; returns (pool [rows, width], off int64 [B])."""
    B = len(counts)
    total = sum(counts) + gap_rows * (B + 1)
    pool = torch.full((max(total, 1), width), float("nan"), dtype=dtype) if gap_rows else \
        torch.empty((max(total, 1), width), dtype=dtype)
    off = torch.zeros(B, dtype=torch.int64)
    cur = gap_rows
    for b, n in enumerate(counts):
        if n:
            pool[cur:cur + n] = _normal(gen, (n, width), std, dtype)
        off[b] = cur - (first[b] if first is not None else 0)
        cur += n + gap_rows
    return pool, off


def _fp8_pool(gen, counts, width, std, gap_rows):
    """Indexer-key pool as FP8 E4M3 codes (uint8 [rows, width]) and a per-row
    fp32 scale: rows drawn as in _pool (NaN gap rows give NaN codes and scales)."""
    keys, off = _pool(gen, counts, width, std, torch.float32, gap_rows)
    amax = keys.abs().amax(dim=1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (keys / scale[:, None]).clamp(-448.0, 448.0)
    codes = torch.where(keys.isnan(), keys, codes)
    return codes.to(torch.float8_e4m3fn).view(torch.uint8).contiguous(), off, scale.contiguous()


def make_batch(wl: Workload, lens=None, seed: int | None = None, gap_rows: int = 0,
               raw_keep: int | None = None, dists: Dists | None = None) -> dict:
    """Host (CPU) tensors for one batch of `wl`.

    lens: optional explicit per-request context lengths (overrides the
    workload's).  raw_keep: trailing raw tokens stored per request (default:
    WIN + S, enough for every window of the step).
    """
    cfg = wl.cfg
    d = dists or wl.dists
    gen = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    dt = cfg.torch_dtype
    if lens is None:
        ctx = context_lengths(wl, gen)
    else:
        ctx = torch.as_tensor(list(lens), dtype=torch.int32)
    B, S = int(ctx.numel()), wl.S
    assert int(ctx.min()) >= S, "every request must hold its S new tokens"
    keep = raw_keep if raw_keep is not None else cfg.win + S
    q = _normal(gen, (B, S, cfg.H, cfg.D), d.q, dt)
    q_idx = _normal(gen, (B, S, cfg.Hi, cfg.Di), d.q_idx, dt)
    w = (torch.rand(B, S, cfg.Hi, generator=gen, dtype=torch.float32) * d.w_hi).contiguous()
    Ls = [int(x) for x in ctx]
    first = [max(0, L - keep) for L in Ls]
    raw_kv, raw_off = _pool(gen, [L - f for L, f in zip(Ls, first)], cfg.D, d.raw, dt, gap_rows, first)
    ncmp = [L // cfg.ratio for L in Ls]
    cmp_kv, cmp_off = _pool(gen, ncmp, cfg.D, d.cmp, dt, gap_rows)
    idx_scale = None
    if cfg.idx_dtype == "fp8":
        idx_k, idx_off, idx_scale = _fp8_pool(gen, ncmp, cfg.Di, d.k_idx, gap_rows)
    else:
        idx_k, idx_off = _pool(gen, ncmp, cfg.Di, d.k_idx, dt, gap_rows)
    batch = dict(B=B, S=S, ctx_len=ctx, q=q, q_idx=q_idx, w=w, _rows_cmp=ncmp, _rows_idx=ncmp,
                 raw_kv=raw_kv, raw_off=raw_off, raw_stride=cfg.D, raw_first=first,
                 cmp_kv=cmp_kv, cmp_off=cmp_off, cmp_stride=cfg.D,
                 idx_k=idx_k, idx_off=idx_off, idx_stride=cfg.Di, idx_scale=idx_scale,
                 hca_kv=None, hca_off=None, hca_stride=0)
    if cfg.hca_ratio:
        nh = [L // cfg.hca_ratio for L in Ls]
        hca_kv, hca_off = _pool(gen, nh, cfg.D, d.hca, dt, gap_rows)
        batch.update(hca_kv=hca_kv, hca_off=hca_off, hca_stride=cfg.D, _rows_hca=nh)
    return batch


def paginate(batch: dict, blocks: dict, seed: int = 0, spare_blocks: int = 2) -> dict:
    """The same batch with paged pools: for each pool named in `blocks`
    ("raw", "cmp", "idx", "hca" -> rows per block), the request's rows are
    cut into logical blocks placed at shuffled pool blocks, and a block table
    per pool maps request b's logical block k to its pool block
    (table[b, k], -1 = unmapped).  Pool rows that hold no request row (the
    tail of a request's last block, spare blocks, raw rows before the window
    a request keeps) are NaN (FP8 keys: the NaN code, scale NaN), so a read
    of a row the step may not use poisons its output.  Layout only: the row
    values are the batch's own."""
    out = dict(batch)
    B = int(batch["B"])
    Ls = [int(x) for x in batch["ctx_len"]]
    gen = torch.Generator().manual_seed(seed)
    keys = {"raw": "raw_kv", "cmp": "cmp_kv", "idx": "idx_k", "hca": "hca_kv"}
    plans = {}
    tstride = 1
    for name, bs in blocks.items():
        if batch.get(keys[name]) is None:
            continue
        if name == "raw":  # rows are positions; a request keeps [first, L)
            rng = [(int(batch["raw_first"][b]), Ls[b]) for b in range(B)]
        else:
            rng = [(0, int(n)) for n in batch["_rows_" + name]]
        nblk = [(hi + bs - 1) // bs for (_, hi) in rng]
        tstride = max(tstride, max(nblk))
        plans[name] = (bs, rng, nblk)
    for name, (bs, rng, nblk) in plans.items():
        key = keys[name]
        src, off = batch[key], batch[name + "_off"]
        # logical blocks that hold at least one existing row get a pool block
        owned = [(b, k) for b in range(B) for k in range(nblk[b]) if (k + 1) * bs > rng[b][0]]
        total = len(owned) + spare_blocks
        perm = torch.randperm(total, generator=gen).tolist()
        if src.dtype == torch.uint8:
            pool = torch.full((total * bs, src.shape[1]), 0x7F, dtype=torch.uint8)
        else:
            pool = torch.full((total * bs, src.shape[1]), float("nan"), dtype=src.dtype)
        scale = None
        if name == "idx" and batch.get("idx_scale") is not None:
            scale = torch.full((total * bs,), float("nan"), dtype=torch.float32)
        table = torch.full((B, tstride), -1, dtype=torch.int32)
        for i, (b, k) in enumerate(owned):
            pb = perm[i]
            table[b, k] = pb
            lo, hi = max(k * bs, rng[b][0]), min((k + 1) * bs, rng[b][1])
            rows = slice(int(off[b]) + lo, int(off[b]) + hi)
            dst = slice(pb * bs + (lo - k * bs), pb * bs + (hi - k * bs))
            pool[dst] = src[rows]
            if scale is not None:
                scale[dst] = batch["idx_scale"][rows]
        out[key] = pool
        out[name + "_table"] = table
        out[name + "_block"] = bs
        out[name + "_off"] = None
        if scale is not None:
            out["idx_scale"] = scale
    out["table_stride"] = tstride
    return out


TENSOR_KEYS = ("ctx_len", "q", "q_idx", "w", "raw_kv", "raw_off", "cmp_kv", "cmp_off",
               "idx_k", "idx_off", "idx_scale", "hca_kv", "hca_off",
               "raw_table", "cmp_table", "idx_table", "hca_table")


def to_device(batch: dict, device) -> dict:
    out = dict(batch)
    for k in TENSOR_KEYS:
        if batch.get(k) is not None:
            out[k] = batch[k].to(device).contiguous()
    return out
