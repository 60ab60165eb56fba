"""Seeded synthetic workloads for decode attention over a quantized paged cache.

This module draws random inputs and lays out block tables; it holds none of
the method's arithmetic (no quantisation, no attention).  Both the CUDA path
and the CPU oracle are fed from it.  Every tensor has its own
``torch.Generator`` whose seed is derived from (workload seed, tensor name,
sequence index), so a sequence's K/V rows are the same whether they are drawn
on their own or as part of a bulk fill, on the CPU or on a GPU (values differ
between the two device kinds, never between runs on one kind).

Workloads (shapes and distributions of the pages' measurements):
  tiny     B=1  Hq=4  Hkv=1 D=64  L=256, int8 per-row, block 256 in order
  gqa      B=1  Hq=24 Hkv=4 D=256, int8 per-row, block 256 in order, K channels
           multiplied by LogNormal(0, 0.5) factors (the kv-quant-attn page's
           27B-class geometry, context 1K..262,144)
  paged    B=16 Hq=32 Hkv=8 D=128, fp8 e4m3 per-tensor, block 16, shuffled
           block table, L_b ~ U{1..32768}, softcap 50 (PagedAttention PR #29912)
  spec     B=4  Hq=24 Hkv=4 D=256, int4 per-channel K and V, block 32,
           L=32768, T=8 query tokens (1 + 7 drafts) (INT4 PR #32515)
  mixed    B=64 Hq=64 Hkv=8 D=128, int8 per-channel K / per-tensor V, block 256,
           L_b = floor(exp(U(ln 16, ln 131072))), head sink ~ N(0,1), sliding
           window 4096 on alternate calls
Static scales are calibrated from the drawn data (max |x| / qmax per channel or
per tensor), so nothing saturates; they are inputs of the method, like the
offline calibration files the pages mention.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Optional

import numpy as np
import torch

INT8, FP8_E4M3, INT4 = 1, 2, 3
PER_ROW, PER_TENSOR, PER_CHANNEL, PER_GROUP = 1, 2, 3, 4
QMAX = {INT8: 127.0, INT4: 7.0, FP8_E4M3: 448.0}


def _seed(*parts) -> int:
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def generator(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


def randn_bf16(shape, device, *parts) -> torch.Tensor:
    g = generator(device, *parts)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


@dataclasses.dataclass
class Workload:
    name: str
    dtype: int
    k_mode: int
    v_mode: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    q_tokens: int
    block_size: int
    seq_lens: np.ndarray           # int32 [B], includes the q_tokens new rows
    block_table: np.ndarray        # int32 [B, max_blocks]
    num_blocks: int
    softcap: float = 0.0
    window: int = 0
    use_sink: bool = False
    k_channel_lognormal: float = 0.0   # sigma of per-(h, d) K factors (0: none)
    seed: int = 0
    group_size: int = 0                # channels per scale group of a PER_GROUP side

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    def row_bytes(self) -> int:
        return (self.head_dim + 1) // 2 if self.dtype == INT4 else self.head_dim

    # -- draws -------------------------------------------------------------
    def k_channel_factors(self, device) -> Optional[torch.Tensor]:
        if self.k_channel_lognormal <= 0:
            return None
        g = generator(device, self.seed, self.name, "kchan")
        z = torch.randn((self.num_kv_heads, self.head_dim), generator=g, device=device, dtype=torch.float32)
        return torch.exp(self.k_channel_lognormal * z)

    def seq_kv(self, b: int, device, lo: int = 0, hi: Optional[int] = None):
        """bf16 K, V rows [hi-lo, Hkv, D] of sequence b (positions lo..hi-1)."""
        L = int(self.seq_lens[b])
        hi = L if hi is None else hi
        shape = (L, self.num_kv_heads, self.head_dim)
        gk = generator(device, self.seed, self.name, "k", b)
        k = torch.randn(shape, generator=gk, device=device, dtype=torch.float32)
        f = self.k_channel_factors(device)
        if f is not None:
            k = k * f
        gv = generator(device, self.seed, self.name, "v", b)
        v = torch.randn(shape, generator=gv, device=device, dtype=torch.float32)
        return k[lo:hi].to(torch.bfloat16), v[lo:hi].to(torch.bfloat16)

    def q(self, device, step: int = 0) -> torch.Tensor:
        """bf16 queries [B, T, Hq, D] of decode step `step`."""
        return randn_bf16((self.batch, self.q_tokens, self.num_q_heads, self.head_dim), device,
                          self.seed, self.name, "q", step)

    def head_sink(self, device) -> Optional[torch.Tensor]:
        if not self.use_sink:
            return None
        g = generator(device, self.seed, self.name, "sink")
        return torch.randn((self.num_q_heads,), generator=g, device=device, dtype=torch.float32)

    def slots(self, b: int, lo: int, hi: int) -> np.ndarray:
        """Cache slots (block * block_size + row) of positions lo..hi-1 of sequence b."""
        t = np.arange(lo, hi, dtype=np.int64)
        return self.block_table[b, t // self.block_size].astype(np.int64) * self.block_size + t % self.block_size

    def window_for_call(self, call: int) -> int:
        """Sliding window of decode call `call` (alternating calls when set)."""
        return self.window if (self.window and call % 2 == 1) else 0


def rope_tables(max_pos: int, rotary_dim: int, base: float = 10000.0):
    """RoPE input tables cos / sin fp32 [max_pos, rotary_dim / 2] for angles
    pos * base^(-2i / rotary_dim) (the usual frequency ladder; the tables are
    the caller's input to the prologue, not part of its arithmetic)."""
    half = rotary_dim // 2
    inv = base ** (-np.arange(half, dtype=np.float64) * 2.0 / rotary_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def norm_weight_bf16(D: int, device, *parts) -> torch.Tensor:
    """A seeded RMSNorm weight vector, bf16 [D], values around 1."""
    g = generator("cpu", *parts)
    w = 1.0 + 0.25 * torch.randn(D, generator=g, dtype=torch.float32)
    return w.to(torch.bfloat16).to(device)


def calibrate_static(w: Workload, device, which: str) -> Optional[torch.Tensor]:
    """Static fp32 scale of side `which` ('k' or 'v') calibrated on the drawn rows:
    PER_TENSOR max|x|/qmax ([1]); PER_CHANNEL max_t |x[t,h,d]|/qmax ([Hkv, D])."""
    mode = w.k_mode if which == "k" else w.v_mode
    if mode in (PER_ROW, PER_GROUP):
        return None
    amax = torch.zeros((w.num_kv_heads, w.head_dim), dtype=torch.float32, device=device)
    for b in range(w.batch):
        if int(w.seq_lens[b]) == 0:
            continue
        k, v = w.seq_kv(b, device)
        x = (k if which == "k" else v).float().abs()
        amax = torch.maximum(amax, x.amax(dim=0))
    if mode == PER_TENSOR:
        amax = amax.max().reshape(1)
    amax = torch.where(amax > 0, amax, torch.ones_like(amax))
    return amax / torch.tensor(QMAX[w.dtype], dtype=torch.float32, device=device)


def _in_order_table(B, max_blocks):
    return (np.arange(B, dtype=np.int32)[:, None] * max_blocks + np.arange(max_blocks, dtype=np.int32)[None, :])


def _shuffled_table(seq_lens, block_size, max_blocks, device_seed_parts, slack=0):
    B = len(seq_lens)
    need = [max(1, math.ceil(int(L) / block_size)) for L in seq_lens]
    nb = sum(need) + slack
    g = generator("cpu", *device_seed_parts)
    perm = torch.randperm(nb, generator=g).numpy().astype(np.int32)
    table = np.zeros((B, max_blocks), dtype=np.int32)
    off = 0
    for b in range(B):
        table[b, :need[b]] = perm[off:off + need[b]]
        table[b, need[b]:] = perm[off + need[b] - 1]   # unused columns: a valid id, never read
        off += need[b]
    return table, nb


def make(name: str, *, ctx: Optional[int] = None, seed: int = 0, batch: Optional[int] = None,
         max_ctx: Optional[int] = None) -> Workload:
    """Build one of the named workloads.  `ctx` sets a uniform context length
    (tiny, gqa, spec); `max_ctx` scales down the ragged length laws (paged,
    mixed) for small test cases; `batch` overrides B."""
    if name == "tiny":
        B, L, bs = batch or 1, ctx or 256, 256
        mb = math.ceil(L / bs)
        return Workload(name, INT8, PER_ROW, PER_ROW, B, 4, 1, 64, 1, bs,
                        np.full(B, L, np.int32), _in_order_table(B, mb), B * mb, seed=seed)
    if name == "gqa":
        B, L, bs = batch or 1, ctx or 16384, 256
        mb = math.ceil(L / bs)
        return Workload(name, INT8, PER_ROW, PER_ROW, B, 24, 4, 256, 1, bs,
                        np.full(B, L, np.int32), _in_order_table(B, mb), B * mb,
                        k_channel_lognormal=0.5, seed=seed)
    if name == "paged":
        B, bs = batch or 16, 16
        hi = max_ctx or 32768
        g = generator("cpu", seed, name, "lengths")
        lens = torch.randint(1, hi + 1, (B,), generator=g).numpy().astype(np.int32)
        mb = math.ceil(hi / bs)
        table, nb = _shuffled_table(lens, bs, mb, (seed, name, "perm"))
        return Workload(name, FP8_E4M3, PER_TENSOR, PER_TENSOR, B, 32, 8, 128, 1, bs, lens, table, nb,
                        softcap=50.0, seed=seed)
    if name == "spec":
        B, L, bs = batch or 4, ctx or 32768, 32
        mb = math.ceil(L / bs)
        table, nb = _shuffled_table(np.full(B, L), bs, mb, (seed, name, "perm"))
        return Workload(name, INT4, PER_CHANNEL, PER_CHANNEL, B, 24, 4, 256, 8, bs,
                        np.full(B, L, np.int32), table, nb, seed=seed)
    if name == "mixed":
        B, bs = batch or 64, 256
        hi = max_ctx or 131072
        lo = min(16, hi)
        g = generator("cpu", seed, name, "lengths")
        u = torch.rand((B,), generator=g, dtype=torch.float64).numpy()
        lens = np.floor(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
        lens = np.clip(lens, lo, hi).astype(np.int32)
        mb = math.ceil(hi / bs)
        table, nb = _shuffled_table(lens, bs, mb, (seed, name, "perm"))
        return Workload(name, INT8, PER_CHANNEL, PER_TENSOR, B, 64, 8, 128, 1, bs, lens, table, nb,
                        window=4096 if hi > 4096 else max(1, hi // 4), use_sink=True, seed=seed)
    raise KeyError(name)


def step_bytes(w: Workload, window: int = 0) -> dict:
    """Algorithmic bytes of one decode step, by component:
      kv     K and V codes (+ per-row scales) of every key some query row sees
      q      the queries, read once
      table  block-table entries of the pages those keys sit in, and seq_lens
      out    the bf16 output, written once
      append the T new rows per sequence: bf16 K/V read, codes (+ scales) and
             slot_mapping written/read
    Split partials in the workspace are implementation overhead, not counted."""
    keys = 0
    pages = 0
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        lo = max(0, L - w.q_tokens + 1 - window) if window > 0 else 0
        keys += max(0, L - lo)
        if L > lo:
            pages += (L - 1) // w.block_size - lo // w.block_size + 1
    def scale_bytes(mode):
        return 4 if mode == PER_ROW else (4 * (w.head_dim // w.group_size) if mode == PER_GROUP else 0)
    scales = scale_bytes(w.k_mode) + scale_bytes(w.v_mode)
    per_key = 2 * w.row_bytes() + scales
    qo = w.batch * w.q_tokens * w.num_q_heads * w.head_dim * 2
    new = w.batch * w.q_tokens
    return dict(kv=keys * w.num_kv_heads * per_key, q=qo, table=4 * pages + 4 * w.batch, out=qo,
                append=new * w.num_kv_heads * (2 * w.head_dim * 2 + per_key) + 8 * new)


def decode_bytes(w: Workload, window: int = 0) -> int:
    """Algorithmic bytes the decode kernel itself moves (kv + q + table)."""
    s = step_bytes(w, window)
    return s["kv"] + s["q"] + s["table"]


def cache_bytes_read(w: Workload, window: int = 0) -> int:
    """All algorithmic bytes of one step (decode, combine output, append)."""
    return sum(step_bytes(w, window).values())
