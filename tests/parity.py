"""Helpers for GPU-vs-oracle parity tests (imported by the gpu test modules).

The oracle gets the same seeded bf16 rows, static scales and queries as the
CUDA path and quantizes them itself; nothing it consumes comes from the CUDA
path.  For large workloads only the sequences a test samples are loaded into
the oracle's cache, with their block ids remapped into a compact pool.
"""
import numpy as np
import torch

from decode_attention_quantized_gb300 import synth
from decode_attention_quantized_gb300.workload import GpuWorkload

REL_L2_BAR = 2e-3     # decode output vs the fp64 oracle, relative L2 (the method's target)
ROW_BAR = 8e-3        # any single (b, t, head) row, relative L2 (catches a broken row)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


class OracleSide:
    """Oracle cache of sequences `seqs` of workload `w` (all their positions)."""

    def __init__(self, orc, w: synth.Workload, seqs, gen_device, k_static, v_static):
        self.w, self.seqs = w, list(seqs)
        bs = w.block_size
        used = []
        for b in self.seqs:
            L = int(w.seq_lens[b])
            used.extend(int(x) for x in w.block_table[b, :max(1, (L + bs - 1) // bs)])
        self.gpu_blocks = sorted(set(used))
        remap = {g: i for i, g in enumerate(self.gpu_blocks)}
        self.table = np.zeros((len(self.seqs), w.max_blocks), np.int32)
        for r, b in enumerate(self.seqs):
            L = int(w.seq_lens[b])
            n = max(1, (L + bs - 1) // bs)
            self.table[r, :n] = [remap[int(x)] for x in w.block_table[b, :n]]
        ks = None if k_static is None else k_static.detach().cpu().numpy()
        vs = None if v_static is None else v_static.detach().cpu().numpy()
        self.cache = orc.OracleCache(w.dtype, w.k_mode, w.v_mode, len(self.gpu_blocks), bs, w.num_kv_heads,
                                     w.head_dim, ks, vs, group_size=w.group_size)
        for r, b in enumerate(self.seqs):
            L = int(w.seq_lens[b])
            if L == 0:
                continue
            k, v = w.seq_kv(b, gen_device)
            t = np.arange(L)
            slots = self.table[r, t // bs].astype(np.int64) * bs + t % bs
            assert self.cache.append(bits(k), bits(v), slots) == 0
        self.lens = np.array([int(w.seq_lens[b]) for b in self.seqs], np.int32)

    def compare_cache(self, gw: GpuWorkload):
        """Codes and per-row / per-group scales of the sampled sequences, byte for byte."""
        ids = torch.tensor(self.gpu_blocks, dtype=torch.long, device=gw.cache.k_codes.device)
        for name in ("k_codes", "v_codes"):
            g = getattr(gw.cache, name).index_select(0, ids).cpu().numpy()
            o = getattr(self.cache, name)
            assert np.array_equal(g, o), f"{name} differ in {np.count_nonzero(g != o)} bytes"
        for side, mode in (("k_scale", self.w.k_mode), ("v_scale", self.w.v_mode)):
            if mode in (synth.PER_ROW, synth.PER_GROUP):
                g = getattr(gw.cache, side).index_select(0, ids).cpu().numpy()
                o = getattr(self.cache, side)
                assert np.array_equal(g.view(np.uint32), o.view(np.uint32)), f"{side} differ"

    def attend(self, q_bf16: torch.Tensor, *, window=0, sink=None, rows=None, nthreads=None):
        """Oracle output for the sampled sequences: q [B, T, Hq, D] of the full batch."""
        q = bits(q_bf16)[self.seqs]
        s = None if sink is None else sink.detach().cpu().numpy()
        r = None
        if rows is not None:
            pos = {b: i for i, b in enumerate(self.seqs)}
            r = np.array([(pos[b], t, h) for (b, t, h) in rows], np.int32)
        return self.cache.attend(q, self.table, self.lens, q_tokens=self.w.q_tokens, softcap=self.w.softcap,
                                 window=window, head_sink=s, rows=r, nthreads=nthreads)


def bf16_bits_to_f64(u) -> np.ndarray:
    return (np.asarray(u, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_neighbours(v):
    """(lower, upper) bf16 values around each fp64 value v (finite) and the
    midpoint between them, exactly in fp64 (spacing 2^(e-7) in the binade
    [2^e, 2^(e+1)), 2^-133 below 2^-126)."""
    v = np.asarray(v, np.float64)
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    q = np.ldexp(1.0, (e - 7).astype(int))
    lo = np.floor(v / q) * q
    return lo, lo + q, lo + q / 2


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / n) if n > 0 else float(np.linalg.norm(got))


def check_rows(got: np.ndarray, ref: np.ndarray, *, bar=REL_L2_BAR, row_bar=ROW_BAR):
    """got, ref [..., D].  Whole-tensor relative L2 within `bar`, every row
    within `row_bar` (relative to its own norm, or absolute for ~zero rows),
    and rows the oracle gives as exactly zero are exactly zero."""
    err = rel_l2(got, ref)
    assert err <= bar, f"relative L2 {err:.3e} > {bar}"
    g = got.reshape(-1, got.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    nr = np.linalg.norm(r, axis=1)
    ne = np.linalg.norm(g - r, axis=1)
    zero = nr == 0
    assert (ne[zero] == 0).all(), "rows with an empty key set must be exactly zero"
    worst = (ne[~zero] / nr[~zero]).max() if (~zero).any() else 0.0
    assert worst <= row_bar, f"worst row relative L2 {worst:.3e} > {row_bar}"
    return err, worst


def check_lse(got: np.ndarray, ref: np.ndarray, tol=2e-3):
    fin = np.isfinite(ref)
    assert (np.isneginf(got) == np.isneginf(ref)).all(), "empty key sets must report lse = -inf"
    assert np.abs(got[fin] - ref[fin]).max(initial=0.0) <= tol * (1 + np.abs(ref[fin]).max(initial=0.0))
