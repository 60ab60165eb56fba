"""Drive a synthetic workload through the kvq C ABI on one GPU.

Fills a device cache through ``kvq_append`` (the history, positions
0 .. L_b - T - 1 of every sequence), then runs decode steps: append the T new
tokens of every sequence, ``kvq_decode``, ``kvq_combine``.  Used by the GPU
tests and by bench.py; all arithmetic happens in the CUDA library.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import kvq, synth


class GpuWorkload:
    def __init__(self, w: synth.Workload, *, device="cuda", gen_device="cuda",
                 k_static: Optional[torch.Tensor] = None, v_static: Optional[torch.Tensor] = None):
        self.w = w
        self.device = device
        self.gen_device = gen_device
        if k_static is None:
            k_static = synth.calibrate_static(w, gen_device, "k")
        if v_static is None:
            v_static = synth.calibrate_static(w, gen_device, "v")
        self.k_static, self.v_static = k_static, v_static
        self.cache = kvq.QuantizedPagedCache(w.dtype, w.k_mode, w.v_mode, w.num_blocks, w.block_size,
                                             w.num_kv_heads, w.head_dim, device=device, k_static=k_static,
                                             v_static=v_static, group_size=w.group_size)
        self.block_table = torch.from_numpy(np.ascontiguousarray(w.block_table)).to(device)
        self.seq_lens = torch.from_numpy(np.ascontiguousarray(w.seq_lens)).to(device)
        sink = w.head_sink(gen_device)
        self.head_sink = None if sink is None else sink.to(device)
        self.max_seq_len = int(w.seq_lens.max()) if w.batch else 0

    # -- cache contents ---------------------------------------------------
    def fill_history(self):
        """Append positions 0 .. L_b - T - 1 of every sequence (bulk fill)."""
        w = self.w
        for b in range(w.batch):
            hi = int(w.seq_lens[b]) - w.q_tokens
            if hi <= 0:
                continue
            k, v = w.seq_kv(b, self.gen_device, 0, hi)
            slots = torch.from_numpy(w.slots(b, 0, hi)).to(self.device)
            kvq.kvq_append(self.cache, k.to(self.device).contiguous(), v.to(self.device).contiguous(), slots)

    def new_tokens(self):
        """bf16 K, V [B*T, Hkv, D] and int64 slots [B*T] of the T newest positions
        (a slot of -1 for positions that do not exist, i.e. L_b < T)."""
        w = self.w
        ks, vs, sl = [], [], []
        for b in range(w.batch):
            L = int(w.seq_lens[b])
            lo = L - w.q_tokens
            k, v = w.seq_kv(b, self.gen_device, max(lo, 0), L)
            pad = max(0, -lo)
            if pad:
                z = torch.zeros((pad, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16, device=k.device)
                k, v = torch.cat([z, k]), torch.cat([z, v])
            ks.append(k)
            vs.append(v)
            s = np.full(w.q_tokens, -1, np.int64)
            if L > max(lo, 0):
                s[pad:] = w.slots(b, max(lo, 0), L)
            sl.append(s)
        return (torch.cat(ks).to(self.device).contiguous(), torch.cat(vs).to(self.device).contiguous(),
                torch.from_numpy(np.concatenate(sl)).to(self.device))

    def params(self, window: int = 0, max_seq_len: Optional[int] = None, flags: int = 0):
        w = self.w
        return kvq.make_params(w.batch, w.num_q_heads, w.q_tokens, w.max_blocks,
                               max_seq_len=self.max_seq_len if max_seq_len is None else max_seq_len,
                               softcap=w.softcap, window=window, flags=flags)

    def buffers(self, params):
        return kvq.alloc_decode_buffers(self.cache, params)

    def step(self, q, k_new, v_new, slots, params, bufs, stream=None):
        """One decode step: append the new tokens, decode, combine."""
        kvq.kvq_append(self.cache, k_new, v_new, slots, stream)
        return kvq.decode_step(self.cache, params, q, self.block_table, self.seq_lens, bufs, self.head_sink, stream)
