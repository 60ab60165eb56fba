"""Guard bands around the device buffers the GPU tests hand to the library.

The sanitizer does not run on this hardware's test pool, so out-of-bounds
writes are caught the old way: every cache code pool, scale array, workspace
and output a GPU test passes to a kvq call sits inside a larger allocation
whose first and last GUARD bytes hold known patterns.  After each GPU test
the bands are read back; a kernel that wrote past either end of a buffer
changes them, and the test fails even when the stray write hit nothing that
a parity check compares.

kvq.QuantizedPagedCache and kvq.alloc_decode_buffers are wrapped for the
whole session (so every cache and decode buffer is banded); tests that
allocate an output themselves call guarded().
"""
from __future__ import annotations

import weakref

import torch

GUARD = 4096        # bytes on each side (a multiple of 512 keeps the inner buffer's alignment)
HEAD, TAIL = 0xA5, 0x5A

_live: list = []    # (strong or weak reference to the inner tensor, nbytes, label)


def guarded(t: torch.Tensor, label: str = "") -> torch.Tensor:
    """A device tensor equal to t (same shape, dtype and contents) placed
    between two guard bands; registered for the check after the test."""
    if t.device.type != "cuda":
        return t
    t = t.contiguous()
    n = t.numel() * t.element_size()
    raw = torch.empty(n + 2 * GUARD, dtype=torch.uint8, device=t.device)
    raw[:GUARD].fill_(HEAD)
    raw[GUARD + n:].fill_(TAIL)
    inner = raw[GUARD:GUARD + n].view(t.dtype).view(t.shape) if n else raw[GUARD:GUARD].view(t.dtype).view(t.shape)
    if n:
        inner.copy_(t)
    _live.append((inner, n, label or f"{tuple(t.shape)} {t.dtype}"))
    return inner


def _bands_intact(inner: torch.Tensor, n: int) -> bool:
    raw = torch.empty(0, dtype=torch.uint8, device=inner.device).set_(inner.untyped_storage())
    assert raw.numel() == n + 2 * GUARD
    return bool((raw[:GUARD] == HEAD).all().item()) and bool((raw[GUARD + n:] == TAIL).all().item())


def check_and_release() -> int:
    """Checks every registered buffer still alive; then keeps only weak
    references (buffers a module-scoped fixture holds stay checked in later
    tests, the others are freed).  Returns the number of buffers checked."""
    torch.cuda.synchronize()
    bad, kept, checked = [], [], 0
    for ref, n, label in _live:
        inner = ref() if isinstance(ref, weakref.ref) else ref
        if inner is None:
            continue
        checked += 1
        if not _bands_intact(inner, n):
            bad.append(label)
        kept.append((weakref.ref(inner), n, label))
    _live[:] = kept
    assert not bad, f"guard bands overwritten around: {bad}"
    return checked


def install(monkeypatch) -> None:
    """Band every cache array and decode buffer the binding allocates."""
    from decode_attention_quantized_gb300 import kvq

    orig_init = kvq.QuantizedPagedCache.__init__
    orig_bufs = kvq.alloc_decode_buffers

    def init(self, *a, **kw):
        orig_init(self, *a, **kw)
        latent = self.v_codes is self.k_codes
        same_scale = self.v_scale is self.k_scale
        self.k_codes = guarded(self.k_codes, "k_codes")
        self.v_codes = self.k_codes if latent else guarded(self.v_codes, "v_codes")
        self.k_scale = guarded(self.k_scale, "k_scale")
        self.v_scale = self.k_scale if same_scale else guarded(self.v_scale, "v_scale")

    def bufs(cache, params):
        b = orig_bufs(cache, params)
        return kvq.DecodeBuffers(guarded(b.workspace, "workspace"), guarded(b.out, "out"),
                                 guarded(b.lse, "lse"))

    monkeypatch.setattr(kvq.QuantizedPagedCache, "__init__", init)
    monkeypatch.setattr(kvq, "alloc_decode_buffers", bufs)
