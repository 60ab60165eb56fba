"""Python binding of the kvq C ABI (include/kvq.h): argument marshalling only.

Every step of the path runs in the CUDA library ``lib/libkvq.so``; this module
passes raw device pointers and the current torch stream through ctypes.  It
never computes anything itself and there is no fallback: when the library is
missing, ``load()`` raises.  Build it with ``__graft_entry__.build()`` (or
``python -m decode_attention_quantized_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

from .build import LIB_PATH

INT8, FP8_E4M3, INT4 = 1, 2, 3
LAYOUT_SEPARATE, LAYOUT_LATENT = 0, 1
PER_ROW, PER_TENSOR, PER_CHANNEL, PER_GROUP = 1, 2, 3, 4
DECODE_EARLY_INPUTS, DECODE_NO_TCGEN05, DECODE_EARLY_CACHE = 0x1, 0x2, 0x4  # kvq_decode_params.flags
DEVERR_SLOT, DEVERR_BLOCK_ID, DEVERR_SEQ_LEN, DEVERR_TIMEOUT, DEVERR_POSITION = 0x1, 0x2, 0x4, 0x8, 0x10
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace too small", 4: "CUDA error",
          5: "device timeout"}


class KvqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {STATUS.get(status, status)} (status {status})")
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("k_mode", ctypes.c_int32), ("v_mode", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("layout", ctypes.c_int32), ("v_head_size", ctypes.c_int32), ("group_size", ctypes.c_int32)]


class DecodeParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("q_tokens", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("sm_scale", ctypes.c_float), ("softcap", ctypes.c_float), ("window", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


class NormRopeDesc(ctypes.Structure):
    _fields_ = [("norm_weight", ctypes.c_void_p), ("norm_eps", ctypes.c_float), ("rotary_dim", ctypes.c_int32),
                ("rotary_offset", ctypes.c_int32), ("rotary_interleaved", ctypes.c_int32),
                ("cos_cache", ctypes.c_void_p), ("sin_cache", ctypes.c_void_p), ("max_position", ctypes.c_int32),
                ("hadamard", ctypes.c_int32)]


# every exported entry point of include/kvq.h with its ctypes signature
_VP, _I32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
SIGNATURES = {
    "kvq_status_string": (ctypes.c_char_p, [_I32]),
    "kvq_append": (_I32, [ctypes.POINTER(CacheDesc), _VP, _VP, _VP, _I32, _VP]),
    "kvq_decode_workspace_size": (_I32, [ctypes.POINTER(CacheDesc), ctypes.POINTER(DecodeParams),
                                         ctypes.POINTER(_SZ)]),
    "kvq_decode": (_I32, [ctypes.POINTER(CacheDesc), ctypes.POINTER(DecodeParams), _VP, _VP, _VP, _VP, _SZ, _VP]),
    "kvq_combine": (_I32, [ctypes.POINTER(CacheDesc), ctypes.POINTER(DecodeParams), _VP, _SZ, _VP, _VP, _VP,
                           _VP]),
    "kvq_check_wait_timeout": (_I32, [ctypes.c_uint32, _VP]),
    "kvq_get_device_error": (_I32, [ctypes.POINTER(ctypes.c_uint32), _I32, _VP]),
    "kvq_norm_rope_apply": (_I32, [ctypes.POINTER(NormRopeDesc), _VP, _VP, _VP, _I32, _I32, _I32, _VP]),
    "kvq_prefill_workspace_size": (_I32, [ctypes.POINTER(CacheDesc), ctypes.POINTER(DecodeParams),
                                          ctypes.POINTER(_SZ)]),
    "kvq_prefill": (_I32, [ctypes.POINTER(CacheDesc), ctypes.POINTER(DecodeParams), _VP, _VP, _VP, _VP, _VP, _VP,
                           _VP, _SZ, _VP]),
    "kvq_append_norm_rope": (_I32, [ctypes.POINTER(CacheDesc), ctypes.POINTER(NormRopeDesc), _VP, _VP, _VP, _VP,
                                    _I32, _VP]),
    "kvq_attend_noalloc": (_I32, [ctypes.POINTER(CacheDesc), ctypes.POINTER(DecodeParams), _VP, _VP, _VP, _VP, _VP,
                                  _VP, _VP]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load libkvq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first (__graft_entry__.build())")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise KvqError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> Optional[ctypes.c_void_p]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---------------------------------------------------------------------------
# cache object (one per layer) holding caller-owned torch device tensors
# ---------------------------------------------------------------------------

class QuantizedPagedCache:
    """A quantized paged KV cache in device memory (torch allocates it).

    codes uint8 [num_blocks, Hkv, block_size, Dp]; PER_ROW scales fp32
    [num_blocks, Hkv, block_size]; PER_GROUP scales fp32 [num_blocks, Hkv,
    block_size, D // group_size]; static scales as given ([1] or [Hkv, D])."""

    def __init__(self, dtype: int, k_mode: int, v_mode: int, num_blocks: int, block_size: int,
                 num_kv_heads: int, head_dim: int, *, device="cuda", k_static: Optional[torch.Tensor] = None,
                 v_static: Optional[torch.Tensor] = None, latent: bool = False, v_head_size: int = 0,
                 group_size: int = 0):
        """latent: one cache (absorbed MLA); V is the leading v_head_size channels
        of each K row, with K's scales, and no V arrays are allocated.
        group_size: channels per scale group of a PER_GROUP side (32, 64, 128)."""
        self.layout = LAYOUT_LATENT if latent else LAYOUT_SEPARATE
        self.v_head_size = v_head_size
        self.group_size = int(group_size)
        if latent:
            v_mode = k_mode
        self.dtype, self.k_mode, self.v_mode = dtype, k_mode, v_mode
        self.num_blocks, self.block_size = num_blocks, block_size
        self.num_kv_heads, self.head_dim = num_kv_heads, head_dim
        dp = head_dim // 2 if dtype == INT4 else head_dim
        shape = (num_blocks, num_kv_heads, block_size, dp)
        self.k_codes = torch.zeros(shape, dtype=torch.uint8, device=device)
        self.v_codes = self.k_codes if latent else torch.zeros(shape, dtype=torch.uint8, device=device)

        def scales(mode, static):
            if mode == PER_ROW:
                return torch.zeros((num_blocks, num_kv_heads, block_size), dtype=torch.float32, device=device)
            if mode == PER_GROUP:
                if group_size <= 0 or head_dim % group_size:
                    raise ValueError("PER_GROUP needs a group_size dividing head_dim")
                return torch.zeros((num_blocks, num_kv_heads, block_size, head_dim // group_size),
                                   dtype=torch.float32, device=device)
            if static is None:
                raise ValueError("static scale mode needs a scale tensor")
            want = (1,) if mode == PER_TENSOR else (num_kv_heads, head_dim)
            return static.to(device=device, dtype=torch.float32).reshape(want).contiguous()

        self.k_scale = scales(k_mode, k_static)
        self.v_scale = self.k_scale if latent else scales(v_mode, v_static)

    def desc(self) -> CacheDesc:
        return CacheDesc(self.dtype, self.k_mode, self.v_mode, self.num_blocks, self.block_size,
                         self.num_kv_heads, self.head_dim, self.k_codes.data_ptr(), self.v_codes.data_ptr(),
                         self.k_scale.data_ptr(), self.v_scale.data_ptr(), self.layout, self.v_head_size,
                         self.group_size)

    @property
    def out_dim(self) -> int:
        """Channels of an output row: head_dim, or v_head_size for a LATENT cache."""
        return (self.v_head_size or self.head_dim) if self.layout == LAYOUT_LATENT else self.head_dim


def make_params(batch, num_q_heads, q_tokens, max_blocks_per_seq, *, max_seq_len=0, sm_scale=0.0, softcap=0.0,
                window=0, flags=0) -> DecodeParams:
    """flags: DECODE_EARLY_INPUTS (q, block table, seq_lens and static scales are
    not written by the kernel enqueued just before kvq_decode), with it
    DECODE_EARLY_CACHE (that kernel writes no cache row but the step's new
    tokens'), and / or DECODE_NO_TCGEN05 (17..64 query rows per kv head on the
    mma.sync layouts)."""
    return DecodeParams(int(batch), int(num_q_heads), int(q_tokens), int(max_blocks_per_seq), int(max_seq_len),
                        float(sm_scale), float(softcap), int(window), int(flags))


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def kvq_append(cache: QuantizedPagedCache, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
               stream=None):
    """k_new, v_new bf16 [N, Hkv, D]; slot_mapping int64 [N] (device)."""
    d = cache.desc()
    _check("kvq_append", load().kvq_append(ctypes.byref(d), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                           int(slot_mapping.numel()), _stream(stream)))


@dataclass
class NormRope:
    """The QK-RMSNorm + RoPE prologue (kvq_norm_rope in kvq.h); tensors on the device.
    norm_weight bf16 [D] or None; cos / sin fp32 [max_position, rotary_dim / 2]."""
    norm_weight: Optional[torch.Tensor] = None
    eps: float = 1e-6
    rotary_dim: int = 0
    rotary_offset: int = 0
    interleaved: bool = False
    cos: Optional[torch.Tensor] = None
    sin: Optional[torch.Tensor] = None
    hadamard: bool = False

    def desc(self) -> NormRopeDesc:
        return NormRopeDesc(None if self.norm_weight is None else self.norm_weight.data_ptr(), float(self.eps),
                            int(self.rotary_dim), int(self.rotary_offset), 1 if self.interleaved else 0,
                            None if self.cos is None else self.cos.data_ptr(),
                            None if self.sin is None else self.sin.data_ptr(),
                            0 if self.cos is None else int(self.cos.shape[0]), 1 if self.hadamard else 0)


def kvq_norm_rope_apply(pro: NormRope, x: torch.Tensor, y: torch.Tensor, positions: Optional[torch.Tensor],
                        stream=None):
    """x, y bf16 [N, H, D] (y may be x); positions int64 [N]."""
    N, H, D = x.shape
    d = pro.desc()
    _check("kvq_norm_rope_apply", load().kvq_norm_rope_apply(ctypes.byref(d), _ptr(x), _ptr(y), _ptr(positions),
                                                             N, H, D, _stream(stream)))


def kvq_append_norm_rope(cache: QuantizedPagedCache, pro: NormRope, k_new: torch.Tensor, v_new: torch.Tensor,
                         slot_mapping: torch.Tensor, positions: Optional[torch.Tensor], stream=None):
    d, p = cache.desc(), pro.desc()
    _check("kvq_append_norm_rope", load().kvq_append_norm_rope(ctypes.byref(d), ctypes.byref(p), _ptr(k_new),
                                                               _ptr(v_new), _ptr(slot_mapping), _ptr(positions),
                                                               k_new.shape[0], _stream(stream)))


def kvq_prefill_workspace_size(cache: QuantizedPagedCache, params: DecodeParams) -> int:
    d = cache.desc()
    n = ctypes.c_size_t(0)
    _check("kvq_prefill_workspace_size", load().kvq_prefill_workspace_size(ctypes.byref(d), ctypes.byref(params),
                                                                           ctypes.byref(n)))
    return n.value


def kvq_prefill(cache: QuantizedPagedCache, params: DecodeParams, q: torch.Tensor, block_table: torch.Tensor,
                seq_lens: torch.Tensor, head_sink: Optional[torch.Tensor], out: torch.Tensor,
                lse_out: Optional[torch.Tensor], workspace: torch.Tensor, stream=None):
    """q, out bf16 [B, C, Hq, D] with C = params.q_tokens; lse_out fp32 [B, C, Hq] or None."""
    d = cache.desc()
    _check("kvq_prefill", load().kvq_prefill(ctypes.byref(d), ctypes.byref(params), _ptr(q), _ptr(block_table),
                                             _ptr(seq_lens), _ptr(head_sink), _ptr(out), _ptr(lse_out),
                                             _ptr(workspace), workspace.numel() * workspace.element_size(),
                                             _stream(stream)))


def kvq_decode_workspace_size(cache: QuantizedPagedCache, params: DecodeParams) -> int:
    n = ctypes.c_size_t(0)
    d = cache.desc()
    _check("kvq_decode_workspace_size",
           load().kvq_decode_workspace_size(ctypes.byref(d), ctypes.byref(params), ctypes.byref(n)))
    return n.value


def kvq_decode(cache: QuantizedPagedCache, params: DecodeParams, q: torch.Tensor, block_table: torch.Tensor,
               seq_lens: torch.Tensor, workspace: torch.Tensor, stream=None):
    d = cache.desc()
    _check("kvq_decode", load().kvq_decode(ctypes.byref(d), ctypes.byref(params), _ptr(q), _ptr(block_table),
                                           _ptr(seq_lens), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream(stream)))


def kvq_combine(cache: QuantizedPagedCache, params: DecodeParams, workspace: torch.Tensor,
                head_sink: Optional[torch.Tensor], out: torch.Tensor, lse_out: Optional[torch.Tensor] = None,
                stream=None):
    d = cache.desc()
    _check("kvq_combine", load().kvq_combine(ctypes.byref(d), ctypes.byref(params), _ptr(workspace),
                                             workspace.numel() * workspace.element_size(), _ptr(head_sink),
                                             _ptr(out), _ptr(lse_out), _stream(stream)))


def kvq_check_wait_timeout(limit_us: int, stream=None):
    """Launch the bounded-wait check: one wait on a barrier nothing arrives on
    gives up after limit_us and sets DEVERR_TIMEOUT (read it with
    kvq_get_device_error)."""
    _check("kvq_check_wait_timeout", load().kvq_check_wait_timeout(int(limit_us), _stream(stream)))


def kvq_get_device_error(clear: bool = True, stream=None) -> int:
    """Synchronizes the stream and returns the KVQ_DEVERR_* flag word."""
    v = ctypes.c_uint32(0)
    st = load().kvq_get_device_error(ctypes.byref(v), 1 if clear else 0, _stream(stream))
    if st not in (0, 5):
        raise KvqError("kvq_get_device_error", st)
    return v.value


def kvq_attend_noalloc(cache: QuantizedPagedCache, params: DecodeParams, q: torch.Tensor, block_table: torch.Tensor,
                       seq_lens: torch.Tensor, head_sink: Optional[torch.Tensor], out: torch.Tensor,
                       lse_out: Optional[torch.Tensor] = None, stream=None):
    """Decode + combine with the library's fixed device scratch (no workspace
    argument, nothing allocated by the library)."""
    d = cache.desc()
    _check("kvq_attend_noalloc", load().kvq_attend_noalloc(ctypes.byref(d), ctypes.byref(params), _ptr(q),
                                                           _ptr(block_table), _ptr(seq_lens), _ptr(head_sink),
                                                           _ptr(out), _ptr(lse_out), _stream(stream)))


@dataclass
class DecodeBuffers:
    workspace: torch.Tensor
    out: torch.Tensor
    lse: torch.Tensor


def alloc_decode_buffers(cache: QuantizedPagedCache, params: DecodeParams) -> DecodeBuffers:
    """Caller-side allocation of the workspace (256-byte aligned) and outputs."""
    nbytes = kvq_decode_workspace_size(cache, params)
    ws = torch.empty(max(nbytes, 256) // 4 + 64, dtype=torch.int32, device=cache.k_codes.device)
    shape = (params.batch, params.q_tokens, params.num_q_heads, cache.out_dim)
    out = torch.empty(shape, dtype=torch.bfloat16, device=cache.k_codes.device)
    lse = torch.empty(shape[:3], dtype=torch.float32, device=cache.k_codes.device)
    return DecodeBuffers(ws, out, lse)


def decode_step(cache: QuantizedPagedCache, params: DecodeParams, q, block_table, seq_lens, bufs: DecodeBuffers,
                head_sink=None, stream=None):
    """kvq_decode followed by kvq_combine into bufs.out / bufs.lse."""
    kvq_decode(cache, params, q, block_table, seq_lens, bufs.workspace, stream)
    kvq_combine(cache, params, bufs.workspace, head_sink, bufs.out, bufs.lse, stream)
    return bufs.out, bufs.lse
