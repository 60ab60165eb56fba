"""CPU oracle for quantized paged-KV decode attention (test infrastructure).

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
import this module; the product path never does, and nothing here touches the
CUDA library.  The arithmetic lives in ``kvq_oracle.c`` (plain C11, fp64,
compiled with gcc by :func:`build`); this file marshals NumPy arrays into it
and adds an independent NumPy brute force for tiny inputs.

What it computes (the pages' statement of the method):
  * append -- per-row absmax quantisation ("kv-quant-attn", section "Method";
    onnxruntime PR #32515, Description: step max/127 for int8, max/7 for int4)
    or static PER_TENSOR / PER_CHANNEL scales (onnxruntime PR #29912, Summary
    of Changes, k_scale / v_scale), written to the slot that slot_mapping names;
    or PER_GROUP: the per-row rule applied to each run of group_size channels
    (the group-wise scaling the kv-quant-attn page lists under "Requirements
    and limits" as not done there).
  * attend -- dequantise every cached row, then fp64 softmax attention with the
    head sink rescale 1/(1+exp(s_h - lse)) (PR #29912, ApplyHeadSink), softcap,
    sliding window and causal drafts (PR #32515, speculative decode).

Cache layout (the library's data format, restated independently here):
codes uint8 [num_blocks, Hkv, block_size, Dp] with Dp = D (int8, e4m3) or
(D+1)//2 (int4, even channel in the low nibble); PER_ROW scales fp32
[num_blocks, Hkv, block_size]; PER_TENSOR one fp32; PER_CHANNEL fp32 [Hkv, D];
PER_GROUP fp32 [num_blocks, Hkv, block_size, D // group_size].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

INT8, FP8_E4M3, INT4 = 1, 2, 3
PER_ROW, PER_TENSOR, PER_CHANNEL, PER_GROUP = 1, 2, 3, 4
QMAX = {INT8: 127.0, INT4: 7.0, FP8_E4M3: 448.0}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkvq_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no FMA contraction, so x86 and Arm agree)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cache(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("k_mode", ctypes.c_int), ("v_mode", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("block_size", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("group_size", ctypes.c_int)]


class _Params(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("num_q_heads", ctypes.c_int), ("q_tokens", ctypes.c_int),
                ("max_blocks_per_seq", ctypes.c_int), ("sm_scale", ctypes.c_double),
                ("softcap", ctypes.c_double), ("window", ctypes.c_int), ("nsplit", ctypes.c_int)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_long
            L.orc_e4m3_encode_n.argtypes = [vp, vp, i64]
            L.orc_e4m3_decode_n.argtypes = [vp, vp, i64]
            L.orc_quantize_row.argtypes = [vp, i32, i32, i32, vp, vp, vp]
            L.orc_quantize_row_g.argtypes = [vp, i32, i32, i32, vp, i32, vp, vp]
            L.orc_append.argtypes = [ctypes.POINTER(_Cache), vp, vp, vp, i32]
            L.orc_append.restype = i32
            L.orc_dequant_seq.argtypes = [ctypes.POINTER(_Cache), vp, i32, i32, vp, vp]
            L.orc_attend.argtypes = [ctypes.POINTER(_Cache), ctypes.POINTER(_Params), vp, vp, vp, vp,
                                     vp, i32, vp, vp, i32]
            L.orc_attend.restype = i32
            L.orc_norm_rope.argtypes = [vp, i32, i32, i32, vp, ctypes.c_double, i32, i32, i32, vp, vp, i32,
                                        vp, i32, vp, vp]
            L.orc_norm_rope.restype = i32
            L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
            L.orc_f64_to_bf16.restype = ctypes.c_uint16
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------
# bf16 helpers (bf16 is carried as its uint16 bit pattern)
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(v: float) -> int:
    """Nearest bf16 (bit pattern) to a double, ties to even."""
    return int(lib().orc_f64_to_bf16(float(v)))


def norm_rope(x_bf16: np.ndarray, *, norm_weight=None, eps: float = 1e-6, rotary_dim: int = 0,
              rotary_offset: int = 0, interleaved: bool = False, cos=None, sin=None, positions=None,
              hadamard: bool = False, return_f64: bool = False):
    """QK-RMSNorm then RoPE on x [N, H, D] (bf16 bits) -> (bf16 bits, rows skipped)
    or, with return_f64, (bf16 bits, rows skipped, the values before rounding).

    onnxruntime PR #29912, Summary of Changes (q_norm_weight / k_norm_weight,
    qk_norm_epsilon default 1e-6, rotary_offset; QkNormRotaryTNH).  Per row:
    y = x / sqrt(mean(x^2) + eps) * w, then each rotated pair (a, b) ->
    (a cos - b sin, b cos + a sin) with cos / sin the tables' row for the
    token's position, then (hadamard) the orthonormal Walsh-Hadamard
    rotation (named as the follow-up to the int4 cache in onnxruntime PR
    #32515's stacked-change note); fp64 from the definitions, one bf16
    rounding.  eps is the fp32 value the library's descriptor carries.
    Tokens whose position is outside the tables are left zero and counted."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    N, H, D = x.shape
    out = np.zeros_like(x)
    out64 = np.zeros(x.shape, np.float64)
    w = None if norm_weight is None else np.ascontiguousarray(norm_weight, dtype=np.uint16)
    if rotary_dim > 0:
        cs = np.ascontiguousarray(cos, dtype=np.float32)
        sn = np.ascontiguousarray(sin, dtype=np.float32)
        pos = np.ascontiguousarray(positions, dtype=np.int64)
        max_pos = cs.shape[0]
    else:
        cs = sn = pos = None
        max_pos = 0
    bad = lib().orc_norm_rope(_ptr(x), N, H, D, _ptr(w), float(np.float32(eps)), int(rotary_dim),
                              int(rotary_offset), 1 if interleaved else 0, _ptr(cs), _ptr(sn), int(max_pos),
                              _ptr(pos), 1 if hadamard else 0, _ptr(out), _ptr(out64))
    if bad < 0:
        raise ValueError("norm_rope: bad shape")
    return (out, bad, out64) if return_f64 else (out, bad)


def row_bytes(dtype: int, D: int) -> int:
    return (D + 1) // 2 if dtype == INT4 else D


# ----------------------------------------------------------------------------
# codec
# ----------------------------------------------------------------------------

def e4m3_encode(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_n(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_decode(c: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().orc_e4m3_decode_n(_ptr(c), _ptr(out), c.size)
    return out


def quantize_row(x_bf16: np.ndarray, dtype: int, mode: int, static_scale=None, group_size: int = 0):
    """One row of D bf16 values -> (codes uint8 [Dp], scale): the row scale
    (PER_ROW), the D // group_size group scales as float32 (PER_GROUP), or
    None (static modes)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    D = x.size
    G = group_size if mode == PER_GROUP else D
    assert G > 0 and D % G == 0
    codes = np.zeros(row_bytes(dtype, D), dtype=np.uint8)
    sc = np.zeros(D // G, dtype=np.float32)
    ss = None if static_scale is None else np.ascontiguousarray(static_scale, dtype=np.float32)
    lib().orc_quantize_row_g(_ptr(x), D, dtype, mode, _ptr(ss), G, _ptr(codes), _ptr(sc))
    if mode == PER_GROUP:
        return codes, sc
    return codes, (float(sc[0]) if mode == PER_ROW else None)


def code_values(codes: np.ndarray, dtype: int, D: int) -> np.ndarray:
    """Code values of a row (or rows, last axis = Dp) as float64."""
    codes = np.asarray(codes, dtype=np.uint8)
    if dtype == INT8:
        return codes.view(np.int8).astype(np.float64)
    if dtype == INT4:
        lo = (codes & 0xF).astype(np.int16)
        hi = (codes >> 4).astype(np.int16)
        nib = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (-1,))[..., :D]
        return np.where(nib >= 8, nib - 16, nib).astype(np.float64)
    return e4m3_decode(codes)


# ----------------------------------------------------------------------------
# paged cache
# ----------------------------------------------------------------------------

class OracleCache:
    """Host copy of a quantized paged cache with the oracle's append/attend."""

    def __init__(self, dtype, k_mode, v_mode, num_blocks, block_size, num_kv_heads, head_dim,
                 k_static=None, v_static=None, latent=False, v_head_size=0, group_size=0):
        """latent: the absorbed-MLA layout of onnxruntime PR #29912 (kv_cache_layout
        LATENT, v_head_size): one cache, V read as the leading v_head_size
        channels of the same row that supplies K, with K's scales.
        group_size: channels per scale group of a PER_GROUP side (divides D)."""
        if PER_GROUP in (k_mode, v_mode):
            assert group_size > 0 and head_dim % group_size == 0
        self.group_size = int(group_size)
        self.latent = bool(latent)
        self.v_head_size = (v_head_size or head_dim) if latent else head_dim
        if latent:
            v_mode, v_static = k_mode, k_static
        self.dtype, self.k_mode, self.v_mode = dtype, k_mode, v_mode
        self.num_blocks, self.block_size = num_blocks, block_size
        self.num_kv_heads, self.head_dim = num_kv_heads, head_dim
        Dp = row_bytes(dtype, head_dim)
        shape = (num_blocks, num_kv_heads, block_size, Dp)
        self.k_codes = np.zeros(shape, dtype=np.uint8)
        self.v_codes = self.k_codes if latent else np.zeros(shape, dtype=np.uint8)

        def scale_arr(mode, static):
            if mode == PER_ROW:
                return np.zeros((num_blocks, num_kv_heads, block_size), dtype=np.float32)
            if mode == PER_GROUP:
                return np.zeros((num_blocks, num_kv_heads, block_size, head_dim // group_size), dtype=np.float32)
            if mode == PER_TENSOR:
                return np.ascontiguousarray(np.asarray(static, dtype=np.float32).reshape(1))
            return np.ascontiguousarray(np.asarray(static, dtype=np.float32).reshape(num_kv_heads, head_dim))

        self.k_scale = scale_arr(k_mode, k_static)
        self.v_scale = self.k_scale if latent else scale_arr(v_mode, v_static)

    def _struct(self):
        return _Cache(self.dtype, self.k_mode, self.v_mode, self.num_blocks, self.block_size,
                      self.num_kv_heads, self.head_dim, self.k_codes.ctypes.data, self.v_codes.ctypes.data,
                      self.k_scale.ctypes.data, self.v_scale.ctypes.data, self.group_size)

    def append(self, k_new_bf16: np.ndarray, v_new_bf16: np.ndarray, slot_mapping: np.ndarray) -> int:
        """k_new/v_new uint16 [N, Hkv, D] (bf16 bits); slot_mapping int64 [N]. Returns #bad slots."""
        k = np.ascontiguousarray(k_new_bf16, dtype=np.uint16)
        # latent: the V side shares the K arrays and rows (writing K twice, identically)
        v = k if self.latent else np.ascontiguousarray(v_new_bf16, dtype=np.uint16)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        st = self._struct()
        return lib().orc_append(ctypes.byref(st), _ptr(k), _ptr(v), _ptr(sm), int(sm.size))

    def dequant_seq(self, bt_row: np.ndarray, h: int, L: int):
        """fp64 dequantized K, V [L, D] of kv head h for a sequence's block-table row."""
        bt = np.ascontiguousarray(bt_row, dtype=np.int32)
        k = np.empty((L, self.head_dim), dtype=np.float64)
        v = np.empty((L, self.head_dim), dtype=np.float64)
        st = self._struct()
        lib().orc_dequant_seq(ctypes.byref(st), _ptr(bt), int(h), int(L), _ptr(k), _ptr(v))
        return k, v

    def attend(self, q_bf16, block_table, seq_lens, *, q_tokens=1, sm_scale=0.0, softcap=0.0,
               window=0, head_sink=None, rows=None, nsplit=1, nthreads=None):
        """q uint16 [B, T, Hq, D] bf16 bits.  Returns (out fp64, lse fp64).

        rows=None: out [B, T, Hq, D], lse [B, T, Hq]; else rows int32 [n, 3] of
        (b, tau, i) triples and out [n, D], lse [n]."""
        q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
        B, T, Hq, D = q.shape
        assert T == q_tokens and D == self.head_dim
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        sink = None if head_sink is None else np.ascontiguousarray(head_sink, dtype=np.float32)
        prm = _Params(B, Hq, T, bt.shape[1], float(sm_scale), float(softcap), int(window), int(nsplit))
        if rows is None:
            out = np.empty((B, T, Hq, D), dtype=np.float64)
            lse = np.empty((B, T, Hq), dtype=np.float64)
            r, nr = None, 0
        else:
            r = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
            nr = r.shape[0]
            out = np.empty((nr, D), dtype=np.float64)
            lse = np.empty((nr,), dtype=np.float64)
        nth = nthreads or os.cpu_count() or 1
        st = self._struct()
        rc = lib().orc_attend(ctypes.byref(st), ctypes.byref(prm), _ptr(bt), _ptr(sl), _ptr(q), _ptr(sink),
                              _ptr(r), nr, _ptr(out), _ptr(lse), int(nth))
        if rc != 0:
            raise ValueError(f"oracle attend rejected its inputs (code {rc})")
        if self.latent:  # V is the leading v_head_size channels of each row
            out = np.ascontiguousarray(out[..., :self.v_head_size])
        return out, lse


# ----------------------------------------------------------------------------
# NumPy brute force (tiny inputs): the definition of attention written as dense
# matrix algebra, independent of the C loop structure above.
# ----------------------------------------------------------------------------

def brute_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, seq_len: int, *, sm_scale=0.0,
                    softcap=0.0, window=0, head_sink=None):
    """q fp64 [T, Hq, D]; k, v fp64 [L, Hkv, D] (dequantized, L >= seq_len).

    Returns out [T, Hq, D], lse [T, Hq]."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    scale = sm_scale if sm_scale > 0 else 1.0 / np.sqrt(D)
    L = seq_len
    out = np.zeros((T, Hq, D))
    lse = np.full((T, Hq), -np.inf)
    j = np.arange(L)
    for tau in range(T):
        pos = L - T + tau
        keep = j <= pos
        if window > 0:
            keep &= j > pos - window
        if not keep.any():
            continue
        for i in range(Hq):
            h = i // G
            s = scale * (k[:L, h, :] @ q[tau, i, :])
            if softcap > 0:
                s = softcap * np.tanh(s / softcap)
            s = np.where(keep, s, -np.inf)
            m = s.max()
            w = np.exp(s - m)
            o = (w @ v[:L, h, :]) / w.sum()
            ls = m + np.log(w.sum())
            if head_sink is not None:
                o = o / (1.0 + np.exp(head_sink[i] - ls))
            out[tau, i] = o
            lse[tau, i] = ls
    return out, lse
