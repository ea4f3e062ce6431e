"""Oracle for the stack-wide paged packed-FP8 decode-attention step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product library
(``paged_fp8_kv_gk_gb300``) never does, and this package never imports it.

The arithmetic lives in ``gk_oracle.c`` (plain single-threaded C, fp64 for the
attention, IEEE fp32 without contraction for the quantised K path).  This file
only builds that C file with gcc and marshals numpy arrays to it.

Sources: "GPT-OSS-120B giga-kernel decode" (sections "Kernel contract" and
"KV-cache layout"), the OCP 8-bit floating point specification (E4M3), and the
plain definition of scaled dot-product attention with rotary embeddings.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gk_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgk_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile gk_oracle.c into a shared library (gcc); returns its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Shape(ctypes.Structure):
    """ora_shape; k_layout 0 = packed K view, 1 = unpacked K (laid out like V)."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "batch", "num_q_heads", "num_kv_heads", "head_dim",
        "block_size", "num_blocks", "window", "max_blocks_full", "max_blocks_swa", "k_layout")]


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            L.ora_e4m3_decode.restype = ctypes.c_double
            L.ora_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.ora_e4m3_encode.restype = ctypes.c_uint8
            L.ora_e4m3_encode.argtypes = [ctypes.c_float]
            L.ora_e4m3_encode_array.argtypes = [vp, vp, i64]
            L.ora_e4m3_decode_array.argtypes = [vp, vp, i64]
            L.ora_round_bf16.restype = ctypes.c_double
            L.ora_round_bf16.argtypes = [ctypes.c_double]
            L.ora_round_bf16_array.argtypes = [vp, vp, i64]
            L.ora_k_offset.restype = i64
            L.ora_k_offset.argtypes = [i32, i32, i32, i64, i32, i32, i32]
            L.ora_v_offset.restype = i64
            L.ora_v_offset.argtypes = [i32, i32, i32, i64, i32, i32, i32]
            L.ora_rope_f32.argtypes = [vp, vp, vp, i32, vp]
            L.ora_rope_f64.argtypes = [vp, vp, vp, i32, vp]
            L.ora_kv_append.restype = ctypes.c_int
            L.ora_kv_append.argtypes = [ctypes.POINTER(Shape)] + [vp] * 11
            L.ora_decode_attn_stack.restype = ctypes.c_int
            L.ora_decode_attn_stack.argtypes = [ctypes.POINTER(Shape)] + [vp] * 14
            L.ora_attn_one_ex.restype = ctypes.c_int
            L.ora_attn_one_ex.argtypes = ([ctypes.POINTER(Shape)] + [vp] * 13
                                          + [i32, i32, i32, i32, vp])
            L.ora_kv_regions.restype = i32
            L.ora_kv_regions.argtypes = [i32, vp, vp, vp]
            L.ora_kv_ingest.restype = i64
            L.ora_kv_ingest.argtypes = [vp, vp, i32, i64, vp, vp, i64, vp]
            L.ora_di_blocks.restype = None
            L.ora_di_blocks.argtypes = [i64, i32, i32, ctypes.POINTER(ctypes.c_int64),
                                        ctypes.POINTER(ctypes.c_int64),
                                        ctypes.POINTER(ctypes.c_int64)]
            _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def _ptr_array(arrs):
    arr_t = ctypes.c_void_p * len(arrs)
    return arr_t(*[a.ctypes.data for a in arrs])


# ---------------------------------------------------------------- E4M3 codec
def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code (ties to even, saturating at +-448; NaN -> 0x7F)."""
    x = _c(np.asarray(x, dtype=np.float32), np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().ora_e4m3_encode_array(_p(x), _p(out), x.size)
    return out


def e4m3_decode(c) -> np.ndarray:
    c = _c(np.asarray(c, dtype=np.uint8), np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().ora_e4m3_decode_array(_p(c), _p(out), c.size)
    return out


def round_bf16(x) -> np.ndarray:
    x = _c(np.asarray(x, dtype=np.float64), np.float64)
    out = np.empty(x.shape, np.float64)
    lib().ora_round_bf16_array(_p(x), _p(out), x.size)
    return out


# ---------------------------------------------------------------- layout
def k_offset(Hkv, B, D, pb, h, t, e) -> int:
    return lib().ora_k_offset(Hkv, B, D, pb, h, t, e)


def v_offset(Hkv, B, D, pb, h, t, e) -> int:
    return lib().ora_v_offset(Hkv, B, D, pb, h, t, e)


# ---------------------------------------------------------------- RoPE
def rope_f32(x, cos, sin) -> np.ndarray:
    x = _c(np.asarray(x, np.float32), np.float32)
    cos = _c(np.asarray(cos, np.float32), np.float32)
    sin = _c(np.asarray(sin, np.float32), np.float32)
    out = np.empty_like(x)
    lib().ora_rope_f32(_p(x), _p(cos), _p(sin), x.shape[-1], _p(out))
    return out


def rope_f64(x, cos, sin) -> np.ndarray:
    x = _c(np.asarray(x, np.float64), np.float64)
    cos = _c(np.asarray(cos, np.float32), np.float32)
    sin = _c(np.asarray(sin, np.float32), np.float32)
    out = np.empty_like(x)
    lib().ora_rope_f64(_p(x), _p(cos), _p(sin), x.shape[-1], _p(out))
    return out


# ---------------------------------------------------------------- the step
def make_shape(**kw) -> Shape:
    return Shape(**{k: int(v) for k, v in kw.items()})


def kv_append(shape: Shape, k_new, v_new, cos, sin, k_scale, v_scale, upd_full, upd_swa,
              active, k_bufs, v_bufs) -> int:
    """Quantise and write the new token's K (packed, or unpacked when
    shape.k_layout == 1) and V (plain) into the group buffers, in place.
    k_new/v_new are bf16 bit patterns (uint16)."""
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    cos = _c(cos, np.float32)
    sin = _c(sin, np.float32)
    k_scale = _c(k_scale, np.float32)
    v_scale = _c(v_scale, np.float32)
    upd_full = _c(upd_full, np.int32)
    upd_swa = _c(upd_swa, np.int32)
    active = _c(active, np.uint8)
    for a in list(k_bufs) + list(v_bufs):
        if not (a.flags["C_CONTIGUOUS"] and a.dtype == np.uint8 and a.flags["WRITEABLE"]):
            raise TypeError("group buffers must be writeable contiguous uint8 arrays")
    kp, vp_ = _ptr_array(k_bufs), _ptr_array(v_bufs)
    return lib().ora_kv_append(ctypes.byref(shape), _p(k_new), _p(v_new), _p(cos), _p(sin),
                               _p(k_scale), _p(v_scale), _p(upd_full), _p(upd_swa), _p(active),
                               ctypes.cast(kp, ctypes.c_void_p), ctypes.cast(vp_, ctypes.c_void_p))


def decode_attn_stack(shape: Shape, q, k_bufs, v_bufs, k_scale, v_scale, cos, sin, bt_full,
                      bt_swa, pos, pos_w, active, sinks=None):
    """Whole-stack decode attention in fp64; returns (out [NL,Bt,Hq,D] float64, status).
    sinks: optional [NL, Hq] attention-sink logits (natural units)."""
    q = _c(q, np.uint16)
    k_bufs = [_c(a, np.uint8) for a in k_bufs]
    v_bufs = [_c(a, np.uint8) for a in v_bufs]
    args = [_c(k_scale, np.float32), _c(v_scale, np.float32), _c(cos, np.float32),
            _c(sin, np.float32), _c(bt_full, np.int32), _c(bt_swa, np.int32),
            _c(pos, np.int32), _c(pos_w, np.int32), _c(active, np.uint8)]
    out = np.zeros((shape.num_layers, shape.batch, shape.num_q_heads, shape.head_dim), np.float64)
    kp, vp_ = _ptr_array(k_bufs), _ptr_array(v_bufs)
    sk = None if sinks is None else _c(np.asarray(sinks, np.float32), np.float32)
    st = lib().ora_decode_attn_stack(ctypes.byref(shape), _p(q), ctypes.cast(kp, ctypes.c_void_p),
                                     ctypes.cast(vp_, ctypes.c_void_p), *[_p(a) for a in args],
                                     None if sk is None else _p(sk), _p(out))
    return out, st


def attn_one(shape: Shape, q, kbuf, vbuf, k_scale, v_scale, cos, sin, bt_full, bt_swa, pos,
             pos_w, active, layer, b, kvh, nsplit=1, sinks=None):
    """One (layer, sequence, kv head): returns (out [G, D] float64, status).
    ``kbuf``/``vbuf`` are the K and V halves of group buffer layer // 2."""
    G = shape.num_q_heads // shape.num_kv_heads
    arrs = [_c(q, np.uint16), _c(kbuf, np.uint8), _c(vbuf, np.uint8), _c(k_scale, np.float32),
            _c(v_scale, np.float32), _c(cos, np.float32), _c(sin, np.float32),
            _c(bt_full, np.int32), _c(bt_swa, np.int32), _c(pos, np.int32), _c(pos_w, np.int32),
            _c(active, np.uint8)]
    out = np.zeros((G, shape.head_dim), np.float64)
    sk = None if sinks is None else _c(np.asarray(sinks, np.float32), np.float32)
    st = lib().ora_attn_one_ex(ctypes.byref(shape), *[_p(a) for a in arrs],
                               None if sk is None else _p(sk), layer, b, kvh, nsplit, _p(out))
    return out, st


# ---------------------------------------------------------------- DI landing
def kv_regions(bases_k, bases_v) -> list:
    """Per-layer K/V base addresses -> the de-duplicated region bases, in order."""
    k = _c(np.asarray(bases_k, np.uint64), np.uint64)
    v = _c(np.asarray(bases_v, np.uint64), np.uint64)
    out = np.zeros(2 * k.size, np.uint64)
    n = lib().ora_kv_regions(k.size, _p(k), _p(v), _p(out))
    return [int(x) for x in out[:n]]


def kv_ingest(regions, block_len: int, dst_region, dst_block, src) -> int:
    """Landing copy into ``regions`` (writeable contiguous uint8 arrays, each a
    whole number of blocks), in place; returns the descriptors skipped."""
    for a in regions:
        if not (a.flags["C_CONTIGUOUS"] and a.dtype == np.uint8 and a.flags["WRITEABLE"]):
            raise TypeError("regions must be writeable contiguous uint8 arrays")
    nblocks = np.array([a.size // block_len for a in regions], np.int64)
    dr = _c(np.asarray(dst_region, np.int32), np.int32)
    db = _c(np.asarray(dst_block, np.int32), np.int32)
    src = _c(np.asarray(src, np.uint8).reshape(-1), np.uint8)
    ptrs = _ptr_array(regions)
    return int(lib().ora_kv_ingest(ctypes.cast(ptrs, ctypes.c_void_p), _p(nblocks), len(regions),
                                   int(block_len), _p(dr), _p(db), dr.size, _p(src)))


def di_blocks(num_tokens: int, block_size: int, window: int):
    """(full_count, swa_first, swa_count) for a prompt of num_tokens tokens."""
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    lib().ora_di_blocks(int(num_tokens), int(block_size), int(window), ctypes.byref(a),
                        ctypes.byref(b), ctypes.byref(c))
    return a.value, b.value, c.value
