"""Python binding of the GB300 stack-wide paged-FP8 decode-attention library.

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of ``libgk.so`` (sources in ``csrc/``, ABI in ``include/gk.h``).  There
is no CPU fallback: if the library cannot be built or loaded, or a tensor is not
on a CUDA device, the calls raise.

The functions carry the C names: ``gk_kv_append``, ``gk_decode_attn_stack``,
``gk_decode_step``, ``gk_decode_attn_stack_static``,
``gk_attn_workspace_bytes``, ``gk_attn_workspace_min_bytes``,
``gk_e4m3_quantize``, ``gk_kv_budget``, ``gk_kv_regions``, ``gk_kv_ingest``,
``gk_di_blocks``, ``gk_read_device_error``, ``gk_status_str``, ``gk_abi_version``.  Tensors are torch tensors; the stream defaults to torch's
current stream on the tensors' device.  The cache is a ``KvCache``: per-group
K and V buffers or stacked ``K_cache`` / ``V_cache``, exactly one of the two,
with packed-ness read from the K tensors' rank as the "GPT-OSS-120B giga-kernel
decode" page describes (section "KV-cache layout": ``k.dim() == v.dim() + 1``).
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional, Sequence

from . import build as _build

GK_OK, GK_ERR_INVALID_ARG, GK_ERR_UNSUPPORTED, GK_ERR_WORKSPACE, GK_ERR_CUDA, \
    GK_ERR_DEVICE_BOUNDS, GK_ERR_BUDGET = range(7)
GK_DEVERR_SLOT, GK_DEVERR_BLOCK, GK_DEVERR_POS, GK_DEVERR_TIMEOUT, GK_DEVERR_PLAN, \
    GK_DEVERR_INGEST = 0x1, 0x2, 0x4, 0x8, 0x10, 0x20
GK_K_PACKED, GK_K_PLAIN = 0, 1

HEADER = os.path.join(_build.INCLUDE, "gk.h")

_lock = threading.Lock()
_lib = None


class GkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gk_status_str(status)} ({status})")


class Shape(ctypes.Structure):
    """gk_shape: all int32."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "batch", "num_q_heads", "num_kv_heads", "head_dim",
        "block_size", "num_blocks", "window", "max_blocks_full", "max_blocks_swa")]

    @classmethod
    def make(cls, **kw) -> "Shape":
        return cls(**{k: int(v) for k, v in kw.items()})


class KvRegion(ctypes.Structure):
    """gk_kv_region: one DI landing region (a group buffer's K or V half)."""
    _fields_ = [("base", ctypes.c_void_p), ("length", ctypes.c_uint64),
                ("block_len", ctypes.c_uint64)]


class KvCacheC(ctypes.Structure):
    """gk_kv_cache."""
    _fields_ = [("k_bufs", ctypes.c_void_p), ("v_bufs", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("k_layout", ctypes.c_int32)]


class KvCache:
    """The KV cache in one of its two forms ("Kernel contract": per-group
    buffers or stacked K_cache / V_cache, exactly one present).

    per-group: ``k_bufs[j]``, ``v_bufs[j]`` are group buffer j's K and V halves:
      V ``[num_blocks, kv, block, d]`` uint8, K the same (unpacked) or the packed
      view ``[num_blocks, kv, block // 2, d, 2]``;
    stacked: ``k_cache``, ``v_cache`` with a leading group axis (``[G, ...]``).
    ``k_layout`` is read from the ranks (``k.dim() == v.dim() + 1`` means packed);
    it must be given only when the buffers are raw device addresses (ints).
    Holds references to the tensors and the pointer arrays it hands the library.
    """

    def __init__(self, k_bufs=None, v_bufs=None, k_cache=None, v_cache=None,
                 k_layout: Optional[int] = None):
        per_group = k_bufs is not None or v_bufs is not None
        stacked = k_cache is not None or v_cache is not None
        if per_group == stacked:
            raise ValueError("pass exactly one KV form: (k_bufs, v_bufs) or (k_cache, v_cache)")
        if per_group and (k_bufs is None or v_bufs is None or len(k_bufs) != len(v_bufs)):
            raise ValueError("k_bufs and v_bufs must both be given, one per group buffer")
        if stacked and (k_cache is None or v_cache is None):
            raise ValueError("k_cache and v_cache must both be given")
        ks = list(k_bufs) if per_group else [k_cache]
        vs = list(v_bufs) if per_group else [v_cache]
        tensors = [(k, v) for k, v in zip(ks, vs) if not isinstance(k, int)
                   and not isinstance(v, int)]
        if tensors:
            inferred = {infer_k_layout(k, v) for k, v in tensors}
            if len(inferred) != 1:
                raise ValueError("all group buffers must have one K layout")
            inferred = inferred.pop()
            if k_layout is not None and k_layout != inferred:
                raise ValueError("k_layout disagrees with the K tensors' rank")
            k_layout = inferred
        elif k_layout is None:
            raise ValueError("k_layout is required for raw device addresses")
        if k_layout not in (GK_K_PACKED, GK_K_PLAIN):
            raise ValueError(f"k_layout {k_layout}")
        self.per_group = per_group
        self.k_layout = int(k_layout)
        self._keep = (ks, vs)
        c = KvCacheC(k_layout=self.k_layout)
        if per_group:
            self._k_arr = _ptr_array(ks, "k_bufs")
            self._v_arr = _ptr_array(vs, "v_bufs")
            c.k_bufs = ctypes.cast(self._k_arr, ctypes.c_void_p)
            c.v_bufs = ctypes.cast(self._v_arr, ctypes.c_void_p)
        else:
            c.k_cache = _ptr(k_cache, None, "k_cache")
            c.v_cache = _ptr(v_cache, None, "v_cache")
        self.c = c

    def check(self, shape) -> None:
        """Buffer sizes against the shape (the C ABI cannot see them)."""
        sh = _as_shape(shape)
        groups = sh.num_layers // 2
        half = sh.num_blocks * sh.num_kv_heads * sh.block_size * sh.head_dim
        ks, vs = self._keep
        if self.per_group and len(ks) < groups:
            raise ValueError(f"{len(ks)} group buffers for {sh.num_layers} layers")
        want = half if self.per_group else groups * half
        for t in ks + vs:
            if not isinstance(t, int) and t.numel() * t.element_size() < want:
                raise ValueError(f"a cache buffer holds {t.numel() * t.element_size()} bytes, "
                                 f"the shape needs {want}")

    def param(self):
        return ctypes.byref(self.c)


def infer_k_layout(k, v) -> int:
    """Packed-ness from the ranks, as the page's bind step infers it
    (``k.dim() == v.dim() + 1``: the packed view's extra trailing axis of 2)."""
    kd, vd = k.dim(), v.dim()
    if kd == vd + 1 and k.shape[-1] == 2:
        return GK_K_PACKED
    if kd == vd:
        return GK_K_PLAIN
    raise ValueError(f"K shape {tuple(k.shape)} vs V shape {tuple(v.shape)}: "
                     "neither the packed view nor the plain layout")


def kv_from_group_buffers(bufs: Sequence, k_layout: int = GK_K_PACKED) -> KvCache:
    """Group buffers [2, num_blocks, kv, block, d] (K half, then V half) -> the
    per-group KvCache, K viewed packed ([.., block // 2, d, 2]) or plain."""
    ks = []
    for b in bufs:
        k = b[0]
        if k_layout == GK_K_PACKED:
            nb, kv, B, D = k.shape
            k = k.view(nb, kv, B // 2, D, 2)
        ks.append(k)
    return KvCache(k_bufs=ks, v_bufs=[b[1] for b in bufs])


def kv_stacked(k_cache, v_cache) -> KvCache:
    """Stacked K_cache / V_cache ([G, num_blocks, kv, block, d], K optionally
    as the packed view [G, num_blocks, kv, block // 2, d, 2])."""
    return KvCache(k_cache=k_cache, v_cache=v_cache)


def _kv(kv, shape) -> "ctypes._CArgObject":
    if not isinstance(kv, KvCache):
        raise TypeError("kv must be a KvCache (kv_from_group_buffers, kv_stacked)")
    kv.check(shape)
    return kv.param()


def declared_functions() -> list:
    """Names of the functions include/gk.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gk_[a-z0-9_]+)\s*\(", text)))


def lib(build_if_needed: bool = True) -> ctypes.CDLL:
    """Load libgk.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_needed else _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: run paged_fp8_kv_gk_gb300.build.build()")
            L = ctypes.CDLL(path)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            sp = ctypes.POINTER(Shape)
            L.gk_status_str.restype = ctypes.c_char_p
            L.gk_status_str.argtypes = [ctypes.c_int]
            L.gk_abi_version.restype = i32
            L.gk_abi_version.argtypes = []
            L.gk_kv_append.restype = ctypes.c_int
            L.gk_kv_append.argtypes = [sp] + [vp] * 11
            L.gk_attn_workspace_bytes.restype = sz
            L.gk_attn_workspace_bytes.argtypes = [sp, vp]
            L.gk_attn_workspace_min_bytes.restype = sz
            L.gk_attn_workspace_min_bytes.argtypes = [sp]
            L.gk_decode_attn_stack.restype = ctypes.c_int
            L.gk_decode_attn_stack.argtypes = [sp] + [vp] * 15 + [sz, vp]
            L.gk_decode_step.restype = ctypes.c_int
            L.gk_decode_step.argtypes = [sp] + [vp] * 19 + [sz, vp]
            L.gk_decode_attn_stack_static.restype = ctypes.c_int
            L.gk_decode_attn_stack_static.argtypes = [sp] + [vp] * 15
            L.gk_e4m3_quantize.restype = ctypes.c_int
            L.gk_e4m3_quantize.argtypes = [vp, ctypes.c_float, vp, i64, vp]
            L.gk_kv_budget.restype = ctypes.c_int
            L.gk_kv_budget.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                       ctypes.c_double, ctypes.c_double, sp,
                                       ctypes.POINTER(ctypes.c_uint64),
                                       ctypes.POINTER(ctypes.c_int64)]
            L.gk_kv_regions.restype = ctypes.c_int
            L.gk_kv_regions.argtypes = [sp, vp, vp, ctypes.POINTER(KvRegion), i32,
                                        ctypes.POINTER(ctypes.c_int32)]
            L.gk_kv_ingest.restype = ctypes.c_int
            L.gk_kv_ingest.argtypes = [ctypes.POINTER(KvRegion), i32, vp, vp, i64, vp, vp]
            L.gk_di_blocks.restype = ctypes.c_int
            L.gk_di_blocks.argtypes = [i64, i32, i32] + [ctypes.POINTER(ctypes.c_int64)] * 3
            L.gk_selftest_wait_timeout.restype = ctypes.c_int
            L.gk_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp,
                                                   ctypes.POINTER(ctypes.c_uint32)]
            L.gk_selftest_decode_attn_split.restype = ctypes.c_int
            L.gk_selftest_decode_attn_split.argtypes = [sp] + [vp] * 15 + [sz, i32, vp]
            L.gk_read_device_error.restype = ctypes.c_int
            L.gk_read_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
            _lib = L
    return _lib


# --------------------------------------------------------------- marshalling
def _ptr(t, dtype=None, name="tensor", allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _ptr_array(ts: Sequence, name: str):
    arr = (ctypes.c_void_p * len(ts))(*[_ptr(t, None, f"{name}[{i}]") for i, t in enumerate(ts)])
    return arr


def _stream(stream, like=None):
    if stream is None:
        import torch
        dev = like.device if like is not None and hasattr(like, "device") else None
        return torch.cuda.current_stream(dev).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != GK_OK:
        raise GkError(status, where)


def _sinks(sinks, shape):
    """Optional attention-sink logits: fp32 [NL, Hq] on the device, or None."""
    import torch
    if sinks is None:
        return None
    if sinks.numel() != shape.num_layers * shape.num_q_heads:
        raise ValueError(f"sinks must hold num_layers * num_q_heads = "
                         f"{shape.num_layers * shape.num_q_heads} values")
    return _ptr(sinks, torch.float32, "sinks")


def _as_shape(shape) -> Shape:
    if isinstance(shape, Shape):
        return shape
    return Shape.make(**shape)


# --------------------------------------------------------------- entry points
def gk_status_str(status: int) -> str:
    return lib().gk_status_str(int(status)).decode()


def gk_abi_version() -> int:
    return int(lib().gk_abi_version())


def gk_attn_workspace_bytes(shape) -> int:
    return int(lib().gk_attn_workspace_bytes(ctypes.byref(_as_shape(shape)), None))


def gk_attn_workspace_min_bytes(shape) -> int:
    return int(lib().gk_attn_workspace_min_bytes(ctypes.byref(_as_shape(shape))))


def gk_kv_append(shape, k_new, v_new, cos, sin, k_scale, v_scale, upd_full, upd_swa, active,
                 kv: KvCache, stream=None) -> None:
    import torch
    sh = _as_shape(shape)
    st = lib().gk_kv_append(
        ctypes.byref(sh), _ptr(k_new, torch.bfloat16, "k_new"), _ptr(v_new, torch.bfloat16, "v_new"),
        _ptr(cos, torch.float32, "cos"), _ptr(sin, torch.float32, "sin"),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale"),
        _ptr(upd_full, torch.int32, "upd_full"), _ptr(upd_swa, torch.int32, "upd_swa"),
        _ptr(active, torch.uint8, "active"), _kv(kv, sh), _stream(stream, k_new))
    _check(st, "gk_kv_append")


def gk_decode_attn_stack(shape, q, kv: KvCache, k_scale, v_scale, cos, sin, bt_full, bt_swa,
                         pos, pos_w, active, out, out_f32=None, workspace=None,
                         stream=None, sinks=None) -> None:
    import torch
    sh = _as_shape(shape)
    if workspace is None:
        raise ValueError("workspace is required (size: gk_attn_workspace_bytes(shape))")
    st = lib().gk_decode_attn_stack(
        ctypes.byref(sh), _ptr(q, torch.bfloat16, "q"), _kv(kv, sh),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale"),
        _ptr(cos, torch.float32, "cos"), _ptr(sin, torch.float32, "sin"),
        _ptr(bt_full, torch.int32, "bt_full"), _ptr(bt_swa, torch.int32, "bt_swa"),
        _ptr(pos, torch.int32, "pos"), _ptr(pos_w, torch.int32, "pos_w"),
        _ptr(active, torch.uint8, "active"), _sinks(sinks, sh), _ptr(out, torch.bfloat16, "out"),
        _ptr(out_f32, torch.float32, "out_f32", allow_none=True),
        _ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()), _stream(stream, q))
    _check(st, "gk_decode_attn_stack")


def gk_decode_step(shape, q, k_new, v_new, cos, sin, k_scale, v_scale, upd_full, upd_swa,
                   bt_full, bt_swa, pos, pos_w, active, kv: KvCache, out, out_f32=None,
                   workspace=None, stream=None, sinks=None) -> None:
    """gk_kv_append + gk_decode_attn_stack in two launches (the append in the planner's)."""
    import torch
    sh = _as_shape(shape)
    if workspace is None:
        raise ValueError("workspace is required (size: gk_attn_workspace_bytes(shape))")
    st = lib().gk_decode_step(
        ctypes.byref(sh), _ptr(q, torch.bfloat16, "q"), _ptr(k_new, torch.bfloat16, "k_new"),
        _ptr(v_new, torch.bfloat16, "v_new"), _ptr(cos, torch.float32, "cos"),
        _ptr(sin, torch.float32, "sin"), _ptr(k_scale, torch.float32, "k_scale"),
        _ptr(v_scale, torch.float32, "v_scale"), _ptr(upd_full, torch.int32, "upd_full"),
        _ptr(upd_swa, torch.int32, "upd_swa"), _ptr(bt_full, torch.int32, "bt_full"),
        _ptr(bt_swa, torch.int32, "bt_swa"), _ptr(pos, torch.int32, "pos"),
        _ptr(pos_w, torch.int32, "pos_w"), _ptr(active, torch.uint8, "active"),
        _sinks(sinks, sh), _kv(kv, sh), _ptr(out, torch.bfloat16, "out"),
        _ptr(out_f32, torch.float32, "out_f32", allow_none=True),
        _ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()), _stream(stream, q))
    _check(st, "gk_decode_step")


def gk_decode_attn_stack_static(shape, q, kv: KvCache, k_scale, v_scale, cos, sin, bt_full,
                                bt_swa, pos, pos_w, active, out, out_f32=None,
                                stream=None, sinks=None) -> None:
    """gk_decode_attn_stack without a caller workspace, for callers that cannot
    allocate device memory: the library's own fixed scratch array
    (GK_STATIC_SCRATCH_BYTES per GPU) serves as the workspace.  Calls on one
    device share that array, so they must not overlap on the GPU."""
    import torch
    sh = _as_shape(shape)
    st = lib().gk_decode_attn_stack_static(
        ctypes.byref(sh), _ptr(q, torch.bfloat16, "q"), _kv(kv, sh),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale"),
        _ptr(cos, torch.float32, "cos"), _ptr(sin, torch.float32, "sin"),
        _ptr(bt_full, torch.int32, "bt_full"), _ptr(bt_swa, torch.int32, "bt_swa"),
        _ptr(pos, torch.int32, "pos"), _ptr(pos_w, torch.int32, "pos_w"),
        _ptr(active, torch.uint8, "active"), _sinks(sinks, sh), _ptr(out, torch.bfloat16, "out"),
        _ptr(out_f32, torch.float32, "out_f32", allow_none=True), _stream(stream, q))
    _check(st, "gk_decode_attn_stack_static")


def gk_e4m3_quantize(x, scale: float, codes, stream=None) -> None:
    import torch
    st = lib().gk_e4m3_quantize(_ptr(x, torch.float32, "x"), float(scale),
                                _ptr(codes, torch.uint8, "codes"), int(x.numel()),
                                _stream(stream, x))
    _check(st, "gk_e4m3_quantize")


def gk_read_device_error(stream=None, clear: bool = True) -> int:
    """Synchronise the stream and return (and by default clear) the device
    error word: GK_DEVERR_* bits, 0 when nothing went out of range."""
    bits = ctypes.c_uint32(0)
    st = lib().gk_read_device_error(_stream(stream), ctypes.byref(bits), 1 if clear else 0)
    if st not in (GK_OK, GK_ERR_DEVICE_BOUNDS):
        raise GkError(st, "gk_read_device_error")
    return int(bits.value)


def gk_kv_budget(total_bytes: int, used_bytes: int, gpu_memory_utilization: float,
                 cap_fraction: float = 0.30, min_budget_gib: float = 1.0, shape=None):
    """KV pool size (host only): returns (status, available_bytes, num_blocks or None).
    GK_ERR_BUDGET is returned, not raised, so that callers can report the
    numbers the minimum-KV guard rejected."""
    avail = ctypes.c_uint64(0)
    nb = ctypes.c_int64(0)
    sh = ctypes.byref(_as_shape(shape)) if shape is not None else None
    st = lib().gk_kv_budget(int(total_bytes), int(used_bytes), float(gpu_memory_utilization),
                            float(cap_fraction), float(min_budget_gib), sh, ctypes.byref(avail),
                            ctypes.byref(nb) if shape is not None else None)
    if st not in (GK_OK, GK_ERR_BUDGET):
        raise GkError(st, "gk_kv_budget")
    return st, int(avail.value), (int(nb.value) if shape is not None else None)


def layer_binding(kv: KvCache, num_layers: int):
    """The per-layer binding of a KvCache (layer i -> group buffer i // 2), as
    device addresses: (layer_k, layer_v), each a list of num_layers ints."""
    ks, vs = kv._keep
    if kv.per_group:
        kb = [_ptr(t, None, "k") for t in ks]
        vb = [_ptr(t, None, "v") for t in vs]
    else:
        k, v = ks[0], vs[0]
        G = k.shape[0]
        half = k.numel() * k.element_size() // G
        kb = [_ptr(k, None, "k_cache") + j * half for j in range(G)]
        vb = [_ptr(v, None, "v_cache") + j * half for j in range(G)]
    return [kb[i // 2] for i in range(num_layers)], [vb[i // 2] for i in range(num_layers)]


def gk_kv_regions(shape, layer_k: Sequence[int], layer_v: Sequence[int]):
    """De-duplicated DI regions of a per-layer binding (host only): a ctypes
    array of KvRegion, K_0, V_0, K_1, V_1, ... for the page's layout."""
    sh = _as_shape(shape)
    n = len(layer_k)
    if n != sh.num_layers or len(layer_v) != n:
        raise ValueError("one K and one V address per layer")
    ka = (ctypes.c_void_p * n)(*layer_k)
    va = (ctypes.c_void_p * n)(*layer_v)
    cap = 2 * n
    out = (KvRegion * cap)()
    cnt = ctypes.c_int32(0)
    st = lib().gk_kv_regions(ctypes.byref(sh), ctypes.cast(ka, ctypes.c_void_p),
                             ctypes.cast(va, ctypes.c_void_p), out, cap, ctypes.byref(cnt))
    _check(st, "gk_kv_regions")
    return (KvRegion * cnt.value)(*out[:cnt.value])


def gk_kv_ingest(regions, dst_region, dst_block, src, stream=None) -> None:
    """Land len(dst_region) blocks from ``src`` (device tensor or pinned host
    tensor, n * block_len bytes) onto regions[dst_region[d]] block dst_block[d]."""
    import torch
    n = int(dst_region.numel())
    if int(dst_block.numel()) != n:
        raise ValueError("dst_region and dst_block must have one entry per descriptor")
    if n == 0:
        return
    if not src.is_contiguous():
        raise ValueError("src must be contiguous")
    if src.is_cuda is False and not src.is_pinned():
        raise ValueError("src must be a CUDA tensor or pinned host memory (no pageable copy)")
    bl = int(regions[0].block_len)
    if src.numel() * src.element_size() < n * bl:
        raise ValueError(f"src holds {src.numel() * src.element_size()} bytes, need {n * bl}")
    st = lib().gk_kv_ingest(regions, len(regions), _ptr(dst_region, torch.int32, "dst_region"),
                            _ptr(dst_block, torch.int32, "dst_block"), n, src.data_ptr(),
                            _stream(stream, dst_region))
    _check(st, "gk_kv_ingest")


def gk_di_blocks(num_tokens: int, block_size: int, window: int):
    """(full_count, swa_first, swa_count): the row blocks a decode engine needs
    for a prompt of num_tokens tokens, both engines operating at N - 1."""
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    st = lib().gk_di_blocks(int(num_tokens), int(block_size), int(window), ctypes.byref(a),
                            ctypes.byref(b), ctypes.byref(c))
    _check(st, "gk_di_blocks")
    return a.value, b.value, c.value


def gk_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """Test hook (include/gk_testing.h): run the bounded barrier wait into its
    limit on the GPU; returns the device error word (GK_DEVERR_TIMEOUT expected)."""
    bits = ctypes.c_uint32(0)
    st = lib().gk_selftest_wait_timeout(int(limit_ns), _stream(stream), ctypes.byref(bits))
    if st not in (GK_OK, GK_ERR_DEVICE_BOUNDS):
        raise GkError(st, "gk_selftest_wait_timeout")
    return int(bits.value)


def gk_selftest_decode_attn_split(shape, q, kv: KvCache, k_scale, v_scale, cos, sin, bt_full,
                                  bt_swa, pos, pos_w, active, out, out_f32, workspace,
                                  split_tokens: int, stream=None, sinks=None) -> None:
    """Test hook (include/gk_testing.h): gk_decode_attn_stack with the split-KV
    chunk length fixed to `split_tokens` (a power of two >= 512)."""
    import torch
    sh = _as_shape(shape)
    st = lib().gk_selftest_decode_attn_split(
        ctypes.byref(sh), _ptr(q, torch.bfloat16, "q"), _kv(kv, sh),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale"),
        _ptr(cos, torch.float32, "cos"), _ptr(sin, torch.float32, "sin"),
        _ptr(bt_full, torch.int32, "bt_full"), _ptr(bt_swa, torch.int32, "bt_swa"),
        _ptr(pos, torch.int32, "pos"), _ptr(pos_w, torch.int32, "pos_w"),
        _ptr(active, torch.uint8, "active"), _sinks(sinks, sh), _ptr(out, torch.bfloat16, "out"),
        _ptr(out_f32, torch.float32, "out_f32", allow_none=True),
        _ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()), int(split_tokens),
        _stream(stream, q))
    _check(st, "gk_selftest_decode_attn_split")


def new_workspace(shape, device="cuda"):
    import torch
    n = gk_attn_workspace_bytes(shape)
    if n == 0:
        raise GkError(GK_ERR_UNSUPPORTED, "gk_attn_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)
