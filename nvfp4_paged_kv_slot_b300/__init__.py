"""Python binding of libfi_nvfp4.so — NVFP4 paged-KV append and causal prefill
for B300 (sm_103a).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels; PyTorch supplies device memory and streams.  The functions keep the C
names (see include/fi_nvfp4.h for the full contract).  Importing this module
fails if the compiled library is missing — there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import math
import pathlib

import numpy as np

_HERE = pathlib.Path(__file__).resolve().parent
LIB_PATH = _HERE / "libfi_nvfp4.so"
if not LIB_PATH.exists():
    raise ImportError(f"{LIB_PATH} is not built: run `python -m nvfp4_paged_kv_slot_b300.build`")

lib = C.CDLL(str(LIB_PATH))

FI_OK = 0
FI_ERR_INVALID_ARGUMENT = 1
FI_ERR_BAD_SCALE = 2
FI_ERR_UNSUPPORTED = 3
FI_ERR_CUDA = 4
FI_ERR_OUT_OF_MEMORY = 5
FI_ERR_SCRATCH_TOO_SMALL = 6

FI_DEV_BAD_K_SCALE = 1
FI_DEV_BAD_V_SCALE = 2
FI_DEV_SLOT_OOB = 4
FI_DEV_PAGE_OOB = 8
FI_DEV_WAIT_TIMEOUT = 16

EXPORTED = ("fi_context_create", "fi_context_destroy", "fi_nvfp4_append",
            "fi_nvfp4_append_host_scale", "fi_plan_create", "fi_plan_destroy",
            "fi_prefill_plan", "fi_plan_get_info", "fi_prefill_run", "fi_prefill_plan_host",
            "fi_device_status", "fi_status_string", "fi_version", "fi_prefill_noalloc",
            "fi_fp8_append", "fi_prefill_run_fp8", "fi_decode_plan", "fi_decode_run",
            "fi_decode_plan_host")


class fi_nvfp4_cache(C.Structure):
    _fields_ = [("k_data", C.c_void_p), ("v_data", C.c_void_p), ("k_sf", C.c_void_p),
                ("v_sf", C.c_void_p), ("k_scale", C.c_void_p), ("v_scale", C.c_void_p),
                ("num_pages", C.c_int32), ("page_size", C.c_int32),
                ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32)]


class fi_plan_options(C.Structure):
    _fields_ = [("schedule", C.c_int32), ("num_ctas", C.c_int32), ("l2_bytes", C.c_int64),
                ("cta_pairs", C.c_int32), ("kv_format", C.c_int32)]


class fi_fp8_cache(C.Structure):
    _fields_ = [("k_data", C.c_void_p), ("v_data", C.c_void_p), ("k_scale", C.c_void_p),
                ("v_scale", C.c_void_p), ("num_pages", C.c_int32), ("page_size", C.c_int32),
                ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32)]


class fi_plan_info(C.Structure):
    _fields_ = [("batch", C.c_int32), ("max_qo_len", C.c_int32), ("max_kv_len", C.c_int32),
                ("total_qo_len", C.c_int64), ("total_kv_len", C.c_int64),
                ("is_uniform", C.c_int32), ("global_reverse", C.c_int32),
                ("q_tiles", C.c_int32), ("heads_per_cta", C.c_int32),
                ("head_units", C.c_int32), ("num_units", C.c_int64), ("kv_bytes", C.c_int64),
                ("num_ctas", C.c_int32), ("ctas_per_unit", C.c_int32),
                ("balanced", C.c_int32), ("max_slot_tiles", C.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_vp, _i32, _i64, _f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_float
_sigs = {
    "fi_context_create": [C.POINTER(_vp)],
    "fi_context_destroy": [_vp],
    "fi_nvfp4_append": [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _vp,
                        C.POINTER(fi_nvfp4_cache), _vp],
    "fi_nvfp4_append_host_scale": [_vp, _vp, _vp, _i64, _i64, _i64, _f32, _f32, _vp,
                                   C.POINTER(fi_nvfp4_cache), _vp],
    "fi_decode_plan": [_vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _vp],
    "fi_decode_run": [_vp, _vp, C.POINTER(fi_nvfp4_cache), _vp, _vp, _vp],
    "fi_fp8_append": [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _vp,
                      C.POINTER(fi_fp8_cache), _vp],
    "fi_prefill_run_fp8": [_vp, _vp, C.POINTER(fi_fp8_cache), _vp, _vp, _vp],
    "fi_plan_create": [_vp, C.POINTER(_vp)],
    "fi_plan_destroy": [_vp],
    "fi_prefill_plan": [_vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _f32,
                        C.POINTER(fi_plan_options), _vp],
    "fi_plan_get_info": [_vp, C.POINTER(fi_plan_info)],
    "fi_prefill_run": [_vp, _vp, C.POINTER(fi_nvfp4_cache), _vp, _vp, _vp],
    "fi_prefill_plan_host": [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64,
                             C.POINTER(fi_plan_options), C.POINTER(fi_plan_info), _vp, _i64],
    "fi_decode_plan_host": [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                            C.POINTER(fi_plan_info), C.POINTER(_i32), C.POINTER(_i64), _vp, _i64,
                            _vp, _i64, _vp, _i64],
    "fi_device_status": [_vp, _vp, C.POINTER(_i32), _i32],
    "fi_prefill_noalloc": [_vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _vp,
                           C.POINTER(fi_nvfp4_cache), _vp, _vp, _vp, _vp],
    "fi_status_string": [_i32],
    "fi_version": [],
}
for _name, _args in _sigs.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = C.c_char_p if _name == "fi_status_string" else C.c_int32


class FiError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.fi_status_string(status).decode()} (status {status})")


def _check(status: int, where: str):
    if status != FI_OK:
        raise FiError(status, where)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _host_i32(a) -> np.ndarray:
    """Host int32 array from a CPU tensor, numpy array or sequence.  Lengths
    given as other integer types (uint32, int64) are converted to int32 at
    entry, with a range check."""
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    a = np.asarray(a)
    if a.dtype != np.int32:
        if not np.issubdtype(a.dtype, np.integer):
            raise TypeError("integer array expected")
        if a.size and (a.min() < np.iinfo(np.int32).min or a.max() > np.iinfo(np.int32).max):
            raise ValueError("values out of int32 range")
        a = a.astype(np.int32)
    return np.ascontiguousarray(a)


def indptr_from_lens(lens) -> np.ndarray:
    """[B] lengths of any integer dtype -> int32 [B+1] exclusive prefix sum."""
    a = _host_i32(lens).astype(np.int64)
    out = np.zeros(a.size + 1, np.int64)
    np.cumsum(a, out=out[1:])
    if out[-1] > np.iinfo(np.int32).max:
        raise ValueError("total length exceeds int32")
    return out.astype(np.int32)


# --- cache -------------------------------------------------------------------
class NVFP4Cache:
    """Device tensors of one NVFP4 paged KV cache (HND layout, see the C header)
    and the ctypes view passed to the library."""

    def __init__(self, num_pages, num_kv_heads, page_size, head_dim, device="cuda",
                 k_scale=None, v_scale=None, fill=None):
        import torch
        shape_d = (num_pages, num_kv_heads, page_size, head_dim // 2)
        shape_s = (num_pages, num_kv_heads, page_size, head_dim // 16)
        mk = (lambda s: torch.full(s, fill, dtype=torch.uint8, device=device)) if fill is not None \
            else (lambda s: torch.empty(s, dtype=torch.uint8, device=device))
        self.k_data, self.v_data = mk(shape_d), mk(shape_d)
        self.k_sf, self.v_sf = mk(shape_s), mk(shape_s)
        self.k_scale = torch.ones(1, dtype=torch.float32, device=device) if k_scale is None \
            else k_scale
        self.v_scale = torch.ones(1, dtype=torch.float32, device=device) if v_scale is None \
            else v_scale
        self.num_pages, self.num_kv_heads = num_pages, num_kv_heads
        self.page_size, self.head_dim = page_size, head_dim

    def c(self) -> fi_nvfp4_cache:
        return fi_nvfp4_cache(self.k_data.data_ptr(), self.v_data.data_ptr(),
                              self.k_sf.data_ptr(), self.v_sf.data_ptr(),
                              self.k_scale.data_ptr(), self.v_scale.data_ptr(),
                              self.num_pages, self.page_size, self.num_kv_heads, self.head_dim)


class FP8Cache:
    """Device tensors of one FP8 (E4M3) paged KV cache, [P][H_kv][ps][D] bytes
    per tensor (see the C header), and the ctypes view passed to the library."""

    def __init__(self, num_pages, num_kv_heads, page_size, head_dim, device="cuda",
                 k_scale=None, v_scale=None, fill=None):
        import torch
        shape = (num_pages, num_kv_heads, page_size, head_dim)
        mk = (lambda: torch.full(shape, fill, dtype=torch.uint8, device=device)) \
            if fill is not None else (lambda: torch.empty(shape, dtype=torch.uint8, device=device))
        self.k_data, self.v_data = mk(), mk()
        self.k_scale = torch.ones(1, dtype=torch.float32, device=device) if k_scale is None \
            else k_scale
        self.v_scale = torch.ones(1, dtype=torch.float32, device=device) if v_scale is None \
            else v_scale
        self.num_pages, self.num_kv_heads = num_pages, num_kv_heads
        self.page_size, self.head_dim = page_size, head_dim

    def c(self) -> fi_fp8_cache:
        return fi_fp8_cache(self.k_data.data_ptr(), self.v_data.data_ptr(),
                            self.k_scale.data_ptr(), self.v_scale.data_ptr(),
                            self.num_pages, self.page_size, self.num_kv_heads, self.head_dim)


# --- entry points (same names as the C ABI) ------------------------------------
def fi_context_create():
    h = C.c_void_p()
    _check(lib.fi_context_create(C.byref(h)), "fi_context_create")
    return h


def fi_context_destroy(ctx):
    _check(lib.fi_context_destroy(ctx), "fi_context_destroy")


def _kv_args(k, v):
    import torch
    for name, t in (("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or t.dim() != 3 or t.stride(2) != 1 or \
                t.stride(1) != t.shape[2]:
            raise ValueError(f"{name}: bf16 [tokens][heads][head_dim] with contiguous rows")
    return k.shape[0], k.stride(0), v.stride(0)


def fi_nvfp4_append(ctx, k, v, k_scale, v_scale, slot_mapping, cache: NVFP4Cache,
                    stream=None):
    """k, v: bf16 [N][H_kv][D] on the device; k_scale, v_scale: device fp32
    scalars (checked by the kernel); slot_mapping: device int64 [N]."""
    import torch
    n, ks, vs = _kv_args(k, v)
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    cc = cache.c()
    _check(lib.fi_nvfp4_append(ctx, _ptr(k), _ptr(v), n, ks, vs, _ptr(k_scale), _ptr(v_scale),
                               _ptr(slot_mapping), C.byref(cc), _stream(stream)),
           "fi_nvfp4_append")


def fi_nvfp4_append_host_scale(ctx, k, v, k_scale: float, v_scale: float, slot_mapping,
                               cache: NVFP4Cache, stream=None):
    n, ks, vs = _kv_args(k, v)
    cc = cache.c()
    _check(lib.fi_nvfp4_append_host_scale(ctx, _ptr(k), _ptr(v), n, ks, vs, float(k_scale),
                                          float(v_scale), _ptr(slot_mapping), C.byref(cc),
                                          _stream(stream)), "fi_nvfp4_append_host_scale")


def fi_plan_create(ctx):
    h = C.c_void_p()
    _check(lib.fi_plan_create(ctx, C.byref(h)), "fi_plan_create")
    return h


def fi_plan_destroy(plan):
    _check(lib.fi_plan_destroy(plan), "fi_plan_destroy")


def fi_prefill_plan(plan, qo_indptr, kv_indptr, page_table, num_qo_heads, num_kv_heads,
                    head_dim, page_size, sm_scale=0.0, schedule=0, num_ctas=0, l2_bytes=0,
                    cta_pairs=0, stream=None, kv_format=0):
    """qo_indptr, kv_indptr: host int32 [B+1] (other integer types are
    converted); page_table: device int32 [B][stride]."""
    qo = _host_i32(qo_indptr)
    kv = _host_i32(kv_indptr)
    if qo.size != kv.size or qo.size < 1:
        raise ValueError("qo_indptr and kv_indptr must both have batch+1 entries")
    opts = fi_plan_options(schedule, num_ctas, l2_bytes, cta_pairs, kv_format)
    _check(lib.fi_prefill_plan(plan, qo.ctypes.data, kv.ctypes.data, qo.size - 1,
                               _ptr(page_table), page_table.stride(0) if page_table is not None
                               else 0, num_qo_heads, num_kv_heads, head_dim, page_size,
                               float(sm_scale), C.byref(opts), _stream(stream)),
           "fi_prefill_plan")


def fi_plan_get_info(plan) -> dict:
    info = fi_plan_info()
    _check(lib.fi_plan_get_info(plan, C.byref(info)), "fi_plan_get_info")
    return info.as_dict()


def fi_prefill_run(plan, q, cache: NVFP4Cache, out, lse=None, stream=None):
    """q, out: bf16 [total_qo][H_q][D] (contiguous); lse: fp32 [total_qo][H_q] or None."""
    import torch
    for name, t in (("q", q), ("out", out)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor")
    cc = cache.c()
    _check(lib.fi_prefill_run(plan, _ptr(q), C.byref(cc), _ptr(out), _ptr(lse),
                              _stream(stream)), "fi_prefill_run")


def fi_decode_plan(plan, qo_indptr, kv_indptr, page_table, num_qo_heads, num_kv_heads,
                   head_dim, page_size, sm_scale=0.0, stream=None):
    """Decode plan (qo_len <= 8 per sequence); arguments as fi_prefill_plan."""
    qo = _host_i32(qo_indptr)
    kv = _host_i32(kv_indptr)
    if qo.size != kv.size or qo.size < 1:
        raise ValueError("qo_indptr and kv_indptr must both have batch+1 entries")
    _check(lib.fi_decode_plan(plan, qo.ctypes.data, kv.ctypes.data, qo.size - 1,
                              _ptr(page_table), page_table.stride(0) if page_table is not None
                              else 0, num_qo_heads, num_kv_heads, head_dim, page_size,
                              float(sm_scale), _stream(stream)), "fi_decode_plan")


def fi_decode_run(plan, q, cache: NVFP4Cache, out, lse=None, stream=None):
    """Runs a decode plan; arguments as fi_prefill_run."""
    import torch
    for name, t in (("q", q), ("out", out)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor")
    cc = cache.c()
    _check(lib.fi_decode_run(plan, _ptr(q), C.byref(cc), _ptr(out), _ptr(lse), _stream(stream)),
           "fi_decode_run")


def fi_fp8_append(ctx, k, v, k_scale, v_scale, slot_mapping, cache: FP8Cache, stream=None):
    """FP8 (E4M3) append; arguments as fi_nvfp4_append."""
    import torch
    n, ks, vs = _kv_args(k, v)
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    cc = cache.c()
    _check(lib.fi_fp8_append(ctx, _ptr(k), _ptr(v), n, ks, vs, _ptr(k_scale), _ptr(v_scale),
                             _ptr(slot_mapping), C.byref(cc), _stream(stream)), "fi_fp8_append")


def fi_prefill_run_fp8(plan, q, cache: FP8Cache, out, lse=None, stream=None):
    """Prefill over the FP8 cache with a plan made with kv_format=1."""
    import torch
    for name, t in (("q", q), ("out", out)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor")
    cc = cache.c()
    _check(lib.fi_prefill_run_fp8(plan, _ptr(q), C.byref(cc), _ptr(out), _ptr(lse),
                                  _stream(stream)), "fi_prefill_run_fp8")


def fi_prefill_plan_host(qo_indptr, kv_indptr, num_qo_heads, num_kv_heads, head_dim, page_size,
                         l2_bytes=126 * 2**20, schedule=0, num_ctas=0, with_list=True,
                         cta_pairs=0, kv_format=0):
    """Host-only planning (no CUDA): returns (info dict, work [units][4] int32)."""
    qo = _host_i32(qo_indptr)
    kv = _host_i32(kv_indptr)
    opts = fi_plan_options(schedule, num_ctas, l2_bytes, cta_pairs, kv_format)
    info = fi_plan_info()
    _check(lib.fi_prefill_plan_host(qo.ctypes.data, kv.ctypes.data, qo.size - 1, num_qo_heads,
                                    num_kv_heads, head_dim, page_size, l2_bytes, C.byref(opts),
                                    C.byref(info), None, 0), "fi_prefill_plan_host")
    work = np.zeros((0, 4), np.int32)
    if with_list and info.num_units:
        work = np.zeros((info.num_units, 4), np.int32)
        _check(lib.fi_prefill_plan_host(qo.ctypes.data, kv.ctypes.data, qo.size - 1,
                                        num_qo_heads, num_kv_heads, head_dim, page_size,
                                        l2_bytes, C.byref(opts), C.byref(info),
                                        work.ctypes.data, info.num_units),
               "fi_prefill_plan_host")
    return info.as_dict(), work


def fi_decode_plan_host(qo_indptr, kv_indptr, num_qo_heads, num_kv_heads, head_dim, page_size,
                        num_sms=148):
    """Host-only decode planning (no CUDA): returns (info dict, number of warps W,
    pieces [n][4] int32, merges [m][4] int32, warp offsets [W + 1] int32)."""
    qo = _host_i32(qo_indptr)
    kv = _host_i32(kv_indptr)
    info = fi_plan_info()
    warps = C.c_int32()
    merges = C.c_int64()
    args = (qo.ctypes.data, kv.ctypes.data, qo.size - 1, num_qo_heads, num_kv_heads, head_dim,
            page_size, num_sms, C.byref(info), C.byref(warps), C.byref(merges))
    _check(lib.fi_decode_plan_host(*args, None, 0, None, 0, None, 0), "fi_decode_plan_host")
    units = np.zeros((info.num_units, 4), np.int32)
    mlist = np.zeros((merges.value, 4), np.int32)
    off = np.zeros(warps.value + 1, np.int32)
    _check(lib.fi_decode_plan_host(*args, units.ctypes.data if units.size else None,
                                   info.num_units, mlist.ctypes.data if mlist.size else None,
                                   merges.value, off.ctypes.data, off.size),
           "fi_decode_plan_host")
    return info.as_dict(), warps.value, units, mlist, off


def fi_device_status(ctx, stream=None, reset=True) -> int:
    bits = C.c_int32()
    _check(lib.fi_device_status(ctx, _stream(stream), C.byref(bits), 1 if reset else 0),
           "fi_device_status")
    return bits.value


def fi_version() -> int:
    return lib.fi_version()


def default_sm_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
