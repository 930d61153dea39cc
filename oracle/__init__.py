"""Python view of the CPU oracle (oracle.cpp), for tests and the CPU baseline.

TEST INFRASTRUCTURE ONLY.  The product package never imports this module; only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg do.
Arrays are numpy; bf16 tensors are passed as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes as C
import numpy as np

from . import build as _build

_lib = None

_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")

BAD_K_SCALE = 1
BAD_V_SCALE = 2
SLOT_OOB = 4


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(str(path))
        L.orc_e2m1_value.argtypes = [C.c_uint8]
        L.orc_e2m1_value.restype = C.c_double
        L.orc_e4m3_value.argtypes = [C.c_uint8]
        L.orc_e4m3_value.restype = C.c_double
        for name in ("orc_e2m1_encode", "orc_e4m3_encode", "orc_e2m1_encode_bits",
                     "orc_e4m3_encode_bits"):
            getattr(L, name).argtypes = [C.c_float]
            getattr(L, name).restype = C.c_uint8
        for name in ("orc_e2m1_encode_span", "orc_e4m3_encode_span"):
            getattr(L, name).argtypes = [C.c_uint32, C.c_uint64, _u8p]
            getattr(L, name).restype = None
        _f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        for name in ("orc_e2m1_encode_array", "orc_e4m3_encode_array"):
            getattr(L, name).argtypes = [_f32p, C.c_int64, C.c_int32, _u8p]
            getattr(L, name).restype = None
        L.orc_quantize_block16.argtypes = [_u16p, C.c_float, _u8p, _u8p]
        L.orc_quantize_block16.restype = None
        L.orc_append.argtypes = [_u16p, _u16p, C.c_int64, C.c_int64, C.c_int64, C.c_int32,
                                 C.c_int32, C.c_float, C.c_float, _i64p, _u8p, _u8p, _u8p,
                                 _u8p, C.c_int32, C.c_int32]
        L.orc_append.restype = C.c_int
        L.orc_dequant_row.argtypes = [_u8p, _u8p, C.c_int32, C.c_int32, C.c_int32, C.c_int64,
                                      C.c_int32, C.c_double, _f64p]
        L.orc_dequant_row.restype = None
        L.orc_prefill.argtypes = [_u16p, C.c_int32, _i32p, _i32p, _i32p, C.c_int32, C.c_int32,
                                  C.c_int32, C.c_int32, C.c_int32, _u8p, _u8p, _u8p, _u8p,
                                  C.c_double, C.c_double, C.c_double, C.c_void_p, C.c_int64,
                                  _f64p, _f64p, C.c_int32]
        L.orc_prefill.restype = C.c_int
        L.orc_prefill_fmt.argtypes = [_u16p, C.c_int32, _i32p, _i32p, _i32p, C.c_int32, C.c_int32,
                                      C.c_int32, C.c_int32, C.c_int32, C.c_int32, _u8p, _u8p,
                                      C.c_void_p, C.c_void_p, C.c_double, C.c_double, C.c_double,
                                      C.c_void_p, C.c_int64, _f64p, _f64p, C.c_int32]
        L.orc_prefill_fmt.restype = C.c_int
        L.orc_fp8_quantize.argtypes = [C.c_float, C.c_float]
        L.orc_fp8_quantize.restype = C.c_uint8
        L.orc_fp8_append.argtypes = [_u16p, _u16p, C.c_int64, C.c_int64, C.c_int64, C.c_int32,
                                     C.c_int32, C.c_float, C.c_float, _i64p, _u8p, _u8p,
                                     C.c_int32, C.c_int32]
        L.orc_fp8_append.restype = C.c_int
        L.orc_fp8_dequant_row.argtypes = [_u8p, C.c_int32, C.c_int32, C.c_int32, C.c_int64,
                                          C.c_int32, C.c_double, _f64p]
        L.orc_fp8_dequant_row.restype = None
        L.orc_dense_causal.argtypes = [_f64p, _f64p, _f64p, C.c_int32, C.c_int32, C.c_int32,
                                       C.c_double, _f64p, _f64p]
        L.orc_dense_causal.restype = None
        L.orc_max_threads.argtypes = []
        L.orc_max_threads.restype = C.c_int32
        _lib = L
    return _lib


def max_threads() -> int:
    return int(lib().orc_max_threads())


# --- codecs -----------------------------------------------------------------
def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def e2m1_encode(y: float) -> int:
    return lib().orc_e2m1_encode(float(np.float32(y)))


def e4m3_encode(t: float) -> int:
    return lib().orc_e4m3_encode(float(np.float32(t)))


def e2m1_encode_bits(y: float) -> int:
    return lib().orc_e2m1_encode_bits(float(np.float32(y)))


def e4m3_encode_bits(t: float) -> int:
    return lib().orc_e4m3_encode_bits(float(np.float32(t)))


def e2m1_encode_span(first_bits: int, count: int) -> np.ndarray:
    out = np.empty(count, np.uint8)
    lib().orc_e2m1_encode_span(first_bits & 0xFFFFFFFF, count, out)
    return out


def e4m3_encode_span(first_bits: int, count: int) -> np.ndarray:
    out = np.empty(count, np.uint8)
    lib().orc_e4m3_encode_span(first_bits & 0xFFFFFFFF, count, out)
    return out


def e2m1_encode_array(y, bit_level: bool = False) -> np.ndarray:
    a = np.ascontiguousarray(y, dtype=np.float32).reshape(-1)
    out = np.empty(a.size, np.uint8)
    lib().orc_e2m1_encode_array(a, a.size, int(bit_level), out)
    return out


def e4m3_encode_array(t, bit_level: bool = False) -> np.ndarray:
    a = np.ascontiguousarray(t, dtype=np.float32).reshape(-1)
    out = np.empty(a.size, np.uint8)
    lib().orc_e4m3_encode_array(a, a.size, int(bit_level), out)
    return out


# --- quantize / append ------------------------------------------------------
def quantize_block16(x_bits: np.ndarray, g: float):
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    assert x.size == 16
    packed = np.zeros(8, np.uint8)
    s8 = np.zeros(1, np.uint8)
    lib().orc_quantize_block16(x, float(np.float32(g)), packed, s8)
    return packed, int(s8[0])


def new_cache(num_pages: int, num_kv_heads: int, page_size: int, head_dim: int,
              fill: int = 0xA5) -> dict:
    """Host cache arrays in the library's HND layout, pre-filled with `fill`."""
    shape_d = (num_pages, num_kv_heads, page_size, head_dim // 2)
    shape_s = (num_pages, num_kv_heads, page_size, head_dim // 16)
    return {
        "k_data": np.full(shape_d, fill, np.uint8),
        "v_data": np.full(shape_d, fill, np.uint8),
        "k_sf": np.full(shape_s, fill, np.uint8),
        "v_sf": np.full(shape_s, fill, np.uint8),
        "num_pages": num_pages, "num_kv_heads": num_kv_heads,
        "page_size": page_size, "head_dim": head_dim,
    }


def append(k_bits: np.ndarray, v_bits: np.ndarray, k_scale: float, v_scale: float,
           slot_mapping: np.ndarray, cache: dict) -> int:
    """k_bits, v_bits: uint16 [N][H_kv][D] (contiguous).  Mutates `cache`."""
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    n, h, d = k.shape
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return lib().orc_append(k.reshape(-1), v.reshape(-1), n, h * d, h * d, h, d,
                            float(np.float32(k_scale)), float(np.float32(v_scale)), slots,
                            cache["k_data"].reshape(-1), cache["v_data"].reshape(-1),
                            cache["k_sf"].reshape(-1), cache["v_sf"].reshape(-1),
                            cache["num_pages"], cache["page_size"])


def dequant_row(cache: dict, which: str, slot: int, head: int, g: float) -> np.ndarray:
    out = np.empty(cache["head_dim"], np.float64)
    lib().orc_dequant_row(cache[f"{which}_data"].reshape(-1), cache[f"{which}_sf"].reshape(-1),
                          cache["num_kv_heads"], cache["head_dim"], cache["page_size"],
                          slot, head, g, out)
    return out


# --- FP8 (E4M3) paged KV variant ---------------------------------------------
def fp8_quantize(x: float, g: float) -> int:
    """E4M3 code of RN32(x / g) (x, g taken as fp32)."""
    return int(lib().orc_fp8_quantize(float(np.float32(x)), float(np.float32(g))))


def new_fp8_cache(num_pages: int, num_kv_heads: int, page_size: int, head_dim: int,
                  fill: int = 0xA5) -> dict:
    """Host FP8 cache arrays [P][H_kv][ps][D], pre-filled with `fill`."""
    shape = (num_pages, num_kv_heads, page_size, head_dim)
    return {"format": "fp8", "k_data": np.full(shape, fill, np.uint8),
            "v_data": np.full(shape, fill, np.uint8), "num_pages": num_pages,
            "num_kv_heads": num_kv_heads, "page_size": page_size, "head_dim": head_dim}


def fp8_append(k_bits: np.ndarray, v_bits: np.ndarray, k_scale: float, v_scale: float,
               slot_mapping: np.ndarray, cache: dict) -> int:
    """k_bits, v_bits: uint16 [N][H_kv][D] (contiguous).  Mutates `cache`."""
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    n, h, d = k.shape
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return lib().orc_fp8_append(k.reshape(-1), v.reshape(-1), n, h * d, h * d, h, d,
                                float(np.float32(k_scale)), float(np.float32(v_scale)), slots,
                                cache["k_data"].reshape(-1), cache["v_data"].reshape(-1),
                                cache["num_pages"], cache["page_size"])


def fp8_dequant_row(cache: dict, which: str, slot: int, head: int, g: float) -> np.ndarray:
    out = np.empty(cache["head_dim"], np.float64)
    lib().orc_fp8_dequant_row(cache[f"{which}_data"].reshape(-1), cache["num_kv_heads"],
                              cache["head_dim"], cache["page_size"], slot, head, g, out)
    return out


# --- attention --------------------------------------------------------------
def prefill(q_bits: np.ndarray, qo_indptr, kv_indptr, page_table: np.ndarray, cache: dict,
            num_qo_heads: int, k_scale: float, v_scale: float, sm_scale: float,
            rows: np.ndarray | None = None, threads: int = 0):
    """q_bits: uint16 [total_q][H_q][D]; cache: an NVFP4 cache (new_cache) or an
    FP8 one (new_fp8_cache).  Returns (out [n][D], lse [n]) in fp64,
    n = total_q*H_q (row r = token r // H_q, head r % H_q) or len(rows)."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16).reshape(-1)
    qo = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    kv = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    batch = qo.size - 1
    d = cache["head_dim"]
    if rows is None:
        n = int(qo[-1]) * num_qo_heads
        rows_arr, rows_ptr = None, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 2)
        n = rows_arr.shape[0]
        rows_ptr = rows_arr.ctypes.data_as(C.c_void_p)
    out = np.empty((n, d), np.float64)
    lse = np.empty(n, np.float64)
    fp8 = cache.get("format") == "fp8"
    rc = lib().orc_prefill_fmt(q, batch, qo, kv, pt.reshape(-1),
                               pt.shape[1] if pt.ndim == 2 else 0, num_qo_heads,
                               cache["num_kv_heads"], d, cache["page_size"], 1 if fp8 else 0,
                               cache["k_data"].reshape(-1), cache["v_data"].reshape(-1),
                               None if fp8 else cache["k_sf"].ctypes.data_as(C.c_void_p),
                               None if fp8 else cache["v_sf"].ctypes.data_as(C.c_void_p),
                               float(k_scale), float(v_scale), float(sm_scale), rows_ptr, n,
                               out.reshape(-1), lse, threads)
    if rc != 0:
        raise ValueError("oracle prefill: invalid arguments")
    return out, lse


def dense_causal(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float):
    q = np.ascontiguousarray(q, np.float64)
    k = np.ascontiguousarray(k, np.float64)
    v = np.ascontiguousarray(v, np.float64)
    lq, d = q.shape
    lkv = k.shape[0]
    out = np.empty((lq, d), np.float64)
    lse = np.empty(lq, np.float64)
    lib().orc_dense_causal(q.reshape(-1), k.reshape(-1), v.reshape(-1), lq, lkv, d,
                           float(sm_scale), out.reshape(-1), lse)
    return out, lse
