"""Binding of the diagnostic probes in libfi_nvfp4_diag.so (include/fi_nvfp4_diag.h).

They run the library's own device code on small inputs so tests can pin each
building block (conversions, block quantizer, tile repack, tcgen05 layouts).
"""
from __future__ import annotations

import ctypes as C
import pathlib

_HERE = pathlib.Path(__file__).resolve().parent
LIB_PATH = _HERE / "libfi_nvfp4_diag.so"
if not LIB_PATH.exists():
    raise ImportError(f"{LIB_PATH} is not built: run `python -m nvfp4_paged_kv_slot_b300.build`")
lib = C.CDLL(str(LIB_PATH))

EXPORTED = ("fi_diag_codec_span", "fi_diag_quantize_blocks", "fi_diag_div_check",
            "fi_diag_repack_tile", "fi_diag_umma", "fi_diag_wait_timeout", "fi_diag_umma_pair")

_vp = C.c_void_p
lib.fi_diag_codec_span.argtypes = [C.c_uint32, C.c_uint64, _vp, _vp, _vp]
lib.fi_diag_quantize_blocks.argtypes = [_vp, C.c_int64, C.c_float, _vp, _vp, _vp]
lib.fi_diag_div_check.argtypes = [_vp, C.c_int32, _vp, _vp, _vp]
lib.fi_diag_repack_tile.argtypes = [_vp, C.c_int32, C.c_int32, C.c_int32, _vp, _vp]
lib.fi_diag_umma.argtypes = [C.c_int32, _vp, _vp, _vp, _vp, _vp]
lib.fi_diag_wait_timeout.argtypes = [C.c_uint64, _vp, _vp, _vp, _vp, _vp]
lib.fi_diag_umma_pair.argtypes = [C.c_int32, _vp, _vp, _vp, _vp, _vp, _vp]
for _n in EXPORTED:
    getattr(lib, _n).restype = C.c_int32


def _s():
    import torch
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ok(rc, name):
    if rc != 0:
        raise RuntimeError(f"{name} failed with {rc}")


def codec_span(first_bits: int, count: int, e4m3_out, e2m1_out):
    _ok(lib.fi_diag_codec_span(first_bits & 0xFFFFFFFF, count, e4m3_out.data_ptr(),
                               e2m1_out.data_ptr(), _s()), "fi_diag_codec_span")


def quantize_blocks(x, g: float, packed_out, s8_out):
    _ok(lib.fi_diag_quantize_blocks(x.data_ptr(), x.numel() // 16, float(g),
                                    packed_out.data_ptr(), s8_out.data_ptr(), _s()),
        "fi_diag_quantize_blocks")


def div_check(d_values, counts, first_bad):
    _ok(lib.fi_diag_div_check(d_values.data_ptr(), d_values.numel(), counts.data_ptr(),
                              first_bad.data_ptr(), _s()), "fi_diag_div_check")


def repack_tile(raw, head_dim: int, is_v: bool, valid: int, out):
    _ok(lib.fi_diag_repack_tile(raw.data_ptr(), head_dim, int(is_v), valid, out.data_ptr(),
                                _s()), "fi_diag_repack_tile")


def umma(mode: int, a, b, c, status):
    _ok(lib.fi_diag_umma(mode, a.data_ptr(), b.data_ptr(), c.data_ptr(), status.data_ptr(),
                         _s()), "fi_diag_umma")


def wait_timeout(timeout_ns: int, copy_src, copy_out, status, report):
    _ok(lib.fi_diag_wait_timeout(int(timeout_ns), copy_src.data_ptr(), copy_out.data_ptr(),
                                 status.data_ptr(), report.data_ptr(), _s()),
        "fi_diag_wait_timeout")


def umma_pair(mode: int, a, b, c, status, tmem_addrs):
    _ok(lib.fi_diag_umma_pair(mode, a.data_ptr(), b.data_ptr(), c.data_ptr(), status.data_ptr(),
                              tmem_addrs.data_ptr(), _s()), "fi_diag_umma_pair")
