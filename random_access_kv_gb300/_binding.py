"""ctypes binding of libfq.so: the C ABI of include/fq.h and include/fractal.h under the same names.

Argument marshalling only: every function takes device buffers as torch CUDA tensors (or raw
integer addresses), passes their addresses and sizes to the C entry point of the same name and
raises ``FQError`` on a non-zero return code. No step of the codec runs here.

The library is loaded from this package directory. If it is missing the import fails loudly
(``FQLibraryMissing``): there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfq.so")
HEADERS = [os.path.join(os.path.dirname(PKG), "include", h) for h in ("fq.h", "fractal.h")]

FQ_OK, FQ_EINVAL, FQ_ENOMEM, FQ_ECUDA, FQ_EALIGN, FQ_ENODEV = range(6)
FQ_FLAG_RANGE, FQ_FLAG_NONFINITE, FQ_FLAG_TIMEOUT = 1, 2, 4
FA_FLAG_SYMBOL, FA_FLAG_RANGE, FA_FLAG_CORRUPT = 1, 2, 4


class FQLibraryMissing(ImportError):
    pass


class FQError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {strerror(code)} ({code})")


_c_void_p, _i64, _int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int

_SIGNATURES = {
    "fq_codebook_load": (_int, [ctypes.POINTER(_c_void_p), _c_void_p, _int, _int, _c_void_p, _int, _int]),
    "fq_encode": (_int, [_c_void_p, _c_void_p, _i64, _c_void_p, _c_void_p, _i64, _c_void_p]),
    "fq_encode_append": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _i64, _c_void_p, _c_void_p, _c_void_p]),
    "fq_decode": (_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p, _c_void_p]),
    "fq_decode_gather": (_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p, _i64, _c_void_p, _c_void_p]),
    "fq_decode_gather_f32": (_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p, _i64, _c_void_p, _c_void_p]),
    "fq_attend": (_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p, _i64, _i64, _i64, _i64, _i64, _i64,
                         ctypes.c_float, _c_void_p, _c_void_p]),
    "fq_centroid_sums": (_int, [_c_void_p, _c_void_p, _i64, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "fq_selftest_wait": (_int, [_c_void_p, ctypes.c_uint64, _c_void_p]),
    "fq_code_words": (_i64, [_c_void_p, _i64]),
    "fq_record_bits": (_int, [_c_void_p]),
    "fq_shape": (_int, [_c_void_p, ctypes.POINTER(_int), ctypes.POINTER(_int), ctypes.POINTER(_int)]),
    "fq_status": (_int, [_c_void_p, _c_void_p, ctypes.POINTER(ctypes.c_uint32)]),
    "fq_destroy": (None, [_c_void_p]),
    "fq_strerror": (ctypes.c_char_p, [_int]),
    "fa_ratio_limit": (ctypes.c_double, [_int]),
    "fa_max_segment": (_int, [_int, ctypes.c_double]),
    "fa_create": (_int, [ctypes.POINTER(_c_void_p), _int, ctypes.c_double, _int, _int]),
    "fa_params": (_int, [_c_void_p, ctypes.POINTER(_int), ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_int)]),
    "fa_vertex_table": (_int, [_c_void_p, _c_void_p]),
    "fa_segments": (_i64, [_c_void_p, _i64]),
    "fa_encode": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _i64, _c_void_p, _c_void_p]),
    "fa_decode": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p]),
    "fa_access": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p, _i64, _c_void_p, _c_void_p]),
    "fa_status": (_int, [_c_void_p, _c_void_p, ctypes.POINTER(ctypes.c_uint32)]),
    "fa_destroy": (None, [_c_void_p]),
}

_lib = None


def header_symbols() -> list[str]:
    """Names of the functions declared in include/fq.h and include/fractal.h."""
    names = set()
    for h in HEADERS:
        with open(h) as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        names.update(re.findall(r"\b((?:fq|fa)_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def lib() -> ctypes.CDLL:
    """The loaded library (loaded on first use)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FQLibraryMissing(f"{LIB_PATH} is not built; run random_access_kv_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().fq_strerror(int(code)).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr() if t.numel() else None
    if hasattr(t, "ctypes"):            # numpy host array
        return t.ctypes.data
    raise TypeError(f"cannot take the address of {type(t)}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> None:
    if rc != FQ_OK:
        raise FQError(fn, rc)


class Context:
    """Owns an ``fq_ctx*``; frees it with ``fq_destroy`` on ``close()`` or garbage collection."""

    _destroy = "fq_destroy"

    def __init__(self, handle: int):
        self.handle = handle

    @property
    def _as_parameter_(self):
        return ctypes.c_void_p(self.handle)

    def close(self) -> None:
        if self.handle:
            getattr(lib(), self._destroy)(ctypes.c_void_p(self.handle))
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fq_codebook_load(C, Pi, device: int = 0) -> Context:
    """C: float32 [N, k] host array; Pi: float32 [d, d] host array (C-contiguous numpy)."""
    import numpy as np
    C = np.ascontiguousarray(C, dtype=np.float32)
    Pi = np.ascontiguousarray(Pi, dtype=np.float32)
    if C.ndim != 2 or Pi.ndim != 2 or Pi.shape[0] != Pi.shape[1]:
        raise ValueError("C must be [N, k] and Pi [d, d]")
    h = _c_void_p()
    rc = lib().fq_codebook_load(ctypes.byref(h), C.ctypes.data, C.shape[0], C.shape[1],
                                Pi.ctypes.data, Pi.shape[0], int(device))
    _check("fq_codebook_load", rc)
    return Context(h.value)


def fq_encode(ctx: Context, x, M: int, nu, codes, row0: int = 0, stream=None) -> None:
    _check("fq_encode", lib().fq_encode(ctx, _ptr(x), int(M), _ptr(nu), _ptr(codes), int(row0),
                                        _stream(stream)))


def fq_encode_append(ctx: Context, x, n_seq: int, n_new: int, seq_capacity: int, t0: int, nu, codes,
                     stream=None) -> None:
    _check("fq_encode_append", lib().fq_encode_append(ctx, _ptr(x), int(n_seq), int(n_new),
                                                      int(seq_capacity), int(t0), _ptr(nu), _ptr(codes),
                                                      _stream(stream)))


def fq_decode(ctx: Context, nu, codes, M: int, out, stream=None) -> None:
    _check("fq_decode", lib().fq_decode(ctx, _ptr(nu), _ptr(codes), int(M), _ptr(out), _stream(stream)))


def fq_decode_gather(ctx: Context, nu, codes, M: int, idx, n: int, out, stream=None) -> None:
    _check("fq_decode_gather", lib().fq_decode_gather(ctx, _ptr(nu), _ptr(codes), int(M), _ptr(idx), int(n),
                                                      _ptr(out), _stream(stream)))


def fq_decode_gather_f32(ctx: Context, nu, codes, M: int, idx, n: int, out, stream=None) -> None:
    _check("fq_decode_gather_f32", lib().fq_decode_gather_f32(ctx, _ptr(nu), _ptr(codes), int(M), _ptr(idx),
                                                              int(n), _ptr(out), _stream(stream)))


def fq_attend(ctx: Context, nu, codes, M: int, q, n_queries: int, q_per_group: int, T: int, k_row0: int,
              v_row0: int, stride: int, scale: float, out, stream=None) -> None:
    _check("fq_attend", lib().fq_attend(ctx, _ptr(nu), _ptr(codes), int(M), _ptr(q), int(n_queries),
                                        int(q_per_group), int(T), int(k_row0), int(v_row0), int(stride),
                                        float(scale), _ptr(out), _stream(stream)))


def fq_centroid_sums(ctx: Context, x, M: int, nu, codes, sums, counts, stream=None) -> None:
    _check("fq_centroid_sums", lib().fq_centroid_sums(ctx, _ptr(x), int(M), _ptr(nu), _ptr(codes), _ptr(sums),
                                                      _ptr(counts), _stream(stream)))


def fq_selftest_wait(ctx: Context, limit_ns: int, stream=None) -> None:
    _check("fq_selftest_wait", lib().fq_selftest_wait(ctx, int(limit_ns), _stream(stream)))


def fq_code_words(ctx: Context, M: int) -> int:
    w = lib().fq_code_words(ctx, int(M))
    if w < 0:
        raise FQError("fq_code_words", FQ_EINVAL)
    return int(w)


def fq_record_bits(ctx: Context) -> int:
    return int(lib().fq_record_bits(ctx))


def fq_shape(ctx: Context) -> tuple[int, int, int]:
    d, k, N = _int(), _int(), _int()
    _check("fq_shape", lib().fq_shape(ctx, ctypes.byref(d), ctypes.byref(k), ctypes.byref(N)))
    return d.value, k.value, N.value


def fq_status(ctx: Context, stream=None) -> int:
    f = ctypes.c_uint32()
    _check("fq_status", lib().fq_status(ctx, _stream(stream), ctypes.byref(f)))
    return int(f.value)


def fq_destroy(ctx: Context) -> None:
    ctx.close()


def fq_strerror(code: int) -> str:
    return strerror(code)


# Iterated-map archive of symbol streams (include/fractal.h).

class ArchiveContext(Context):
    """Owns an ``fa_ctx*``; frees it with ``fa_destroy``."""

    _destroy = "fa_destroy"


def fa_ratio_limit(N: int) -> float:
    return float(lib().fa_ratio_limit(int(N)))


def fa_max_segment(N: int, r: float) -> int:
    return int(lib().fa_max_segment(int(N), float(r)))


def fa_create(N: int, r: float, L: int, device: int = 0) -> ArchiveContext:
    h = _c_void_p()
    _check("fa_create", lib().fa_create(ctypes.byref(h), int(N), float(r), int(L), int(device)))
    return ArchiveContext(h.value)


def fa_params(ctx: ArchiveContext) -> tuple[int, float, int]:
    N, r, L = _int(), ctypes.c_double(), _int()
    _check("fa_params", lib().fa_params(ctx, ctypes.byref(N), ctypes.byref(r), ctypes.byref(L)))
    return N.value, r.value, L.value


def fa_vertex_table(ctx: ArchiveContext):
    """The context's vertex table as a float64 numpy array [N, 2]."""
    import numpy as np
    N, _, _ = fa_params(ctx)
    V = np.zeros((N, 2), dtype=np.float64)
    _check("fa_vertex_table", lib().fa_vertex_table(ctx, V.ctypes.data))
    return V


def fa_segments(ctx: ArchiveContext, T_cap: int) -> int:
    s = lib().fa_segments(ctx, int(T_cap))
    if s < 0:
        raise FQError("fa_segments", FQ_EINVAL)
    return int(s)


def fa_encode(ctx: ArchiveContext, sym, n_streams: int, n_new: int, T_cap: int, T_old: int, anchors,
              stream=None) -> None:
    _check("fa_encode", lib().fa_encode(ctx, _ptr(sym), int(n_streams), int(n_new), int(T_cap), int(T_old),
                                        _ptr(anchors), _stream(stream)))


def fa_decode(ctx: ArchiveContext, anchors, n_streams: int, T_cap: int, T: int, out, stream=None) -> None:
    _check("fa_decode", lib().fa_decode(ctx, _ptr(anchors), int(n_streams), int(T_cap), int(T), _ptr(out),
                                        _stream(stream)))


def fa_access(ctx: ArchiveContext, anchors, n_streams: int, T_cap: int, T: int, pos, n: int, out,
              stream=None) -> None:
    _check("fa_access", lib().fa_access(ctx, _ptr(anchors), int(n_streams), int(T_cap), int(T), _ptr(pos), int(n),
                                        _ptr(out), _stream(stream)))


def fa_status(ctx: ArchiveContext, stream=None) -> int:
    f = ctypes.c_uint32()
    _check("fa_status", lib().fa_status(ctx, _stream(stream), ctypes.byref(f)))
    return int(f.value)


def fa_destroy(ctx: ArchiveContext) -> None:
    ctx.close()
