"""fp64 CPU oracle for paged GQA decode attention and the fp8 sliding-window variant.

TEST INFRASTRUCTURE ONLY: the tests, the package's smoke check and the benchmark's
CPU-baseline leg are the only callers.  The library path never imports this package, and
this package imports nothing from the library.  The arithmetic lives in ``dap_oracle.c``
(plain C, double precision, OpenMP over output rows); this module compiles it with gcc on
first use and marshals numpy arrays.

Inputs are raw bit patterns: bf16 tensors arrive as ``np.uint16`` arrays, the fp8 cache
as ``np.uint8``.  Outputs are ``np.float64``.

Every function is pinned by tests/test_oracle_pins.py (closed forms, brute force against
torch's float64 scaled_dot_product_attention, page-permutation invariance, the e4m3 table
against torch's float8_e4m3fn conversion).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dap_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile dap_oracle.c into oracle/_build/liboracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        LL = ctypes.c_longlong
        D = ctypes.c_double
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_value.restype = D
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = D
        lib.oracle_round_to_bf16.argtypes = [D]
        lib.oracle_round_to_bf16.restype = D
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = I
        lib.oracle_set_num_threads.argtypes = [I]
        lib.oracle_set_num_threads.restype = None
        lib.oracle_decode_paged.argtypes = [P, LL, LL, P, P, I, P, I, P, I, I, I, I, I, D, P]
        lib.oracle_decode_paged.restype = I
        lib.oracle_decode_paged_rows.argtypes = [P, LL, LL, P, P, I, P, I, P, I, I, I, I, I,
                                                 D, P, I, P]
        lib.oracle_decode_paged_rows.restype = I
        lib.oracle_decode_contig.argtypes = [P, LL, LL, P, P, I, P, I, I, I, I, D, P]
        lib.oracle_decode_contig.restype = I
        lib.oracle_fp8_swa_range.argtypes = [P, P, P, P, P, I, I, I, I, I, I, D, I, I, P]
        lib.oracle_fp8_swa_range.restype = None
        lib.oracle_kv_append_paged.argtypes = [P, P, P, P, I, I, P, I, P, I, I, I]
        lib.oracle_kv_append_paged.restype = I
        lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
        lib.oracle_kv_append_fp8.argtypes = [P, P, P, P, I, I, I, I]
        lib.oracle_kv_append_fp8.restype = I
        lib.oracle_decode_paged_multi.argtypes = [P, P, P, I, P, I, P, P, P, LL, I, I, I, I, I, D, P]
        lib.oracle_decode_paged_multi.restype = I
        lib.oracle_q_tile_map.argtypes = [P, I, I, P, P, P, I]
        lib.oracle_q_tile_map.restype = I
        lib.oracle_decode_paged_masked.argtypes = [P, LL, LL, P, P, I, P, I, P, P, LL, I, I, I, I, I, D, P]
        lib.oracle_decode_paged_masked.restype = I
        lib.oracle_decode_paged_fp8kv.argtypes = [P, LL, LL, P, P, P, P, I, P, I, P, I, I, I, I, I, D, P]
        lib.oracle_decode_paged_fp8kv.restype = I
        lib.oracle_kv_append_paged_fp8.argtypes = [P, P, P, P, P, P, I, I, P, I, P, I, I, I]
        lib.oracle_kv_append_paged_fp8.restype = I
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return np.ascontiguousarray(a)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def bf16_value(bits: int) -> float:
    return _load().oracle_bf16_value(int(bits))


def e4m3_value(byte: int) -> float:
    return _load().oracle_e4m3_value(int(byte))


def e4m3_table() -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_e4m3_value(b) for b in range(256)], dtype=np.float64)


def round_to_bf16(x: float) -> float:
    return _load().oracle_round_to_bf16(float(x))


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale: float) -> np.ndarray:
    """Paged GQA decode.  q [B,Hq,D] u16, caches [P,ps,Hkv,D] u16, block_table [B,max_pages]
    int32, seq_lens [B] int32.  Returns [B,Hq,D] float64."""
    q = _u16(q); k_cache = _u16(k_cache); v_cache = _u16(v_cache)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, D = q.shape
    P, ps, Hkv, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape and Hq % Hkv == 0
    out = np.empty((B, Hq, D), dtype=np.float64)
    bad = _load().oracle_decode_paged(_ptr(q), Hq * D, D, _ptr(k_cache), _ptr(v_cache), P,
                                      _ptr(bt), bt.shape[1], _ptr(sl), B, Hq, Hkv, D, ps,
                                      float(scale), _ptr(out))
    if bad:
        raise ValueError(f"{bad} output rows would read outside the given cache/table")
    return out


def decode_paged_rows(q, k_cache, v_cache, block_table, seq_lens, scale: float,
                      rows) -> np.ndarray:
    """Selected output rows of paged decode; rows[i] = b * Hq + h.  Returns [n, D]."""
    q = _u16(q); k_cache = _u16(k_cache); v_cache = _u16(v_cache)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    B, Hq, D = q.shape
    P, ps, Hkv, _ = k_cache.shape
    out = np.empty((rows.shape[0], D), dtype=np.float64)
    bad = _load().oracle_decode_paged_rows(_ptr(q), Hq * D, D, _ptr(k_cache), _ptr(v_cache),
                                           P, _ptr(bt), bt.shape[1], _ptr(sl), B, Hq, Hkv, D,
                                           ps, float(scale), _ptr(rows), rows.shape[0],
                                           _ptr(out))
    if bad:
        raise ValueError(f"{bad} output rows would read outside the given cache/table")
    return out


def decode_contig(q, k, v, seq_lens, scale: float) -> np.ndarray:
    """Contiguous GQA decode.  k, v [B,max_len,Hkv,D] u16.  Returns [B,Hq,D] float64."""
    q = _u16(q); k = _u16(k); v = _u16(v)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, D = q.shape
    B2, max_len, Hkv, D2 = k.shape
    assert B2 == B and D2 == D and v.shape == k.shape and Hq % Hkv == 0
    out = np.empty((B, Hq, D), dtype=np.float64)
    bad = _load().oracle_decode_contig(_ptr(q), Hq * D, D, _ptr(k), _ptr(v), max_len,
                                       _ptr(sl), B, Hq, Hkv, D, float(scale), _ptr(out))
    if bad:
        raise ValueError(f"{bad} sequences are longer than the contiguous cache")
    return out


def fp8_swa(q, kv_cache, inv_scale, indices, lens, block_size: int, scale: float,
            tokens: tuple[int, int] | None = None) -> np.ndarray:
    """fp8 sliding-window latent decode (K = V).  q [T,NH,HD] u16; kv_cache
    [num_blocks,block_size,HD] u8; inv_scale [num_blocks*block_size] (or [...,1]) u16;
    indices [T,W] int64; lens [T] int64.  Returns [T,NH,HD] float64 (only the rows of
    ``tokens`` = (t0, t1) are filled when given; the rest are NaN)."""
    q = _u16(q)
    cache = np.ascontiguousarray(kv_cache, dtype=np.uint8)
    inv = _u16(np.asarray(inv_scale).reshape(-1))
    idx = np.ascontiguousarray(indices, dtype=np.int64)
    ln = np.ascontiguousarray(lens, dtype=np.int64)
    T, NH, HD = q.shape
    NB, bs, HD2 = cache.shape
    assert HD2 == HD and int(block_size) == bs and inv.shape[0] >= NB * bs
    W = idx.shape[1]
    t0, t1 = (0, T) if tokens is None else tokens
    out = np.full((T, NH, HD), np.nan, dtype=np.float64)
    _load().oracle_fp8_swa_range(_ptr(q), _ptr(cache), _ptr(inv), _ptr(idx), _ptr(ln), T, NH,
                                 HD, W, NB, bs, float(scale), int(t0), int(t1), _ptr(out))
    return out


def e4m3_from_float(x: float) -> int:
    """Nearest E4M3FN code of a binary32 value (ties to even, saturating)."""
    return int(_load().oracle_e4m3_from_float(float(x)))


def kv_append_paged(k_new, v_new, k_cache, v_cache, block_table, pos):
    """Return copies of the caches with each sequence's new K/V rows written at position
    pos[b].  k_new, v_new [B,Hkv,D] u16; caches [P,ps,Hkv,D] u16."""
    k_new = _u16(k_new); v_new = _u16(v_new)
    kc = np.array(k_cache, dtype=np.uint16, copy=True)
    vc = np.array(v_cache, dtype=np.uint16, copy=True)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    ps_ = np.ascontiguousarray(pos, dtype=np.int32)
    B, Hkv, D = k_new.shape
    P, page_size = kc.shape[0], kc.shape[1]
    bad = _load().oracle_kv_append_paged(_ptr(k_new), _ptr(v_new), _ptr(kc), _ptr(vc), P, page_size,
                                         _ptr(bt), bt.shape[1], _ptr(ps_), B, Hkv, D)
    return kc, vc, bad


def kv_append_fp8(rows, kv_cache, inv_scale, slots):
    """Return copies of (kv_cache u8 [NB,bs,HD], inv_scale u16 [NB*bs]) with rows [T,HD]
    quantised into their slots."""
    rows = _u16(rows)
    cache = np.array(kv_cache, dtype=np.uint8, copy=True)
    inv = np.array(np.asarray(inv_scale).reshape(-1), dtype=np.uint16, copy=True)
    sl = np.ascontiguousarray(slots, dtype=np.int64)
    T, HD = rows.shape
    NB, bs, _ = cache.shape
    bad = _load().oracle_kv_append_fp8(_ptr(rows), _ptr(cache), _ptr(inv), _ptr(sl), T, HD, NB, bs)
    return cache, inv, bad


def decode_paged_multi(q, k_cache, v_cache, block_table, seq_lens, qo_indptr, scale: float,
                       mask=None) -> np.ndarray:
    """Multi-token decode: q packed [total_q, Hq, D] u16, qo_indptr [B+1]; token i of
    sequence b attends keys up to position seq_lens[b] - q_len_b + i, and, with a mask
    [total_q, >= max kv_len] (bool / uint8, nonzero = keep), only the kept ones.  Returns
    float64 [total_q, Hq, D]."""
    q = _u16(q); k_cache = _u16(k_cache); v_cache = _u16(v_cache)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qi = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    total, Hq, D = q.shape
    P, ps, Hkv, _ = k_cache.shape
    B = sl.shape[0]
    out = np.empty((total, Hq, D), dtype=np.float64)
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8)
    if m is not None:
        assert m.ndim == 2 and m.shape[0] == total
    bad = _load().oracle_decode_paged_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache), P, _ptr(bt), bt.shape[1],
                                            _ptr(sl), _ptr(qi), None if m is None else _ptr(m),
                                            0 if m is None else m.shape[1], B, Hq, Hkv, D, ps, float(scale),
                                            _ptr(out))
    if bad:
        raise ValueError(f"{bad} output rows would read outside the given cache/table")
    return out


def q_tile_map(q_lens, tokens_per_tile: int):
    """(qo_indptr, tile_batch, tile_index) of the packed-Q work map."""
    ql = np.ascontiguousarray(q_lens, dtype=np.int32)
    B = ql.shape[0]
    cap = int(sum((int(x) + tokens_per_tile - 1) // tokens_per_tile for x in ql)) + 1
    qi = np.zeros(B + 1, np.int32)
    tb = np.zeros(cap, np.int32)
    ti = np.zeros(cap, np.int32)
    n = _load().oracle_q_tile_map(_ptr(ql), B, int(tokens_per_tile), _ptr(qi), _ptr(tb), _ptr(ti), cap)
    return qi, tb[:n], ti[:n]


def decode_paged_fp8kv(q, k_codes, v_codes, k_scale, v_scale, block_table, seq_lens, scale: float) -> np.ndarray:
    """Paged GQA decode over an e4m3 cache: codes [P, ps, Hkv, D] uint8, factors
    [P, Hkv, ps] bf16 bits (uint16); K = e4m3(code) * factor exactly.  q [B, Hq, D] u16.
    Returns float64 [B, Hq, D]."""
    q = _u16(q)
    kc = np.ascontiguousarray(k_codes, dtype=np.uint8)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    ks = _u16(k_scale)
    vs = _u16(v_scale)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, D = q.shape
    P, ps, Hkv, _ = kc.shape
    assert ks.shape == (P, Hkv, ps) and vs.shape == (P, Hkv, ps) and vc.shape == kc.shape
    out = np.empty((B, Hq, D), dtype=np.float64)
    bad = _load().oracle_decode_paged_fp8kv(_ptr(q), Hq * D, D, _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), P, _ptr(bt),
                                            bt.shape[1], _ptr(sl), B, Hq, Hkv, D, ps, float(scale), _ptr(out))
    if bad:
        raise ValueError(f"{bad} output rows would read outside the given cache/table")
    return out


def kv_append_paged_fp8(k_new, v_new, k_codes, v_codes, k_scale, v_scale, block_table, pos):
    """Quantise k_new / v_new [B, Hkv, D] (u16 bits) into the e4m3 GQA cache at pos[b]; the
    code arrays and factor arrays are updated in place (numpy).  Returns rows skipped."""
    kn = _u16(k_new)
    vn = _u16(v_new)
    for a in (k_codes, v_codes):
        assert a.dtype == np.uint8 and a.flags.c_contiguous
    for a in (k_scale, v_scale):
        assert a.dtype == np.uint16 and a.flags.c_contiguous
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    ps_ = np.ascontiguousarray(pos, dtype=np.int32)
    B, Hkv, D = kn.shape
    P, page_size = k_codes.shape[0], k_codes.shape[1]
    return _load().oracle_kv_append_paged_fp8(_ptr(kn), _ptr(vn), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale),
                                              _ptr(v_scale), P, page_size, _ptr(bt), bt.shape[1], _ptr(ps_), B,
                                              Hkv, D)


def decode_paged_masked(q, k_cache, v_cache, block_table, seq_lens, mask, scale: float) -> np.ndarray:
    """Masked paged decode: mask [B, >= max kv_len] (bool / uint8, nonzero = keep); key t of
    sequence b takes part iff t < seq_lens[b] and mask[b, t].  Returns float64 [B, Hq, D]."""
    q = _u16(q); k_cache = _u16(k_cache); v_cache = _u16(v_cache)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    B, Hq, D = q.shape
    P, ps, Hkv, _ = k_cache.shape
    assert m.ndim == 2 and m.shape[0] == B
    out = np.empty((B, Hq, D), dtype=np.float64)
    bad = _load().oracle_decode_paged_masked(_ptr(q), Hq * D, D, _ptr(k_cache), _ptr(v_cache), P, _ptr(bt),
                                             bt.shape[1], _ptr(sl), _ptr(m), m.shape[1], B, Hq, Hkv, D, ps,
                                             float(scale), _ptr(out))
    if bad:
        raise ValueError(f"{bad} output rows would read outside the given cache/table")
    return out
