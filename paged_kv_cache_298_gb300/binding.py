"""Thin Python binding of the C ABI in include/dap.h (ctypes; argument marshalling only).

Every function here takes torch tensors, checks dtypes and devices, and passes raw
pointers, sizes and the current CUDA stream to ``libdap.so``.  All arithmetic runs in the
library's CUDA kernels: there is no fallback, and a missing or unloadable library raises
``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libdap.so")
_lock = threading.Lock()
_lib = None

DAP_OK = 0
STATUS_NAMES = {0: "DAP_OK", 1: "DAP_ERR_NULL", 2: "DAP_ERR_SHAPE", 3: "DAP_ERR_UNSUPPORTED",
                4: "DAP_ERR_WORKSPACE", 5: "DAP_ERR_ALIGN", 6: "DAP_ERR_CUDA", 7: "DAP_ERR_SCRATCH_LIMIT"}
NOALLOC_SCRATCH_BYTES = 16 << 20
DEVERR_TIMEOUT, DEVERR_SEQLEN, DEVERR_PAGE, DEVERR_SLOT, DEVERR_QMAP = 0x1, 0x2, 0x4, 0x8, 0x10

# every symbol include/dap.h declares
EXPORTS = ("dap_status_string", "dap_version", "dap_device_sm_count", "dap_plan_splits",
           "dap_chunk_tokens", "dap_resolve_splits", "dap_workspace_bytes", "decode_attn_paged", "decode_attn_contig",
           "decode_attn_paged_fp8", "decode_attn_paged_noalloc", "kv_append_paged", "kv_append_fp8",
           "dap_set_trace_events", "dap_get_device_errors", "dap_multi_tokens_per_tile",
           "dap_q_tile_map", "dap_workspace_bytes_multi", "decode_attn_paged_multi",
           "decode_attn_paged_fp8kv", "kv_append_paged_fp8", "decode_attn_paged_masked",
           "dap_selftest_wait_timeout")


SPLITS_BALANCED = -1   # include/dap.h: DAP_SPLITS_BALANCED


class DapError(RuntimeError):
    """A library status other than DAP_OK (``status`` is its code), or, with status None, a
    tensor the binding refused before calling the library (not a CUDA tensor, or on another
    device than q)."""

    def __init__(self, status, what: str):
        self.status = status
        if status is None:
            super().__init__(what)
        else:
            super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


def library_path() -> str:
    return _LIB_PATH


def load(build_if_missing: bool = True):
    """Load libdap.so (building it with nvcc when absent or stale, if allowed)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing:
            from . import build as _build
            try:
                _build.build()
            except Exception as e:  # no nvcc or a compile error: fail loudly
                if not os.path.exists(_LIB_PATH):
                    raise RuntimeError(f"libdap.so is missing and could not be built: {e}") from e
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libdap.so not found at {_LIB_PATH}; run __graft_entry__.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, LL, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float, ctypes.c_size_t
        lib.dap_status_string.argtypes = [I]
        lib.dap_status_string.restype = ctypes.c_char_p
        lib.dap_version.argtypes = []
        lib.dap_version.restype = I
        lib.dap_device_sm_count.argtypes = []
        lib.dap_device_sm_count.restype = I
        lib.dap_plan_splits.argtypes = [I, I, I, I, I, I, I, LL]
        lib.dap_plan_splits.restype = I
        lib.dap_chunk_tokens.argtypes = [I, I]
        lib.dap_chunk_tokens.restype = I
        lib.dap_resolve_splits.argtypes = [I, I, I, I, I, I, I, I, LL]
        lib.dap_resolve_splits.restype = I
        lib.dap_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.dap_workspace_bytes.restype = SZ
        lib.decode_attn_paged.argtypes = [P, LL, LL, P, P, I, I, P, I, P, I, I, I, I, I, F, I, P, SZ,
                                          P, LL, LL, P]
        lib.decode_attn_paged.restype = I
        lib.decode_attn_contig.argtypes = [P, LL, LL, P, P, I, P, I, I, I, I, I, F, I, P, SZ, P, LL,
                                           LL, P]
        lib.decode_attn_contig.restype = I
        lib.decode_attn_paged_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P, P]
        lib.decode_attn_paged_fp8.restype = I
        lib.decode_attn_paged_noalloc.argtypes = [P, LL, LL, P, P, I, I, P, I, P, I, I, I, I, I, F, I,
                                                  P, LL, LL, P]
        lib.decode_attn_paged_noalloc.restype = I
        lib.kv_append_paged.argtypes = [P, P, P, P, I, I, P, I, P, I, I, I, P]
        lib.kv_append_paged.restype = I
        lib.kv_append_fp8.argtypes = [P, P, P, P, I, I, I, I, P]
        lib.kv_append_fp8.restype = I
        lib.dap_multi_tokens_per_tile.argtypes = [I, I, I, I]
        lib.dap_multi_tokens_per_tile.restype = I
        lib.dap_q_tile_map.argtypes = [P, I, I, P, P, P, I]
        lib.dap_q_tile_map.restype = I
        lib.dap_workspace_bytes_multi.argtypes = [I, I, I, I]
        lib.dap_workspace_bytes_multi.restype = SZ
        lib.decode_attn_paged_multi.argtypes = [P, LL, LL, P, P, I, I, P, I, P, P, P, P, I, I, I, P, LL, I, I, I,
                                                I, I, F, I, P, SZ, P, LL, LL, P]
        lib.decode_attn_paged_masked.argtypes = [P, LL, LL, P, P, I, I, P, I, P, P, LL, I, I, I, I, I, F, I, P, SZ,
                                                 P, LL, LL, P]
        lib.decode_attn_paged_masked.restype = I
        lib.decode_attn_paged_multi.restype = I
        lib.decode_attn_paged_fp8kv.argtypes = [P, LL, LL, P, P, P, P, I, I, P, I, P, I, I, I, I, I, F, I, P, SZ,
                                                P, LL, LL, P]
        lib.decode_attn_paged_fp8kv.restype = I
        lib.kv_append_paged_fp8.argtypes = [P, P, P, P, P, P, I, I, P, I, P, I, I, I, P]
        lib.kv_append_paged_fp8.restype = I
        lib.dap_set_trace_events.argtypes = [P, P, P]
        lib.dap_set_trace_events.restype = None
        lib.dap_get_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint), I]
        lib.dap_get_device_errors.restype = I
        lib.dap_selftest_wait_timeout.argtypes = [ctypes.c_void_p]
        lib.dap_selftest_wait_timeout.restype = I
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().dap_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != DAP_OK:
        raise DapError(status, what)


def _ptr(t):
    # a plain int: ctypes turns it into the void* argument (cheaper than a c_void_p object)
    return None if t is None else t.data_ptr()


def _device_of(what: str, first, **others) -> torch.device:
    """The CUDA device of `first`; every other tensor given must be a CUDA tensor on it.
    Raises DapError (status None) before the library sees a pointer it could not use: a CPU
    tensor or one on another GPU would reach the kernels as a foreign address."""
    if not getattr(first, "is_cuda", False):
        raise DapError(None, f"{what}: the first tensor must be a CUDA tensor")
    dev = first.device
    idx = dev.index
    for name, t in others.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise DapError(None, f"{what}: {name} is not a CUDA tensor")
        if t.device.index != idx:
            raise DapError(None, f"{what}: {name} is on {t.device}, the call's tensors on {dev}")
    return dev


class _on:
    """Makes `dev` the current device for the library call (skipped when it already is)."""

    def __init__(self, dev):
        self.idx = dev.index
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.idx:
            self.prev = cur
            torch.cuda.set_device(self.idx)

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
        return False


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, dev: torch.device):
    """The stream handle for a call on `dev`: the given stream (which must belong to `dev`)
    or that device's current stream."""
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(dev.index)
        stream = torch.cuda.current_stream(dev)
    elif stream.device.index != dev.index:
        raise DapError(None, f"the stream belongs to {stream.device}, the call's tensors to {dev}")
    return stream.cuda_stream


def _splits(lib, num_splits, units, Hq, Hkv, D, page_size, max_kv_len, total_kv):
    """The split count passed to the library.  num_splits 0 is the planner's choice: the
    library resolves it with the summed lengths unknown; when the caller knows them
    (`total_kv`), the plan is made here with them and passed as an explicit count."""
    S = int(num_splits)
    if S == 0 and total_kv:
        S = lib.dap_resolve_splits(0, lib.dap_device_sm_count(), units, Hq, Hkv, D, page_size, int(max_kv_len),
                                   int(total_kv))
    return S


def _workspace(lib, workspace, S, units, Hq, Hkv, D, page_size, max_kv_len, need_of, dev):
    """The caller's workspace, or one allocated for the split count the call will run
    (dap_resolve_splits); returns (tensor or None, its bytes)."""
    if workspace is None:
        sms = lib.dap_device_sm_count() if S == 0 else 0
        run = lib.dap_resolve_splits(S, sms, units, Hq, Hkv, D, page_size, int(max_kv_len), 0)
        need = need_of(run)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    return workspace, (0 if workspace is None else workspace.numel() * workspace.element_size())


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


# ---- host planning -------------------------------------------------------------------

def device_sm_count() -> int:
    return load().dap_device_sm_count()


def plan_splits(sm_count, B, Hq, Hkv, D, page_size, max_kv_len, total_kv=0) -> int:
    return load().dap_plan_splits(sm_count, B, Hq, Hkv, D, page_size, max_kv_len, total_kv)


def chunk_tokens(max_kv_len, num_splits) -> int:
    return load().dap_chunk_tokens(max_kv_len, num_splits)


def resolve_splits(num_splits, sm_count, B, Hq, Hkv, D, page_size, max_kv_len, total_kv=0) -> int:
    """include/dap.h: dap_resolve_splits (the split count a decode call runs)."""
    return load().dap_resolve_splits(int(num_splits), int(sm_count), int(B), int(Hq), int(Hkv), int(D),
                                     int(page_size), int(max_kv_len), int(total_kv))


def workspace_bytes(B, Hq, Hkv, D, num_splits) -> int:
    return load().dap_workspace_bytes(B, Hq, Hkv, D, num_splits)


def set_trace_events(split_begin=None, split_end=None, combine_end=None):
    """Record torch.cuda.Event objects around the next calls' split / combine kernels."""
    h = lambda e: None if e is None else ctypes.c_void_p(e.cuda_event)
    load().dap_set_trace_events(h(split_begin), h(split_end), h(combine_end))


def get_device_errors(clear: bool = True) -> int:
    v = ctypes.c_uint(0)
    _check(load().dap_get_device_errors(ctypes.byref(v), int(clear)), "dap_get_device_errors")
    return v.value


def selftest_wait_timeout(stream=None) -> None:
    """include/dap.h: dap_selftest_wait_timeout (one bounded wait that runs out on purpose;
    about a second later the device error word holds DEVERR_TIMEOUT)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if stream is None else stream.device
    _check(load().dap_selftest_wait_timeout(_stream(stream, dev)), "dap_selftest_wait_timeout")


# ---- decode entry points ---------------------------------------------------------------

def _bf16_3d(t, name):
    _need(t.dtype == torch.bfloat16 and t.dim() == 3 and t.stride(2) == 1,
          f"{name} must be a bf16 [*, *, D] tensor with unit stride in D")


def _paged_cache(q, k_cache, v_cache, block_table, seq_lens, B):
    _need(k_cache.dtype == torch.bfloat16 and k_cache.dim() == 4 and k_cache.is_contiguous()
          and v_cache.shape == k_cache.shape and v_cache.dtype == torch.bfloat16
          and v_cache.is_contiguous(), "k_cache/v_cache must be contiguous bf16 [P, ps, Hkv, D]")
    _need(k_cache.shape[3] == q.shape[2], "head dims differ")
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.is_contiguous()
          and block_table.shape[0] == B, "block_table must be contiguous int32 [B, max_pages]")
    _need(seq_lens.dtype == torch.int32 and seq_lens.numel() == B and seq_lens.is_contiguous(),
          "seq_lens must be contiguous int32 [B]")
    return k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]


def decode_attn_paged(q, k_cache, v_cache, block_table, seq_lens, *, max_kv_len: int,
                      scale: float | None = None, num_splits: int = 0, total_kv: int = 0, workspace=None,
                      out=None, stream=None):
    """Paged GQA decode (include/dap.h: decode_attn_paged).  num_splits S > 0 = per-sequence
    splits, 0 = the planner's S (made with the summed lengths ``total_kv`` when given),
    SPLITS_BALANCED = the balanced persistent schedule.  Returns ``out`` [B, Hq, D]."""
    _bf16_3d(q, "q")
    B, Hq, D = q.shape
    dev = _device_of("decode_attn_paged", q, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                     seq_lens=seq_lens, workspace=workspace, out=out)
    P, ps, Hkv = _paged_cache(q, k_cache, v_cache, block_table, seq_lens, B)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    _bf16_3d(out, "out")
    lib = load()
    with _on(dev):
        S = _splits(lib, num_splits, B, Hq, Hkv, D, ps, max_kv_len, total_kv)
        workspace, wbytes = _workspace(lib, workspace, S, B, Hq, Hkv, D, ps, max_kv_len,
                                       lambda r: lib.dap_workspace_bytes(B, Hq, Hkv, D, r), dev)
        st = lib.decode_attn_paged(_ptr(q), q.stride(0), q.stride(1), _ptr(k_cache), _ptr(v_cache), P, ps,
                                   _ptr(block_table), block_table.shape[1], _ptr(seq_lens), int(max_kv_len),
                                   B, Hq, Hkv, D, float(scale), int(S), _ptr(workspace), wbytes, _ptr(out),
                                   out.stride(0), out.stride(1), _stream(stream, dev))
    _check(st, "decode_attn_paged")
    return out


def decode_attn_paged_noalloc(q, k_cache, v_cache, block_table, seq_lens, *, max_kv_len: int,
                              scale: float | None = None, num_splits: int = 0, out=None, stream=None):
    """Paged GQA decode without a workspace (include/dap.h: decode_attn_paged_noalloc).

    For callers that cannot give the library scratch memory: the split partials go to a
    fixed 16 MiB device array inside the library (num_splits 0 = the planner's S, lowered
    until its partials fit).  The first call on a device reserves that array (make it at
    start-up); calls that overlap on the GPU race on it, so keep them on one stream.
    Returns ``out`` [B, Hq, D]."""
    _bf16_3d(q, "q")
    B, Hq, D = q.shape
    dev = _device_of("decode_attn_paged_noalloc", q, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                     seq_lens=seq_lens, out=out)
    P, ps, Hkv = _paged_cache(q, k_cache, v_cache, block_table, seq_lens, B)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    _bf16_3d(out, "out")
    with _on(dev):
        st = load().decode_attn_paged_noalloc(_ptr(q), q.stride(0), q.stride(1), _ptr(k_cache), _ptr(v_cache), P,
                                              ps, _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                              int(max_kv_len), B, Hq, Hkv, D, float(scale), int(num_splits),
                                              _ptr(out), out.stride(0), out.stride(1), _stream(stream, dev))
    _check(st, "decode_attn_paged_noalloc")
    return out


def decode_attn_contig(q, k, v, seq_lens, *, max_kv_len: int, scale: float | None = None,
                       num_splits: int = 0, total_kv: int = 0, workspace=None, out=None, stream=None):
    """Contiguous-cache GQA decode (include/dap.h: decode_attn_contig); k, v [B, max_len, Hkv, D].
    num_splits as decode_attn_paged."""
    _bf16_3d(q, "q")
    B, Hq, D = q.shape
    dev = _device_of("decode_attn_contig", q, k=k, v=v, seq_lens=seq_lens, workspace=workspace, out=out)
    _need(k.dtype == torch.bfloat16 and k.dim() == 4 and k.is_contiguous() and v.shape == k.shape
          and v.dtype == torch.bfloat16 and v.is_contiguous() and k.shape[0] == B and k.shape[3] == D,
          "k/v must be contiguous bf16 [B, max_len, Hkv, D]")
    _, max_len, Hkv, _ = k.shape
    _need(seq_lens.dtype == torch.int32 and seq_lens.numel() == B and seq_lens.is_contiguous(),
          "seq_lens must be contiguous int32 [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    _bf16_3d(out, "out")
    lib = load()
    with _on(dev):
        S = _splits(lib, num_splits, B, Hq, Hkv, D, max_len, max_kv_len, total_kv)
        workspace, wbytes = _workspace(lib, workspace, S, B, Hq, Hkv, D, max_len, max_kv_len,
                                       lambda r: lib.dap_workspace_bytes(B, Hq, Hkv, D, r), dev)
        st = lib.decode_attn_contig(_ptr(q), q.stride(0), q.stride(1), _ptr(k), _ptr(v), max_len,
                                    _ptr(seq_lens), int(max_kv_len), B, Hq, Hkv, D, float(scale), int(S),
                                    _ptr(workspace), wbytes, _ptr(out), out.stride(0), out.stride(1),
                                    _stream(stream, dev))
    _check(st, "decode_attn_contig")
    return out


def decode_attn_paged_fp8(q, kv_cache, inv_scale, slot_idx, lens, *, scale: float | None = None,
                          out=None, stream=None):
    """fp8 sliding-window latent decode, K = V (include/dap.h: decode_attn_paged_fp8)."""
    dev = _device_of("decode_attn_paged_fp8", q, kv_cache=kv_cache, inv_scale=inv_scale, slot_idx=slot_idx,
                     lens=lens, out=out)
    _need(q.dtype == torch.bfloat16 and q.dim() == 3 and q.is_contiguous(), "q must be contiguous bf16 [T, NH, HD]")
    T, NH, HD = q.shape
    _need(kv_cache.dtype == torch.uint8 and kv_cache.dim() == 3 and kv_cache.is_contiguous()
          and kv_cache.shape[2] == HD, "kv_cache must be contiguous uint8 [num_blocks, block_size, HD]")
    NB, bs, _ = kv_cache.shape
    _need(inv_scale.dtype == torch.bfloat16 and inv_scale.is_contiguous() and inv_scale.numel() >= NB * bs,
          "inv_scale must be contiguous bf16 with one entry per slot")
    _need(slot_idx.dtype == torch.int64 and slot_idx.dim() == 2 and slot_idx.is_contiguous()
          and slot_idx.shape[0] == T, "slot_idx must be contiguous int64 [T, W]")
    _need(lens.dtype == torch.int64 and lens.numel() == T and lens.is_contiguous(), "lens must be int64 [T]")
    if scale is None:
        scale = 1.0 / math.sqrt(HD)
    if out is None:
        out = torch.empty((T, NH, HD), dtype=torch.bfloat16, device=dev)
    _need(out.dtype == torch.bfloat16 and out.shape == q.shape and out.is_contiguous(), "out must match q")
    with _on(dev):
        st = load().decode_attn_paged_fp8(_ptr(q), _ptr(kv_cache), _ptr(inv_scale), _ptr(slot_idx), _ptr(lens),
                                          T, NH, HD, slot_idx.shape[1], NB, bs, float(scale), _ptr(out),
                                          _stream(stream, dev))
    _check(st, "decode_attn_paged_fp8")
    return out


def decode_attn_paged_masked(q, k_cache, v_cache, block_table, seq_lens, mask, *, max_kv_len: int,
                             scale: float | None = None, num_splits: int = 0, total_kv: int = 0, workspace=None,
                             out=None, stream=None):
    """Masked paged GQA decode (include/dap.h: decode_attn_paged_masked): mask [B, >=
    max_kv_len] bool/uint8, nonzero = keep, rows 16-byte strided.  num_splits 0 = the
    planner's choice (made with ``total_kv`` when given).  Returns ``out``."""
    _bf16_3d(q, "q")
    B, Hq, D = q.shape
    dev = _device_of("decode_attn_paged_masked", q, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                     seq_lens=seq_lens, mask=mask, workspace=workspace, out=out)
    P, ps, Hkv = _paged_cache(q, k_cache, v_cache, block_table, seq_lens, B)
    mask = _mask(mask, B, int(max_kv_len))
    _need(mask is not None, "mask is required")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    _bf16_3d(out, "out")
    lib = load()
    with _on(dev):
        S = _splits(lib, num_splits, B, Hq, Hkv, D, ps, max_kv_len, total_kv)
        workspace, wbytes = _workspace(lib, workspace, S, B, Hq, Hkv, D, ps, max_kv_len,
                                       lambda r: lib.dap_workspace_bytes(B, Hq, Hkv, D, r), dev)
        st = lib.decode_attn_paged_masked(_ptr(q), q.stride(0), q.stride(1), _ptr(k_cache), _ptr(v_cache), P, ps,
                                          _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(mask),
                                          mask.stride(0), int(max_kv_len), B, Hq, Hkv, D, float(scale), int(S),
                                          _ptr(workspace), wbytes, _ptr(out), out.stride(0), out.stride(1),
                                          _stream(stream, dev))
    _check(st, "decode_attn_paged_masked")
    return out


# ---- GQA decode over an fp8 (e4m3) cache -----------------------------------------------

def _fp8kv_cache(k_codes, v_codes, k_scale, v_scale):
    _need(k_codes.dtype == torch.uint8 and k_codes.dim() == 4 and k_codes.is_contiguous()
          and v_codes.shape == k_codes.shape and v_codes.dtype == torch.uint8 and v_codes.is_contiguous(),
          "k_codes/v_codes must be contiguous uint8 [P, ps, Hkv, D]")
    P, ps, Hkv, D = k_codes.shape
    for f in (k_scale, v_scale):
        _need(f.dtype == torch.bfloat16 and f.is_contiguous() and tuple(f.shape) == (P, Hkv, ps),
              "k_scale/v_scale must be contiguous bf16 [P, Hkv, ps]")
    return P, ps, Hkv, D


def decode_attn_paged_fp8kv(q, k_codes, v_codes, k_scale, v_scale, block_table, seq_lens, *, max_kv_len: int,
                            scale: float | None = None, num_splits: int = 0, total_kv: int = 0, workspace=None,
                            out=None, stream=None):
    """Paged GQA decode over an e4m3 K/V cache (include/dap.h: decode_attn_paged_fp8kv).
    num_splits 0 = the planner's choice (made with the host-known sum of seq_lens
    ``total_kv`` when given).  Returns ``out`` [B, Hq, D]."""
    _bf16_3d(q, "q")
    B, Hq, D = q.shape
    dev = _device_of("decode_attn_paged_fp8kv", q, k_codes=k_codes, v_codes=v_codes, k_scale=k_scale,
                     v_scale=v_scale, block_table=block_table, seq_lens=seq_lens, workspace=workspace, out=out)
    P, ps, Hkv, D2 = _fp8kv_cache(k_codes, v_codes, k_scale, v_scale)
    _need(D2 == D, "head dims differ")
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.is_contiguous()
          and block_table.shape[0] == B, "block_table must be contiguous int32 [B, max_pages]")
    _need(seq_lens.dtype == torch.int32 and seq_lens.numel() == B and seq_lens.is_contiguous(),
          "seq_lens must be contiguous int32 [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    _bf16_3d(out, "out")
    lib = load()
    with _on(dev):
        S = _splits(lib, num_splits, B, Hq, Hkv, D, ps, max_kv_len, total_kv)
        workspace, wbytes = _workspace(lib, workspace, S, B, Hq, Hkv, D, ps, max_kv_len,
                                       lambda r: lib.dap_workspace_bytes(B, Hq, Hkv, D, r), dev)
        st = lib.decode_attn_paged_fp8kv(_ptr(q), q.stride(0), q.stride(1), _ptr(k_codes), _ptr(v_codes),
                                         _ptr(k_scale), _ptr(v_scale), P, ps, _ptr(block_table), block_table.shape[1],
                                         _ptr(seq_lens), int(max_kv_len), B, Hq, Hkv, D, float(scale), int(S),
                                         _ptr(workspace), wbytes, _ptr(out), out.stride(0), out.stride(1),
                                         _stream(stream, dev))
    _check(st, "decode_attn_paged_fp8kv")
    return out


# ---- multi-token decode ------------------------------------------------------------------

def multi_tokens_per_tile(Hq: int, Hkv: int, max_q_len: int = 0, D: int = 0) -> int:
    """include/dap.h: dap_multi_tokens_per_tile (16 / G; for longer new-token runs 128 / G
    where the head dim D has the 128-row tiles (64, 128, 256), else 32 / G; D = 0: not known)."""
    return load().dap_multi_tokens_per_tile(int(Hq), int(Hkv), int(D), int(max_q_len))


def workspace_bytes_multi(total_q, Hq, D, num_splits) -> int:
    return load().dap_workspace_bytes_multi(int(total_q), int(Hq), int(D), int(num_splits))


def q_tile_map(q_lens, tokens_per_tile: int):
    """Host work map of the packed new tokens (include/dap.h: dap_q_tile_map).
    Returns int32 CPU tensors (qo_indptr [B+1], tile_batch [n], tile_index [n])."""
    ql = torch.as_tensor(q_lens, dtype=torch.int32).cpu().contiguous().reshape(-1)
    B = ql.numel()
    cap = sum((int(x) + tokens_per_tile - 1) // tokens_per_tile for x in ql.tolist() if x > 0)
    qi = torch.zeros(B + 1, dtype=torch.int32)
    tb = torch.zeros(max(cap, 1), dtype=torch.int32)
    ti = torch.zeros(max(cap, 1), dtype=torch.int32)
    n = load().dap_q_tile_map(_ptr(ql), B, int(tokens_per_tile), _ptr(qi), _ptr(tb), _ptr(ti), cap)
    _need(n >= 0, "invalid q_lens or tokens_per_tile")
    return qi, tb[:n].clone(), ti[:n].clone()


class MultiPlan:
    """The work map of one batch of new-token counts, copied to the device once so that
    repeated decode calls on the same counts pass it straight to the library.  Without
    tokens_per_tile the library's rule picks it from the longest count and the head dim D
    (None: not known, so no 128-row tiles)."""

    def __init__(self, q_lens, Hq: int, Hkv: int, device, tokens_per_tile: int | None = None,
                 D: int | None = None):
        ql = [int(x) for x in torch.as_tensor(q_lens).reshape(-1).tolist()]
        if tokens_per_tile is None:
            tokens_per_tile = multi_tokens_per_tile(Hq, Hkv, max(ql, default=0), D or 0)
        self.tokens_per_tile = int(tokens_per_tile)
        _need(self.tokens_per_tile > 0, "Hq must be a multiple of Hkv with G <= 16")
        qi, tb, ti = q_tile_map(q_lens, self.tokens_per_tile)
        self.B = qi.numel() - 1
        self.total_q = int(qi[-1])
        self.num_tiles = tb.numel()
        self.qo_indptr = qi.to(device)
        self.tile_batch = tb.to(device)
        self.tile_index = ti.to(device)


def _mask(mask, rows, max_kv_len):
    if mask is None:
        return None
    _need(mask.dtype in (torch.uint8, torch.bool) and mask.dim() == 2 and mask.shape[0] == rows
          and mask.stride(1) == 1 and mask.stride(0) >= max(1, max_kv_len) and mask.stride(0) % 16 == 0,
          "mask must be bool/uint8 [rows, >= max_kv_len] with unit inner stride and a row stride "
          "that is a multiple of 16 bytes")
    return mask


def decode_attn_paged_multi(q, k_cache, v_cache, block_table, seq_lens, plan: MultiPlan, *, max_kv_len: int,
                            scale: float | None = None, num_splits: int = 0, total_kv: int = 0, mask=None,
                            workspace=None, out=None, stream=None):
    """Multi-token causal decode over a paged cache (include/dap.h: decode_attn_paged_multi).
    q [total_q, Hq, D] holds the new tokens of all sequences back to back; ``plan`` is the
    MultiPlan of their counts.  num_splits 0 = the planner's choice over the plan's tiles
    (made with the host-known sum of seq_lens ``total_kv`` when given).  Returns ``out``
    [total_q, Hq, D]."""
    _bf16_3d(q, "q")
    total_q, Hq, D = q.shape
    _need(total_q == plan.total_q, "q rows differ from the plan's token count")
    dev = _device_of("decode_attn_paged_multi", q, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                     seq_lens=seq_lens, qo_indptr=plan.qo_indptr, tile_batch=plan.tile_batch,
                     tile_index=plan.tile_index, mask=mask, workspace=workspace, out=out)
    B = plan.B
    P, ps, Hkv = _paged_cache(q, k_cache, v_cache, block_table, seq_lens, B)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((total_q, Hq, D), dtype=torch.bfloat16, device=dev)
    _bf16_3d(out, "out")
    lib = load()
    mask = _mask(mask, total_q, int(max_kv_len))
    with _on(dev):
        S = _splits(lib, num_splits, max(plan.num_tiles, 0), Hq, Hkv, D, ps, max_kv_len, total_kv)
        workspace, wbytes = _workspace(lib, workspace, S, max(plan.num_tiles, 0), Hq, Hkv, D, ps, max_kv_len,
                                       lambda r: lib.dap_workspace_bytes_multi(total_q, Hq, D, r), dev)
        st = lib.decode_attn_paged_multi(_ptr(q), q.stride(0), q.stride(1), _ptr(k_cache), _ptr(v_cache), P, ps,
                                         _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                         _ptr(plan.qo_indptr), _ptr(plan.tile_batch), _ptr(plan.tile_index),
                                         plan.num_tiles, plan.tokens_per_tile, total_q, _ptr(mask),
                                         0 if mask is None else mask.stride(0),
                                         int(max_kv_len), B, Hq, Hkv, D, float(scale), int(S), _ptr(workspace),
                                         wbytes, _ptr(out), out.stride(0), out.stride(1), _stream(stream, dev))
    _check(st, "decode_attn_paged_multi")
    return out


# ---- cache writes ------------------------------------------------------------------------

def kv_append_paged(k_new, v_new, k_cache, v_cache, block_table, positions, *, stream=None):
    """Write each sequence's new K/V rows [B, Hkv, D] at positions[b] (include/dap.h:
    kv_append_paged).  Returns (k_cache, v_cache), updated in place."""
    dev = _device_of("kv_append_paged", k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                     block_table=block_table, positions=positions)
    _need(k_new.dtype == torch.bfloat16 and k_new.dim() == 3 and k_new.is_contiguous()
          and v_new.shape == k_new.shape and v_new.dtype == torch.bfloat16 and v_new.is_contiguous(),
          "k_new/v_new must be contiguous bf16 [B, Hkv, D]")
    B, Hkv, D = k_new.shape
    _need(k_cache.dtype == torch.bfloat16 and k_cache.dim() == 4 and k_cache.is_contiguous()
          and v_cache.shape == k_cache.shape and v_cache.is_contiguous() and k_cache.shape[2:] == (Hkv, D),
          "caches must be contiguous bf16 [P, ps, Hkv, D]")
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.is_contiguous()
          and block_table.shape[0] == B, "block_table must be contiguous int32 [B, max_pages]")
    _need(positions.dtype == torch.int32 and positions.numel() == B and positions.is_contiguous(),
          "positions must be contiguous int32 [B]")
    with _on(dev):
        st = load().kv_append_paged(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                    k_cache.shape[1], _ptr(block_table), block_table.shape[1], _ptr(positions), B,
                                    Hkv, D, _stream(stream, dev))
    _check(st, "kv_append_paged")
    return k_cache, v_cache


def kv_append_fp8(rows, kv_cache, inv_scale, slots, *, stream=None):
    """Quantise rows [T, HD] into their fp8 cache slots (include/dap.h: kv_append_fp8).
    Returns (kv_cache, inv_scale), updated in place."""
    dev = _device_of("kv_append_fp8", rows, kv_cache=kv_cache, inv_scale=inv_scale, slots=slots)
    _need(rows.dtype == torch.bfloat16 and rows.dim() == 2 and rows.is_contiguous(), "rows must be bf16 [T, HD]")
    T, HD = rows.shape
    _need(kv_cache.dtype == torch.uint8 and kv_cache.dim() == 3 and kv_cache.is_contiguous()
          and kv_cache.shape[2] == HD, "kv_cache must be contiguous uint8 [num_blocks, block_size, HD]")
    NB, bs, _ = kv_cache.shape
    _need(inv_scale.dtype == torch.bfloat16 and inv_scale.is_contiguous() and inv_scale.numel() >= NB * bs,
          "inv_scale must be contiguous bf16 with one entry per slot")
    _need(slots.dtype == torch.int64 and slots.numel() == T and slots.is_contiguous(), "slots must be int64 [T]")
    with _on(dev):
        st = load().kv_append_fp8(_ptr(rows), _ptr(kv_cache), _ptr(inv_scale), _ptr(slots), T, HD, NB, bs,
                                  _stream(stream, dev))
    _check(st, "kv_append_fp8")
    return kv_cache, inv_scale


def kv_append_paged_fp8(k_new, v_new, k_codes, v_codes, k_scale, v_scale, block_table, positions, *, stream=None):
    """Quantise each sequence's new K/V rows [B, Hkv, D] into the e4m3 GQA cache at
    positions[b] (include/dap.h: kv_append_paged_fp8).  Returns the four cache arrays,
    updated in place."""
    dev = _device_of("kv_append_paged_fp8", k_new, v_new=v_new, k_codes=k_codes, v_codes=v_codes, k_scale=k_scale,
                     v_scale=v_scale, block_table=block_table, positions=positions)
    _need(k_new.dtype == torch.bfloat16 and k_new.dim() == 3 and k_new.is_contiguous()
          and v_new.shape == k_new.shape and v_new.dtype == torch.bfloat16 and v_new.is_contiguous(),
          "k_new/v_new must be contiguous bf16 [B, Hkv, D]")
    B, Hkv, D = k_new.shape
    P, ps, Hkv2, D2 = _fp8kv_cache(k_codes, v_codes, k_scale, v_scale)
    _need((Hkv2, D2) == (Hkv, D), "cache heads / dims differ from the new rows")
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.is_contiguous()
          and block_table.shape[0] == B, "block_table must be contiguous int32 [B, max_pages]")
    _need(positions.dtype == torch.int32 and positions.numel() == B and positions.is_contiguous(),
          "positions must be contiguous int32 [B]")
    with _on(dev):
        st = load().kv_append_paged_fp8(_ptr(k_new), _ptr(v_new), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale),
                                        _ptr(v_scale), P, ps, _ptr(block_table), block_table.shape[1],
                                        _ptr(positions), B, Hkv, D, _stream(stream, dev))
    _check(st, "kv_append_paged_fp8")
    return k_codes, v_codes, k_scale, v_scale
