"""ctypes binding of ``libpda.so`` (declared in ``include/pda.h``).

Argument marshalling only: tensors become device pointers, the stream becomes
a ``cudaStream_t`` handle, statuses become exceptions. Every step of the decode
path runs in the library's CUDA kernels. If the library has not been built the
first call raises; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpda.so")

(PDA_OK, PDA_ERR_INVALID_ARG, PDA_ERR_UNSUPPORTED, PDA_ERR_WORKSPACE, PDA_ERR_CUDA,
 PDA_ERR_OUT_OF_BLOCKS) = range(6)
PDA_FP16, PDA_BF16 = 0, 1
PDA_KIND_GQA, PDA_KIND_MLA = 0, 1
PDA_KV_SAME_AS_Q, PDA_KV_FP8_E4M3 = 0, 1

_lib = None


class PdaError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        super().__init__(f"{func} failed with {status_name(status)}: {detail}")
        self.status = status


class Problem(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("dtype", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim_qk", ctypes.c_int32), ("head_dim_v", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_blocks", ctypes.c_int64), ("num_sms", ctypes.c_int32),
                ("force_num_ctas", ctypes.c_int32), ("kv_format", ctypes.c_int32),
                ("seq_len_q", ctypes.c_int32)]


def _declare(lib):
    P, I32, I64, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    sig = {
        "pda_plan_create": (I32, [ctypes.POINTER(P), ctypes.POINTER(Problem), P]),
        "pda_plan_destroy": (None, [P]),
        "pda_plan_workspace_bytes": (SZ, [P]),
        "pda_plan_num_ctas": (I32, [P]),
        "pda_plan_num_splits": (I32, [P, I32]),
        "pda_plan_num_launches": (I32, [P]),
        "pda_workspace_init": (I32, [P, P, P]),
        "pda_read_device_error": (I32, [P, P, ctypes.POINTER(I32)]),
        "paged_decode_attn": (I32, [P, P, P, P, P, F32, P, P, P, P, P]),
        "paged_decode_attn_fp8": (I32, [P, P, P, F32, F32, P, P, F32, P, P, P, P, P]),
        "mla_decode": (I32, [P, P, P, P, F32, P, P, P, P, P]),
        "mla_decode_fp8": (I32, [P, P, F32, P, P, F32, P, P, P, P, P]),
        "pda_combine_splits": (I32, [P, P, I32, I32, I32, P, I32, P, P]),
        "paged_decode_attn_no_alloc": (I32, [P, P, P, P, P, F32, P, P, P, P]),
        "pda_no_alloc_read_device_error": (I32, [P, P]),
        "pda_kv_append": (I32, [P, P, P, P, P, P, P, P, P]),
        "pda_kv_append_fp8": (I32, [P, P, P, P, F32, F32, P, P, P, P, P]),
        "pda_mla_append_fp8": (I32, [P, P, F32, P, P, P, P, P]),
        "pda_mla_append": (I32, [P, P, P, P, P, P, P]),
        "pda_pool_create": (I32, [ctypes.POINTER(P), I64]),
        "pda_pool_destroy": (None, [P]),
        "pda_pool_num_free": (I64, [P]),
        "pda_pool_grow": (I32, [P, P, I32, I32, I32, I32]),
        "pda_pool_release": (I32, [P, P, I32, I32]),
        "pda_status_string": (ctypes.c_char_p, [I32]),
        "pda_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args


def lib():
    """The loaded library (loads it on first use; raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run paged_kv_cache_61_gb300.build.build() "
                               "(the decode path has no CPU fallback)")
        handle = ctypes.CDLL(LIB_PATH)
        _declare(handle)
        _lib = handle
    return _lib


def status_name(status: int) -> str:
    try:
        return lib().pda_status_string(status).decode()
    except Exception:  # pragma: no cover - only for messages
        return str(status)


def _check(status: int, func: str):
    if status != PDA_OK:
        raise PdaError(status, func, lib().pda_last_error().decode())


def _ptr(x) -> Optional[int]:
    """Device pointer of a tensor (or an int address, or None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("tensors passed to libpda must be contiguous")
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owns a ``pda_plan`` (see ``pda_plan_create`` in ``include/pda.h``)."""

    def __init__(self, *, kind: int, dtype: int, batch: int, num_q_heads: int, num_kv_heads: int,
                 head_dim_qk: int, head_dim_v: int, page_size: int, max_blocks_per_seq: int,
                 num_blocks: int, context_lens: Sequence[int], num_sms: int = 0,
                 force_num_ctas: int = 0, kv_format: int = PDA_KV_SAME_AS_Q,
                 seq_len_q: int = 1):
        self.problem = Problem(kind, dtype, batch, num_q_heads, num_kv_heads, head_dim_qk,
                               head_dim_v, page_size, max_blocks_per_seq, num_blocks, num_sms,
                               force_num_ctas, kv_format, seq_len_q)
        ctx = (ctypes.c_int32 * max(1, len(context_lens)))(*[int(c) for c in context_lens])
        handle = ctypes.c_void_p()
        _check(lib().pda_plan_create(ctypes.byref(handle), ctypes.byref(self.problem),
                                     ctx if batch > 0 else None), "pda_plan_create")
        self.handle = handle

    @property
    def workspace_bytes(self) -> int:
        return int(lib().pda_plan_workspace_bytes(self.handle))

    @property
    def num_ctas(self) -> int:
        return int(lib().pda_plan_num_ctas(self.handle))

    @property
    def num_launches(self) -> int:
        """Kernel launches of one decode call (2 when a split-merge kernel follows)."""
        return int(lib().pda_plan_num_launches(self.handle))

    def num_splits(self, b: int) -> int:
        return int(lib().pda_plan_num_splits(self.handle, b))

    def close(self):
        if getattr(self, "handle", None):
            lib().pda_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def workspace_init(plan: Plan, workspace, stream=None):
    _check(lib().pda_workspace_init(plan.handle, _ptr(workspace), _stream(stream)),
           "pda_workspace_init")


def read_device_error(workspace, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(lib().pda_read_device_error(_ptr(workspace), _stream(stream), ctypes.byref(code)),
           "pda_read_device_error")
    return int(code.value)


def paged_decode_attn(q, k_cache, v_cache, block_tables, context_lens, scale: float, out, lse,
                      plan: Plan, workspace, stream=None):
    _check(lib().paged_decode_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                   _ptr(context_lens), float(scale), _ptr(out), _ptr(lse),
                                   plan.handle, _ptr(workspace), _stream(stream)),
           "paged_decode_attn")


def paged_decode_attn_fp8(q, k_cache, v_cache, k_scale: float, v_scale: float, block_tables,
                          context_lens, scale: float, out, lse, plan: Plan, workspace,
                          stream=None):
    """paged_decode_attn over E4M3 caches (uint8 codes) with per-tensor scales."""
    _check(lib().paged_decode_attn_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), float(k_scale),
                                       float(v_scale), _ptr(block_tables), _ptr(context_lens),
                                       float(scale), _ptr(out), _ptr(lse), plan.handle,
                                       _ptr(workspace), _stream(stream)),
           "paged_decode_attn_fp8")


def paged_decode_attn_no_alloc(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                               out, lse, plan: Plan, stream=None):
    """paged_decode_attn without a workspace (library-owned scratch; see include/pda.h)."""
    _check(lib().paged_decode_attn_no_alloc(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                            _ptr(block_tables), _ptr(context_lens), float(scale),
                                            _ptr(out), _ptr(lse), plan.handle, _stream(stream)),
           "paged_decode_attn_no_alloc")


def no_alloc_read_device_error(stream=None) -> int:
    """Read and clear the error word of paged_decode_attn_no_alloc's library array."""
    code = ctypes.c_int32(0)
    _check(lib().pda_no_alloc_read_device_error(_stream(stream), ctypes.byref(code)),
           "pda_no_alloc_read_device_error")
    return int(code.value)


def mla_decode(q, kv_cache, block_tables, context_lens, scale: float, out, lse, plan: Plan,
               workspace, stream=None):
    _check(lib().mla_decode(_ptr(q), _ptr(kv_cache), _ptr(block_tables), _ptr(context_lens),
                            float(scale), _ptr(out), _ptr(lse), plan.handle, _ptr(workspace),
                            _stream(stream)), "mla_decode")


def mla_decode_fp8(q, kv_cache, kv_scale: float, block_tables, context_lens, scale: float, out,
                   lse, plan: Plan, workspace, stream=None):
    """mla_decode over an E4M3 record cache (uint8 codes) with its per-tensor scale."""
    _check(lib().mla_decode_fp8(_ptr(q), _ptr(kv_cache), float(kv_scale), _ptr(block_tables),
                                _ptr(context_lens), float(scale), _ptr(out), _ptr(lse),
                                plan.handle, _ptr(workspace), _stream(stream)),
           "mla_decode_fp8")


def combine_splits(partial_out, partial_lse, rows: int, num_splits: int, head_dim_v: int, out,
                   out_dtype: int, lse, stream=None):
    _check(lib().pda_combine_splits(_ptr(partial_out), _ptr(partial_lse), rows, num_splits,
                                    head_dim_v, _ptr(out), out_dtype, _ptr(lse), _stream(stream)),
           "pda_combine_splits")


def kv_append(k_new, v_new, k_cache, v_cache, block_tables, context_lens, plan: Plan, workspace,
              stream=None):
    """Write the S new tokens of each sequence into 16-bit GQA caches (see include/pda.h)."""
    _check(lib().pda_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                               _ptr(block_tables), _ptr(context_lens), plan.handle,
                               _ptr(workspace), _stream(stream)), "pda_kv_append")


def kv_append_fp8(k_new, v_new, k_cache, v_cache, k_scale: float, v_scale: float, block_tables,
                  context_lens, plan: Plan, workspace, stream=None):
    """kv_append into E4M3 caches: codes of value / scale."""
    _check(lib().pda_kv_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                   float(k_scale), float(v_scale), _ptr(block_tables),
                                   _ptr(context_lens), plan.handle, _ptr(workspace),
                                   _stream(stream)), "pda_kv_append_fp8")


def mla_append(kv_new, kv_cache, block_tables, context_lens, plan: Plan, workspace, stream=None):
    """Write the S new MLA records of each sequence into the latent cache."""
    _check(lib().pda_mla_append(_ptr(kv_new), _ptr(kv_cache), _ptr(block_tables),
                                _ptr(context_lens), plan.handle, _ptr(workspace),
                                _stream(stream)), "pda_mla_append")


def mla_append_fp8(kv_new, kv_cache, kv_scale: float, block_tables, context_lens, plan: Plan,
                   workspace, stream=None):
    """mla_append into an E4M3 record cache (uint8 codes of value / kv_scale)."""
    _check(lib().pda_mla_append_fp8(_ptr(kv_new), _ptr(kv_cache), float(kv_scale),
                                    _ptr(block_tables), _ptr(context_lens), plan.handle,
                                    _ptr(workspace), _stream(stream)), "pda_mla_append_fp8")


class BlockPool:
    """Owns a ``pda_block_pool``: the free list of physical blocks behind block tables.

    Table rows are int32 numpy arrays (host memory) that the calls update in place.
    """

    def __init__(self, num_blocks: int):
        handle = ctypes.c_void_p()
        _check(lib().pda_pool_create(ctypes.byref(handle), int(num_blocks)), "pda_pool_create")
        self.handle = handle

    @property
    def num_free(self) -> int:
        return int(lib().pda_pool_num_free(self.handle))

    @staticmethod
    def _row(row):
        import numpy as np
        if not (isinstance(row, np.ndarray) and row.dtype == np.int32 and row.flags.c_contiguous):
            raise ValueError("table rows must be contiguous int32 numpy arrays")
        return row.ctypes.data

    def grow(self, table_row, page_size: int, old_len: int, new_len: int):
        _check(lib().pda_pool_grow(self.handle, self._row(table_row), int(table_row.shape[0]),
                                   int(page_size), int(old_len), int(new_len)), "pda_pool_grow")

    def release(self, table_row, page_size: int, length: int):
        _check(lib().pda_pool_release(self.handle, self._row(table_row), int(page_size),
                                      int(length)), "pda_pool_release")

    def close(self):
        if getattr(self, "handle", None):
            lib().pda_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
