"""Oracle for the paged KV cache hot path -- TEST INFRASTRUCTURE ONLY.

A plain fp64 CPU restatement (``oracle.c``) of what the paged KV cache
computes, plus this thin ctypes wrapper.  Only the test suite, the package
smoke check and the benchmark's CPU-baseline leg use it; the CUDA library
never imports it, and the two share no code.

Functions (each cites the passage it restates in ``oracle.c``):

* ``slot_of``                -- slot of one logical position
  (nano-vLLM lab manual §5.2.3 / appendix B.2.3; nano-vllm KV-cache post §3.1).
* ``decode_slot_mapping``    -- one new token per sequence at position
  ``context_len - 1``; padding rows get -1 (lab manual §5.2.1 and B.4;
  KV-cache post §4.4).
* ``kv_store``               -- store_kvcache bit copy, slot -1 skipped
  (MinivLLM review, "注意力内核的三个分支").
* ``paged_decode``           -- q_len = 1 GQA attention over the paged cache in
  fp64 (mini-vLLM README §5; lab manual appendix B.1.2).
* ``partial_state`` / ``merge_states`` -- split-K state (m, l, acc) of a token
  range and its merge (the online-softmax state of mini-vLLM README §5).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

_lib = None

OK, EINVAL, EBOUNDS = 0, -1, -5


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc into ``liboracle.so`` (no CUDA involved)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_version.restype = ctypes.c_int
    lib.oracle_slot_of.argtypes = [P, i32, i32, i64, P]
    lib.oracle_decode_slot_mapping.argtypes = [P, i32, P, i32, i32, i32, P]
    lib.oracle_kv_store.argtypes = [P, P, P, i32, P, P, i64, i32]
    lib.oracle_paged_decode.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, f64, P, i32]
    lib.oracle_partial_state.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f64,
                                         i32, i32, P, P, P]
    lib.oracle_merge_states.argtypes = [P, P, P, i32, i32, P]
    lib.oracle_copy_blocks.argtypes = [P, P, P, i32, i32, i64]
    lib.oracle_e4m3_decode.argtypes = [P, i64, P]
    lib.oracle_e4m3_encode.argtypes = [P, i64, P]
    lib.oracle_kv_store_fp8.argtypes = [P, P, P, i32, P, P, i64, i32, i32, P, P]
    lib.oracle_paged_attention.argtypes = [P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32, f64, P, i32]
    lib.oracle_paged_decode_fp8.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, f64, P, i32]
    for name in ("oracle_slot_of", "oracle_decode_slot_mapping", "oracle_kv_store",
                 "oracle_paged_decode", "oracle_partial_state", "oracle_merge_states"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise OracleError(f"{what}: oracle status {rc}")


def slot_of(block_table_row, block_size: int, pos: int) -> int:
    row = _c(block_table_row, np.int32)
    out = np.zeros(1, np.int64)
    _check(_load().oracle_slot_of(_ptr(row), row.size, block_size, pos, _ptr(out)), "slot_of")
    return int(out[0])


def decode_slot_mapping(block_tables, context_lens, block_size: int, num_tokens: int | None = None) -> np.ndarray:
    bt = _c(block_tables, np.int32)
    ctx = _c(context_lens, np.int32)
    B = ctx.size
    T = B if num_tokens is None else int(num_tokens)
    out = np.empty(T, np.int32)
    _check(_load().oracle_decode_slot_mapping(_ptr(bt), bt.shape[1], _ptr(ctx), B, block_size, T, _ptr(out)),
           "decode_slot_mapping")
    return out


def kv_store(k_bits, v_bits, slot_mapping, k_cache_bits, v_cache_bits) -> None:
    """In-place store into ``k_cache_bits``/``v_cache_bits`` (uint16 bf16 bit arrays)."""
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    slots = _c(slot_mapping, np.int32)
    for c in (k_cache_bits, v_cache_bits):
        if c.dtype != np.uint16 or not c.flags.c_contiguous:
            raise OracleError("caches must be C-contiguous uint16 arrays")
    T = slots.size
    row = int(np.prod(k_cache_bits.shape[2:]))
    num_slots = k_cache_bits.shape[0] * k_cache_bits.shape[1]
    _check(_load().oracle_kv_store(_ptr(k), _ptr(v), _ptr(slots), T, _ptr(k_cache_bits), _ptr(v_cache_bits),
                                   num_slots, row), "kv_store")


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of E4M3 codes (uint8), NaN for 0x7F / 0xFF."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _check(_load().oracle_e4m3_decode(_ptr(c), c.size, _ptr(out)), "e4m3_decode")
    return out


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes (uint8) of float32 values: nearest, ties to even, saturating at +-448."""
    f = _c(x, np.float32)
    out = np.empty(f.shape, np.uint8)
    _check(_load().oracle_e4m3_encode(_ptr(f), f.size, _ptr(out)), "e4m3_encode")
    return out


def kv_store_fp8(k_bits, v_bits, slot_mapping, k_cache8, v_cache8, k_scale, v_scale) -> None:
    """In-place store into E4M3 caches (uint8 [NB, bs, Hkv, D]) of bf16 rows divided by per-head scales."""
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    slots = _c(slot_mapping, np.int32)
    ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
    for c in (k_cache8, v_cache8):
        if c.dtype != np.uint8 or not c.flags.c_contiguous:
            raise OracleError("fp8 caches must be C-contiguous uint8 arrays")
    NB, bs, Hkv, D = k_cache8.shape
    _check(_load().oracle_kv_store_fp8(_ptr(k), _ptr(v), _ptr(slots), slots.size, _ptr(k_cache8), _ptr(v_cache8),
                                       NB * bs, Hkv, D, _ptr(ks), _ptr(vs)), "kv_store_fp8")


def paged_decode_fp8(q_bits, k_cache8, v_cache8, k_scale, v_scale, block_tables, context_lens, scale: float,
                     nthreads: int = 1) -> np.ndarray:
    """fp64 output [B, Hq, D] of decode attention over E4M3 caches with per-kv-head scales."""
    q = _c(q_bits, np.uint16)
    kc, vc = _c(k_cache8, np.uint8), _c(v_cache8, np.uint8)
    ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
    bt = _c(block_tables, np.int32)
    ctx = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = kc.shape
    out = np.empty((B, Hq, D), np.float64)
    _check(_load().oracle_paged_decode_fp8(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt), bt.shape[1],
                                           _ptr(ctx), B, Hq, Hkv, D, bs, NB, float(scale), _ptr(out),
                                           int(nthreads)), "paged_decode_fp8")
    return out


def paged_attention(q_bits, k_cache_bits, v_cache_bits, block_tables, cu_seqlens_q, context_lens, scale: float,
                    nthreads: int = 1) -> np.ndarray:
    """fp64 output [T, Hq, D]: causal attention of each sequence's last n new tokens (query rows
    cu_seqlens_q[b] .. cu_seqlens_q[b+1]) over its L = context_lens[b] cached tokens."""
    q = _c(q_bits, np.uint16)
    kc, vc = _c(k_cache_bits, np.uint16), _c(v_cache_bits, np.uint16)
    bt = _c(block_tables, np.int32)
    cu = _c(cu_seqlens_q, np.int32)
    ctx = _c(context_lens, np.int32)
    T, Hq, D = q.shape
    B = ctx.size
    if cu.size != B + 1 or int(cu[-1]) != T:
        raise OracleError("cu_seqlens_q must have B + 1 entries ending at the number of query rows")
    NB, bs, Hkv, _ = kc.shape
    out = np.empty((T, Hq, D), np.float64)
    _check(_load().oracle_paged_attention(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cu), _ptr(ctx), B,
                                          Hq, Hkv, D, bs, NB, float(scale), _ptr(out), int(nthreads)),
           "paged_attention")
    return out


def copy_blocks(k_cache_bits, v_cache_bits, pairs) -> None:
    """In place: for each (src, dst) row of ``pairs`` in order, block dst of both caches becomes a bit
    copy of block src.  Raises on an id outside the pool (the other pairs are still applied)."""
    for c in (k_cache_bits, v_cache_bits):
        if c.dtype != np.uint16 or not c.flags.c_contiguous:
            raise OracleError("caches must be C-contiguous uint16 arrays")
    pr = _c(np.asarray(pairs, np.int32).reshape(-1, 2), np.int32)
    NB = k_cache_bits.shape[0]
    elems = int(np.prod(k_cache_bits.shape[1:]))
    _check(_load().oracle_copy_blocks(_ptr(k_cache_bits), _ptr(v_cache_bits), _ptr(pr), pr.shape[0], NB, elems),
           "copy_blocks")


def paged_decode(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens, scale: float,
                 nthreads: int = 1) -> np.ndarray:
    """fp64 output [B, Hq, D] for bf16-bit inputs q [B, Hq, D], caches [NB, bs, Hkv, D]."""
    q = _c(q_bits, np.uint16)
    kc = _c(k_cache_bits, np.uint16)
    vc = _c(v_cache_bits, np.uint16)
    bt = _c(block_tables, np.int32)
    ctx = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = kc.shape
    if D2 != D or vc.shape != kc.shape or bt.shape[0] != B or ctx.size != B:
        raise OracleError("shape mismatch")
    out = np.zeros((B, Hq, D), np.float64)
    _check(_load().oracle_paged_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(ctx), B, Hq, Hkv,
                                       D, bs, NB, float(scale), _ptr(out), int(nthreads)), "paged_decode")
    return out


def partial_state(q_bits, k_cache_bits, v_cache_bits, block_tables, b: int, h: int, scale: float, j0: int, j1: int):
    q = _c(q_bits, np.uint16)
    kc = _c(k_cache_bits, np.uint16)
    vc = _c(v_cache_bits, np.uint16)
    bt = _c(block_tables, np.int32)
    _, Hq, D = q.shape
    NB, bs, Hkv, _ = kc.shape
    m = np.zeros(1)
    l = np.zeros(1)
    acc = np.zeros(D)
    _check(_load().oracle_partial_state(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], b, h, Hq, Hkv, D, bs,
                                        NB, float(scale), j0, j1, _ptr(m), _ptr(l), _ptr(acc)), "partial_state")
    return float(m[0]), float(l[0]), acc


def merge_states(ms, ls, accs) -> np.ndarray:
    m = _c(ms, np.float64)
    l = _c(ls, np.float64)
    acc = _c(accs, np.float64)
    n = m.size
    D = acc.shape[-1]
    out = np.zeros(D)
    _check(_load().oracle_merge_states(_ptr(m), _ptr(l), _ptr(acc), n, D, _ptr(out)), "merge_states")
    return out
