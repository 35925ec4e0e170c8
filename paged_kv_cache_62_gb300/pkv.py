"""ctypes binding of ``libpkv.so`` (declared in ``include/pkv.h``).

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (device memory and streams come from torch);
shapes and dtypes are checked here, then raw device pointers go through the
C ABI.  There is no fallback: if the library is missing or the tensors are not
on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

OK, EINVAL, EUNSUPPORTED, ECUDA, EWORKSPACE, EBOUNDS, EFULL = 0, -1, -2, -3, -4, -5, -6
ERR_SLOT_RANGE, ERR_BLOCK_RANGE, ERR_CONTEXT_RANGE, ERR_WAIT_TIMEOUT, ERR_WORKSPACE = 0x1, 0x2, 0x4, 0x8, 0x10
MAX_SEQS, MAX_WORKERS = 16384, 4096

# name -> (restype, argtypes), mirroring include/pkv.h
_P, _I32, _SZ, _F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "pkv_abi_version": (ctypes.c_int, []),
    "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_last_cuda_error": (ctypes.c_char_p, []),
    "pkv_decode_slot_mapping": (ctypes.c_int, [_P, _I32, _P, _I32, _I32, _I32, _P, _I32, _P, _P]),
    "pkv_kv_store": (ctypes.c_int, [_P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _P, _P]),
    "pkv_paged_decode_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "pkv_paged_decode": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                                        _F32, _P, _P, _SZ, _I32, _P, _P]),
    "pkv_paged_decode_store": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32,
                                              _I32, _I32, _F32, _P, _P, _P, _SZ, _I32, _P, _P]),
    "pkv_paged_decode_store_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32,
                                                  _I32, _I32, _I32, _I32, _F32, _P, _P, _P, _SZ, _I32, _P, _P]),
    "pkv_paged_decode_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                                                _I32, _F32, _P, _I32, _P, _P]),
    "pkv_diag_wait_timeout": (ctypes.c_int, [_P, _P]),
    "pkv_copy_blocks": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P]),
    "pkv_paged_attention_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "pkv_paged_attention": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                                           _I32, _F32, _P, _I32, _P, _SZ, _I32, _P, _P]),
    "pkv_decode_store": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P]),
    "pkv_kv_store_fp8": (ctypes.c_int, [_P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P]),
    "pkv_paged_decode_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                                            _I32, _F32, _P, _P, _SZ, _I32, _P, _P]),
    "pkv_allocator_create": (_P, [_I32, _I32]),
    "pkv_allocator_destroy": (None, [_P]),
    "pkv_allocator_add": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32]),
    "pkv_allocator_fork": (ctypes.c_int, [_P, _I32, _I32]),
    "pkv_allocator_append": (ctypes.c_int, [_P, _I32, _P, _P]),
    "pkv_allocator_free": (ctypes.c_int, [_P, _I32]),
    "pkv_allocator_num_free": (_I32, [_P]),
    "pkv_allocator_ref_count": (_I32, [_P, _I32]),
    "pkv_allocator_num_tokens": (_I32, [_P, _I32]),
    "pkv_allocator_tables": (ctypes.c_int, [_P, _P, _I32, _P, _I32, _P]),
}
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

_lib = None


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        detail = f" [{load().pkv_last_cuda_error().decode()}]" if status == ECUDA else ""
        super().__init__(f"{what}: {status_string(status)} (status {status}){detail}")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libpkv.so (built by ``paged_kv_cache_62_gb300.build``); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libpkv.so not found at {p}: build it with `python -m paged_kv_cache_62_gb300.build`")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise PkvError(status, what)


def _dev(t: torch.Tensor, dtype, name: str, ndim: int | None = None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t.data_ptr()


def _opt(t) -> int | None:
    return None if t is None else _dev(t, torch.int32, "err_word")


def _stream(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def decode_slot_mapping(block_tables: torch.Tensor, context_lens: torch.Tensor, block_size: int, num_blocks: int,
                        slot_mapping: torch.Tensor, err_word: torch.Tensor | None = None, stream=None) -> None:
    """Slot of each sequence's appended token (position context_len - 1); rows beyond the batch get -1."""
    B, mb = block_tables.shape
    _check(load().pkv_decode_slot_mapping(
        _dev(block_tables, torch.int32, "block_tables", 2), mb, _dev(context_lens, torch.int32, "context_lens", 1),
        B, int(block_size), int(num_blocks), _dev(slot_mapping, torch.int32, "slot_mapping", 1),
        slot_mapping.numel(), _opt(err_word), _stream(stream)), "pkv_decode_slot_mapping")


def kv_store(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
             v_cache: torch.Tensor, err_word: torch.Tensor | None = None, stream=None) -> None:
    """store_kvcache: k_cache/v_cache[slot] = k/v[t] for every slot != -1."""
    T, Hkv, D = k.shape
    NB, bs, Hkv2, D2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or (Hkv2, D2) != (Hkv, D) or slot_mapping.numel() != T:
        raise ValueError("kv_store: shape mismatch")
    _check(load().pkv_kv_store(
        _dev(k, torch.bfloat16, "k", 3), _dev(v, torch.bfloat16, "v", 3),
        _dev(slot_mapping, torch.int32, "slot_mapping", 1), T,
        _dev(k_cache, torch.bfloat16, "k_cache", 4), _dev(v_cache, torch.bfloat16, "v_cache", 4),
        NB, bs, Hkv, D, _opt(err_word), _stream(stream)), "pkv_kv_store")


def paged_decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    n = load().pkv_paged_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim)
    if n == 0:
        raise PkvError(EINVAL, "pkv_paged_decode_workspace_size")
    return int(n)


def alloc_workspace(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int, device=None) -> torch.Tensor:
    """A decode workspace, zero-filled as the library requires before its first use."""
    n = paged_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def paged_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                 context_lens: torch.Tensor, scale: float, out: torch.Tensor, workspace: torch.Tensor,
                 max_context_len: int | None = None, num_workers: int = 0, err_word: torch.Tensor | None = None,
                 stream=None) -> None:
    """Decode PagedAttention: out[b, h] = softmax(scale * q[b, h] K^T) V over the paged cache."""
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or block_tables.shape[0] != B or context_lens.numel() != B \
            or out.shape != q.shape:
        raise ValueError("paged_decode: shape mismatch")
    mb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = mb * bs
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA uint8 tensor")
    _check(load().pkv_paged_decode(
        _dev(q, torch.bfloat16, "q", 3), _dev(k_cache, torch.bfloat16, "k_cache", 4),
        _dev(v_cache, torch.bfloat16, "v_cache", 4), _dev(block_tables, torch.int32, "block_tables", 2), mb,
        _dev(context_lens, torch.int32, "context_lens", 1), B, Hq, Hkv, D, bs, NB, int(max_context_len),
        float(scale), _dev(out, torch.bfloat16, "out", 3), workspace.data_ptr(), workspace.numel(),
        int(num_workers), _opt(err_word), _stream(stream)), "pkv_paged_decode")


def paged_decode_store(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                       v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                       out: torch.Tensor, workspace: torch.Tensor, slot_mapping: torch.Tensor | None = None,
                       max_context_len: int | None = None, num_workers: int = 0,
                       err_word: torch.Tensor | None = None, stream=None) -> None:
    """A decode step in one launch: store row b of k_new / v_new at position context_lens[b] - 1 of
    sequence b and attend over 0..context_lens[b] - 1 (pkv_decode_store + pkv_paged_decode)."""
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or block_tables.shape[0] != B or context_lens.numel() != B \
            or out.shape != q.shape or k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) \
            or (slot_mapping is not None and slot_mapping.numel() != B):
        raise ValueError("paged_decode_store: shape mismatch")
    mb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = mb * bs
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA uint8 tensor")
    _check(load().pkv_paged_decode_store(
        _dev(q, torch.bfloat16, "q", 3), _dev(k_new, torch.bfloat16, "k_new", 3),
        _dev(v_new, torch.bfloat16, "v_new", 3), _dev(k_cache, torch.bfloat16, "k_cache", 4),
        _dev(v_cache, torch.bfloat16, "v_cache", 4), _dev(block_tables, torch.int32, "block_tables", 2), mb,
        _dev(context_lens, torch.int32, "context_lens", 1), B, Hq, Hkv, D, bs, NB, int(max_context_len),
        float(scale), _dev(out, torch.bfloat16, "out", 3),
        None if slot_mapping is None else _dev(slot_mapping, torch.int32, "slot_mapping", 1),
        workspace.data_ptr(), workspace.numel(), int(num_workers), _opt(err_word), _stream(stream)),
        "pkv_paged_decode_store")


class DecodeStoreStep:
    """A decode step (paged_decode_store) bound to persistent buffers: the arguments are checked once, here,
    and run() issues the C call with them, so a serving loop that reuses its buffers step after step (as a
    CUDA-graph engine does) pays no per-call checks.  The buffers' contents may change between runs; their
    shapes, dtypes and addresses may not (make a new step for new buffers).  max_context_len must bound every
    run's context_lens (run() takes a new bound)."""

    _MAXLEN = 14  # position of max_context_len in pkv_paged_decode_store's arguments

    def __init__(self, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out, workspace,
                 slot_mapping=None, max_context_len=None, num_workers=0, err_word=None):
        B, Hq, D = q.shape
        NB, bs, Hkv, D2 = k_cache.shape
        if D2 != D or v_cache.shape != k_cache.shape or block_tables.shape[0] != B or context_lens.numel() != B \
                or out.shape != q.shape or k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) \
                or (slot_mapping is not None and slot_mapping.numel() != B):
            raise ValueError("DecodeStoreStep: shape mismatch")
        mb = block_tables.shape[1]
        if max_context_len is None:
            max_context_len = mb * bs
        if workspace.dtype != torch.uint8 or not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA uint8 tensor")
        self._fn = load().pkv_paged_decode_store
        self._args = [
            _dev(q, torch.bfloat16, "q", 3), _dev(k_new, torch.bfloat16, "k_new", 3),
            _dev(v_new, torch.bfloat16, "v_new", 3), _dev(k_cache, torch.bfloat16, "k_cache", 4),
            _dev(v_cache, torch.bfloat16, "v_cache", 4), _dev(block_tables, torch.int32, "block_tables", 2), mb,
            _dev(context_lens, torch.int32, "context_lens", 1), B, Hq, Hkv, D, bs, NB, int(max_context_len),
            float(scale), _dev(out, torch.bfloat16, "out", 3),
            None if slot_mapping is None else _dev(slot_mapping, torch.int32, "slot_mapping", 1),
            workspace.data_ptr(), workspace.numel(), int(num_workers), _opt(err_word)]
        # the tensors stay referenced as long as the step exists
        self._keep = (q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, workspace, slot_mapping,
                      err_word)

    def run(self, stream=None, max_context_len: int | None = None) -> None:
        """Issue the step on `stream` (a torch stream, a raw cudaStream_t handle as an int, or None for the
        current stream)."""
        if max_context_len is not None:
            self._args[self._MAXLEN] = int(max_context_len)
        st = stream if isinstance(stream, int) else _stream(stream)
        status = self._fn(*self._args, st)
        if status != OK:
            raise PkvError(status, "pkv_paged_decode_store")


def paged_decode_store_fp8(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                           v_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                           workspace: torch.Tensor, slot_mapping: torch.Tensor | None = None,
                           max_context_len: int | None = None, num_workers: int = 0,
                           err_word: torch.Tensor | None = None, stream=None) -> None:
    """paged_decode_store over E4M3 caches (uint8 [NB, bs, Hkv, D]) with per-kv-head float32 scales: the new
    rows (bf16) are quantised as kv_store_fp8 does, stored and attended in one launch."""
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or block_tables.shape[0] != B or context_lens.numel() != B \
            or out.shape != q.shape or k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) \
            or k_scale.numel() != Hkv or v_scale.numel() != Hkv \
            or (slot_mapping is not None and slot_mapping.numel() != B):
        raise ValueError("paged_decode_store_fp8: shape mismatch")
    mb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = mb * bs
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA uint8 tensor")
    _check(load().pkv_paged_decode_store_fp8(
        _dev(q, torch.bfloat16, "q", 3), _dev(k_new, torch.bfloat16, "k_new", 3),
        _dev(v_new, torch.bfloat16, "v_new", 3), _dev(k_cache, torch.uint8, "k_cache", 4),
        _dev(v_cache, torch.uint8, "v_cache", 4), _dev(k_scale, torch.float32, "k_scale"),
        _dev(v_scale, torch.float32, "v_scale"), _dev(block_tables, torch.int32, "block_tables", 2), mb,
        _dev(context_lens, torch.int32, "context_lens", 1), B, Hq, Hkv, D, bs, NB, int(max_context_len),
        float(scale), _dev(out, torch.bfloat16, "out", 3),
        None if slot_mapping is None else _dev(slot_mapping, torch.int32, "slot_mapping", 1),
        workspace.data_ptr(), workspace.numel(), int(num_workers), _opt(err_word), _stream(stream)),
        "pkv_paged_decode_store_fp8")


def diag_wait_timeout(err_word: torch.Tensor, stream=None) -> None:
    """Diagnostic: a bounded wait that runs out on purpose; sets ERR_WAIT_TIMEOUT in err_word after the wait's
    limit."""
    _check(load().pkv_diag_wait_timeout(_dev(err_word, torch.int32, "err_word"), _stream(stream)),
           "pkv_diag_wait_timeout")


def paged_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                         context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                         max_context_len: int | None = None, num_workers: int = 0,
                         err_word: torch.Tensor | None = None, stream=None) -> None:
    """paged_decode without a caller workspace: the library's fixed per-device scratch is used.

    For callers that cannot allocate device memory.  Calls that overlap on the
    GPU share that scratch and race; the first call on a device should come
    before any stream capture.
    """
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or block_tables.shape[0] != B or context_lens.numel() != B \
            or out.shape != q.shape:
        raise ValueError("paged_decode_noalloc: shape mismatch")
    mb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = mb * bs
    _check(load().pkv_paged_decode_noalloc(
        _dev(q, torch.bfloat16, "q", 3), _dev(k_cache, torch.bfloat16, "k_cache", 4),
        _dev(v_cache, torch.bfloat16, "v_cache", 4), _dev(block_tables, torch.int32, "block_tables", 2), mb,
        _dev(context_lens, torch.int32, "context_lens", 1), B, Hq, Hkv, D, bs, NB, int(max_context_len),
        float(scale), _dev(out, torch.bfloat16, "out", 3), int(num_workers), _opt(err_word), _stream(stream)),
        "pkv_paged_decode_noalloc")


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, pairs: torch.Tensor,
                err_word: torch.Tensor | None = None, stream=None) -> None:
    """Copy-on-write copies: for each row (src, dst) of ``pairs`` (int32 [n, 2], device), block dst of
    both caches becomes a bit copy of block src."""
    NB, bs, Hkv, D = k_cache.shape
    if v_cache.shape != k_cache.shape or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("copy_blocks: shape mismatch")
    _check(load().pkv_copy_blocks(
        _dev(k_cache, torch.bfloat16, "k_cache", 4), _dev(v_cache, torch.bfloat16, "v_cache", 4),
        _dev(pairs, torch.int32, "pairs", 2), pairs.shape[0], NB, bs, Hkv, D, _opt(err_word), _stream(stream)),
        "pkv_copy_blocks")


class BlockAllocator:
    """Host-side block allocator of the library (reference counts, copy-on-write; see include/pkv.h)."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = load()
        self._h = self._lib.pkv_allocator_create(int(num_blocks), int(block_size))
        if not self._h:
            raise ValueError(f"pkv_allocator_create({num_blocks}, {block_size}) failed")
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self) -> None:
        if self._h:
            self._lib.pkv_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add(self, seq_id: int, num_tokens: int, parent_id: int = -1, shared_blocks: int = 0) -> None:
        _check(self._lib.pkv_allocator_add(self._h, seq_id, num_tokens, parent_id, shared_blocks),
               "pkv_allocator_add")

    def fork(self, parent_id: int, child_id: int) -> None:
        _check(self._lib.pkv_allocator_fork(self._h, parent_id, child_id), "pkv_allocator_fork")

    def append(self, seq_id: int) -> tuple[int, int]:
        """One token for seq_id; returns the (src, dst) copy-on-write pair, (-1, -1) if none."""
        src, dst = ctypes.c_int32(-1), ctypes.c_int32(-1)
        _check(self._lib.pkv_allocator_append(self._h, seq_id, ctypes.byref(src), ctypes.byref(dst)),
               "pkv_allocator_append")
        return src.value, dst.value

    def free(self, seq_id: int) -> None:
        _check(self._lib.pkv_allocator_free(self._h, seq_id), "pkv_allocator_free")

    def num_free(self) -> int:
        return self._lib.pkv_allocator_num_free(self._h)

    def ref_count(self, block_id: int) -> int:
        return self._lib.pkv_allocator_ref_count(self._h, block_id)

    def num_tokens(self, seq_id: int) -> int:
        return self._lib.pkv_allocator_num_tokens(self._h, seq_id)

    def tables(self, seq_ids, max_blocks: int):
        """(block_tables int32 [n, max_blocks] -1 padded, context_lens int32 [n]) as host tensors."""
        ids = torch.as_tensor(list(seq_ids), dtype=torch.int32)
        bt = torch.empty(len(ids), max_blocks, dtype=torch.int32)
        lens = torch.empty(len(ids), dtype=torch.int32)
        _check(self._lib.pkv_allocator_tables(self._h, ids.data_ptr(), len(ids), bt.data_ptr(), int(max_blocks),
                                              lens.data_ptr()), "pkv_allocator_tables")
        return bt, lens


def kv_store_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                 err_word: torch.Tensor | None = None, stream=None) -> None:
    """kv_store into E4M3 caches (uint8 [NB, bs, Hkv, D]) with per-kv-head float32 scales."""
    T, Hkv, D = k.shape
    NB, bs, Hkv2, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or v.shape != k.shape or v_cache.shape != k_cache.shape or slot_mapping.numel() != T \
            or k_scale.numel() != Hkv or v_scale.numel() != Hkv:
        raise ValueError("kv_store_fp8: shape mismatch")
    _check(load().pkv_kv_store_fp8(
        _dev(k, torch.bfloat16, "k", 3), _dev(v, torch.bfloat16, "v", 3), _dev(slot_mapping, torch.int32, "slot_mapping"),
        T, _dev(k_cache, torch.uint8, "k_cache", 4), _dev(v_cache, torch.uint8, "v_cache", 4), NB, bs, Hkv, D,
        _dev(k_scale, torch.float32, "k_scale"), _dev(v_scale, torch.float32, "v_scale"), _opt(err_word),
        _stream(stream)), "pkv_kv_store_fp8")


def paged_decode_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor,
                     v_scale: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                     out: torch.Tensor, workspace: torch.Tensor, max_context_len: int | None = None,
                     num_workers: int = 0, err_word: torch.Tensor | None = None, stream=None) -> None:
    """paged_decode over E4M3 caches (uint8 [NB, bs, Hkv, D]) with per-kv-head float32 scales."""
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or block_tables.shape[0] != B or context_lens.numel() != B \
            or out.shape != q.shape or k_scale.numel() != Hkv or v_scale.numel() != Hkv:
        raise ValueError("paged_decode_fp8: shape mismatch")
    mx = int(block_tables.shape[1]) * bs if max_context_len is None else int(max_context_len)
    _check(load().pkv_paged_decode_fp8(
        _dev(q, torch.bfloat16, "q", 3), _dev(k_cache, torch.uint8, "k_cache", 4), _dev(v_cache, torch.uint8, "v_cache", 4),
        _dev(k_scale, torch.float32, "k_scale"), _dev(v_scale, torch.float32, "v_scale"),
        _dev(block_tables, torch.int32, "block_tables", 2), block_tables.shape[1],
        _dev(context_lens, torch.int32, "context_lens"), B, Hq, Hkv, D, bs, NB, mx, float(scale),
        _dev(out, torch.bfloat16, "out", 3), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        int(num_workers), _opt(err_word), _stream(stream)), "pkv_paged_decode_fp8")


def decode_store(k: torch.Tensor, v: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                 k_cache: torch.Tensor, v_cache: torch.Tensor, slot_mapping: torch.Tensor | None = None,
                 err_word: torch.Tensor | None = None, stream=None) -> None:
    """A decode step's slot computation and store in one launch (row b -> position context_lens[b] - 1)."""
    B, Hkv, D = k.shape
    NB, bs, Hkv2, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or v.shape != k.shape or v_cache.shape != k_cache.shape or \
            block_tables.shape[0] != B or context_lens.numel() != B or \
            (slot_mapping is not None and slot_mapping.numel() != B):
        raise ValueError("decode_store: shape mismatch")
    sm = None if slot_mapping is None else _dev(slot_mapping, torch.int32, "slot_mapping")
    _check(load().pkv_decode_store(
        _dev(k, torch.bfloat16, "k", 3), _dev(v, torch.bfloat16, "v", 3), _dev(block_tables, torch.int32, "block_tables", 2),
        block_tables.shape[1], _dev(context_lens, torch.int32, "context_lens"), B,
        _dev(k_cache, torch.bfloat16, "k_cache", 4), _dev(v_cache, torch.bfloat16, "v_cache", 4), NB, bs, Hkv, D, sm,
        _opt(err_word), _stream(stream)), "pkv_decode_store")


def alloc_attention_workspace(num_rows: int, num_q_heads: int, num_kv_heads: int, head_dim: int, device=None):
    """A zero-filled workspace for paged_attention with num_rows query rows."""
    n = load().pkv_paged_attention_workspace_size(num_rows, num_q_heads, num_kv_heads, head_dim)
    if n == 0:
        raise ValueError("paged_attention: unsupported sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def paged_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                    cu_seqlens_q: torch.Tensor | None, context_lens: torch.Tensor, scale: float, out: torch.Tensor,
                    workspace: torch.Tensor, max_context_len: int | None = None, num_workers: int = 0,
                    err_word: torch.Tensor | None = None, stream=None, new_per_seq: int = 0) -> None:
    """Causal paged attention of each sequence's new tokens (rows cu_seqlens_q[b]..cu_seqlens_q[b+1], or
    b*n..b*n+n-1 with new_per_seq = n) over its context_lens[b] cached tokens."""
    T, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    B = context_lens.numel()
    if D2 != D or v_cache.shape != k_cache.shape or block_tables.shape[0] != B or out.shape != q.shape \
            or (cu_seqlens_q is None and new_per_seq <= 0) \
            or (cu_seqlens_q is not None and cu_seqlens_q.numel() != B + 1):
        raise ValueError("paged_attention: shape mismatch")
    cu = None if cu_seqlens_q is None else _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    mx = int(block_tables.shape[1]) * bs if max_context_len is None else int(max_context_len)
    _check(load().pkv_paged_attention(
        _dev(q, torch.bfloat16, "q", 3), _dev(k_cache, torch.bfloat16, "k_cache", 4),
        _dev(v_cache, torch.bfloat16, "v_cache", 4), _dev(block_tables, torch.int32, "block_tables", 2),
        block_tables.shape[1], cu,
        _dev(context_lens, torch.int32, "context_lens"), B, T, Hq, Hkv, D, bs, NB, mx, float(scale),
        _dev(out, torch.bfloat16, "out", 3), int(new_per_seq), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(),
        int(num_workers), _opt(err_word), _stream(stream)), "pkv_paged_attention")
