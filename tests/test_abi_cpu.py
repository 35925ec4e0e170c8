"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_cache_62_gb300 import build as pkv_build
from paged_kv_cache_62_gb300 import pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("pkv_decode_slot_mapping", "pkv_kv_store", "pkv_paged_decode", "pkv_paged_decode_workspace_size",
                 "pkv_status_string", "pkv_abi_version"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT (pkv_\w+)", out.stdout))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    assert set(pkv.SIGNATURES) == set(declared_functions())


def test_version_and_status_strings(lib):
    assert lib.pkv_abi_version() == 2
    for st in (0, -1, -2, -3, -4, -5, 42):
        assert lib.pkv_status_string(st)


def test_workspace_size_host_arithmetic(lib):
    f = lib.pkv_paged_decode_workspace_size
    assert f(64, 16, 8, 128) > 0
    assert f(64, 16, 8, 128) < f(128, 16, 8, 128)
    assert f(0, 16, 8, 128) > 0
    assert f(-1, 16, 8, 128) == 0
    assert f(64, 16, 6, 128) == 0          # 16 % 6 != 0
    assert f(pkv.MAX_SEQS + 1, 16, 8, 128) == 0
    # holds every split-K partial: (max workers + B*Hkv) slots of G*(D + 2) floats, plus a 64-bit
    # arrival counter per (sequence, kv head)
    B, Hq, Hkv, D = 64, 16, 8, 128
    assert f(B, Hq, Hkv, D) >= (pkv.MAX_WORKERS + B * Hkv) * (Hq // Hkv) * (D + 2) * 4 + B * Hkv * 8


NULL = None
FAKE = 0x10000  # never dereferenced: every call below is rejected before touching the device


def decode_args(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mb=4, lens=FAKE, B=2, Hq=16, Hkv=8, D=128, bs=16, NB=10, maxctx=64,
             scale=0.1, out=FAKE, ws=FAKE, wsb=1 << 30, workers=0, err=NULL, stream=NULL)
    a.update(kw)
    return [a[k] for k in ("q", "k", "v", "bt", "mb", "lens", "B", "Hq", "Hkv", "D", "bs", "NB", "maxctx", "scale",
                           "out", "ws", "wsb", "workers", "err", "stream")]


@pytest.mark.parametrize("kw,status", [
    (dict(q=NULL), pkv.EINVAL),
    (dict(out=NULL), pkv.EINVAL),
    (dict(Hq=12), pkv.EINVAL),                 # 12 % 8
    (dict(D=96), pkv.EUNSUPPORTED),
    (dict(Hq=136, Hkv=8), pkv.EUNSUPPORTED),   # group of 17 (bf16 caches take up to 16)
    (dict(bs=12), pkv.EUNSUPPORTED),
    (dict(bs=4), pkv.EUNSUPPORTED),
    (dict(bs=2048), pkv.EUNSUPPORTED),
    (dict(B=-1), pkv.EINVAL),
    (dict(B=pkv.MAX_SEQS + 1), pkv.EBOUNDS),
    (dict(maxctx=-1), pkv.EINVAL),
    (dict(workers=-1), pkv.EINVAL),
    (dict(workers=pkv.MAX_WORKERS + 1), pkv.EBOUNDS),
    (dict(scale=float("nan")), pkv.EINVAL),
    (dict(q=FAKE + 8), pkv.EINVAL),            # misaligned
    (dict(ws=NULL), pkv.EWORKSPACE),
    (dict(wsb=16), pkv.EWORKSPACE),
    (dict(NB=1 << 27, bs=256), pkv.EBOUNDS),       # rows beyond int32
])
def test_paged_decode_host_validation(lib, kw, status):
    assert lib.pkv_paged_decode(*decode_args(**kw)) == status


def test_paged_decode_empty_batch_is_noop(lib):
    assert lib.pkv_paged_decode(*decode_args(B=0, q=NULL, out=NULL, ws=NULL)) == pkv.OK


def test_kv_store_host_validation(lib):
    f = lib.pkv_kv_store
    assert f(NULL, FAKE, FAKE, 4, FAKE, FAKE, 10, 16, 8, 128, NULL, NULL) == pkv.EINVAL
    assert f(FAKE, FAKE, FAKE, -1, FAKE, FAKE, 10, 16, 8, 128, NULL, NULL) == pkv.EINVAL
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 10, 16, 1, 4, NULL, NULL) == pkv.EINVAL   # 8-byte rows
    assert f(FAKE + 4, FAKE, FAKE, 4, FAKE, FAKE, 10, 16, 8, 128, NULL, NULL) == pkv.EINVAL
    assert f(NULL, NULL, NULL, 0, NULL, NULL, 10, 16, 8, 128, NULL, NULL) == pkv.OK


def test_slot_mapping_host_validation(lib):
    f = lib.pkv_decode_slot_mapping
    assert f(FAKE, 4, FAKE, 8, 16, 10, FAKE, 4, NULL, NULL) == pkv.EINVAL   # fewer tokens than seqs
    assert f(FAKE, 4, FAKE, 2, 12, 10, FAKE, 4, NULL, NULL) == pkv.EINVAL   # block size not a power of 2
    assert f(FAKE, 0, FAKE, 2, 16, 10, FAKE, 4, NULL, NULL) == pkv.EINVAL
    assert f(NULL, 4, NULL, 0, 16, 10, NULL, 0, NULL, NULL) == pkv.OK


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(2, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkv.paged_decode(q, torch.zeros(4, 16, 8, 128, dtype=torch.bfloat16),
                         torch.zeros(4, 16, 8, 128, dtype=torch.bfloat16), torch.zeros(2, 4, dtype=torch.int32),
                         torch.zeros(2, dtype=torch.int32), 0.1, torch.empty_like(q), torch.empty(16, dtype=torch.uint8))


def test_bound_step_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    t = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    kv = torch.zeros(2, 2, 64, dtype=torch.bfloat16)
    cache = torch.zeros(8, 16, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkv.DecodeStoreStep(t, kv, kv, cache, cache, torch.zeros(2, 4, dtype=torch.int32),
                            torch.zeros(2, dtype=torch.int32), 0.1, t.clone(), torch.zeros(64, dtype=torch.uint8))


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        pkv.load(str(tmp_path / "libpkv.so"))


def test_newer_entry_points_validate_on_the_host(lib):
    """Rejected before any CUDA call (FAKE pointers are never dereferenced), or no-ops when empty."""
    # pkv_decode_store(k, v, bt, max_blocks, lens, B, kc, vc, NB, bs, Hkv, D, slots, err, stream)
    ds = lib.pkv_decode_store
    assert ds(FAKE, FAKE, FAKE, 4, FAKE, 2, FAKE, FAKE, 10, 12, 8, 128, NULL, NULL, NULL) == pkv.EINVAL   # bs not 2^k
    assert ds(NULL, FAKE, FAKE, 4, FAKE, 2, FAKE, FAKE, 10, 16, 8, 128, NULL, NULL, NULL) == pkv.EINVAL
    assert ds(FAKE + 8, FAKE, FAKE, 4, FAKE, 2, FAKE, FAKE, 10, 16, 8, 128, NULL, NULL, NULL) == pkv.EINVAL
    assert ds(NULL, NULL, NULL, 4, NULL, 0, NULL, NULL, 10, 16, 8, 128, NULL, NULL, NULL) == pkv.OK
    # pkv_paged_decode_store(q, k_new, v_new, kc, vc, bt, max_blocks, lens, B, Hq, Hkv, D, bs, NB, max_ctx,
    #                        scale, out, slots, ws, ws_bytes, workers, err, stream)
    pds = lib.pkv_paged_decode_store
    tail = [FAKE, 4, FAKE, 2, 16, 8, 128, 16, 10, 64, 0.1, FAKE, NULL, FAKE, 1 << 30, 0, NULL, NULL]
    assert pds(FAKE, NULL, FAKE, FAKE, FAKE, *tail) == pkv.EINVAL          # no k_new
    assert pds(FAKE, FAKE + 8, FAKE, FAKE, FAKE, *tail) == pkv.EINVAL      # k_new not 16-byte aligned
    assert pds(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 0, 16, 8, 128, 16, 10, 64, 0.1, FAKE, NULL, FAKE,
               1 << 30, 0, NULL, NULL) == pkv.OK                          # empty batch
    # pkv_paged_decode_store_fp8(q, k_new, v_new, kc8, vc8, ks, vs, bt, max_blocks, lens, B, Hq, Hkv, D, bs, NB,
    #                            max_ctx, scale, out, slots, ws, ws_bytes, workers, err, stream)
    pf = lib.pkv_paged_decode_store_fp8
    tail8 = [FAKE, 4, FAKE, 2, 16, 8, 128, 16, 10, 64, 0.1, FAKE, NULL, FAKE, 1 << 30, 0, NULL, NULL]
    assert pf(FAKE, NULL, FAKE, FAKE, FAKE, FAKE, FAKE, *tail8) == pkv.EINVAL     # no k_new
    assert pf(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, *tail8) == pkv.EINVAL     # no k_scale
    assert lib.pkv_diag_wait_timeout(NULL, NULL) == pkv.EINVAL
    # pkv_kv_store_fp8(k, v, slots, T, kc8, vc8, NB, bs, Hkv, D, ks, vs, err, stream)
    kf = lib.pkv_kv_store_fp8
    assert kf(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 10, 16, 8, 128, NULL, FAKE, NULL, NULL) == pkv.EINVAL     # no k_scale
    assert kf(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 10, 16, 8, 60, FAKE, FAKE, NULL, NULL) == pkv.EINVAL      # D % 8
    assert kf(NULL, NULL, NULL, 0, NULL, NULL, 10, 16, 8, 128, NULL, NULL, NULL, NULL) == pkv.OK
    # pkv_paged_decode_fp8 shares pkv_paged_decode's checks and needs both scales
    fd = lib.pkv_paged_decode_fp8
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 2, 16, 8, 128, 16, 10, 64, 0.1, FAKE, FAKE, 1 << 30, 0,
            NULL, NULL]
    bad = list(args); bad[3] = NULL
    assert fd(*bad) == pkv.EINVAL
    bad = list(args); bad[11] = 96
    assert fd(*bad) == pkv.EUNSUPPORTED
    # pkv_copy_blocks(kc, vc, pairs, n, NB, bs, Hkv, D, err, stream)
    cb = lib.pkv_copy_blocks
    assert cb(FAKE, FAKE, NULL, 3, 10, 16, 8, 128, NULL, NULL) == pkv.EINVAL
    assert cb(FAKE, FAKE, FAKE, -1, 10, 16, 8, 128, NULL, NULL) == pkv.EINVAL
    assert cb(FAKE, FAKE, FAKE, 3, 10, 1, 1, 4, NULL, NULL) == pkv.EINVAL                              # 8-byte blocks
    assert cb(NULL, NULL, NULL, 0, 10, 16, 8, 128, NULL, NULL) == pkv.OK
    # pkv_paged_attention(q, kc, vc, bt, max_blocks, cu, lens, B, rows, Hq, Hkv, D, bs, NB, maxctx, scale, out,
    #                     ws, ws_bytes, workers, err, stream)
    pa = lib.pkv_paged_attention
    att = [FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 2, 5, 16, 8, 128, 16, 10, 64, 0.1, FAKE, 0, FAKE, 1 << 30, 0,
           NULL, NULL]
    bad = list(att); bad[5] = NULL
    assert pa(*bad) == pkv.EINVAL                                                                       # no offsets
    bad = list(att); bad[19] = 64
    assert pa(*bad) == pkv.EWORKSPACE
    bad = list(att); bad[17] = 3                                                                        # 2 * 3 != 5 rows
    assert pa(*bad) == pkv.EINVAL
    bad = list(att); bad[8] = pkv.MAX_SEQS + 1
    assert pa(*bad) == pkv.EBOUNDS
    bad = list(att); bad[8] = 0
    assert pa(*bad) == pkv.OK                                                                           # no rows


def test_attention_workspace_holds_the_rows(lib):
    """One decode entry per row with up to max(1, 8 // G) queries (qg * G virtual heads), then the
    three row arrays (sequence, length, query count)."""
    f, g = lib.pkv_paged_attention_workspace_size, lib.pkv_paged_decode_workspace_size
    for rows in (1, 7, 256, 4096):
        for hq, hkv, d in ((16, 8, 128), (6, 2, 64), (8, 8, 64), (14, 2, 64)):
            qg = max(1, 8 // (hq // hkv))
            assert f(rows, hq, hkv, d) >= g(rows, hq * qg, hkv, d) + 3 * 4 * rows
    assert f(-1, 16, 8, 128) == 0 and f(4, 16, 6, 128) == 0
