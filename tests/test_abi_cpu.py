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
    assert lib.pkv_abi_version() == 1
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
    (dict(Hq=72, Hkv=8), pkv.EUNSUPPORTED),    # group of 9
    (dict(bs=12), pkv.EUNSUPPORTED),
    (dict(bs=4), pkv.EUNSUPPORTED),
    (dict(bs=2048), pkv.EUNSUPPORTED),
    (dict(B=-1), pkv.EINVAL),
    (dict(B=pkv.MAX_SEQS + 1), pkv.EUNSUPPORTED),
    (dict(maxctx=-1), pkv.EINVAL),
    (dict(workers=-1), pkv.EINVAL),
    (dict(workers=pkv.MAX_WORKERS + 1), pkv.EINVAL),
    (dict(scale=float("nan")), pkv.EINVAL),
    (dict(q=FAKE + 8), pkv.EINVAL),            # misaligned
    (dict(ws=NULL), pkv.EWORKSPACE),
    (dict(wsb=16), pkv.EWORKSPACE),
    (dict(NB=1 << 27, bs=256), pkv.EUNSUPPORTED),  # rows beyond int32
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


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        pkv.load(str(tmp_path / "libpkv.so"))
