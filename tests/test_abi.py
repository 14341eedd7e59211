"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/pkv.h declares, and rejects bad arguments on the host before any
device work."""

import ctypes
import os
import re

import pytest

import paged_kv_cache_rmsnorm_gb300 as pkv
from paged_kv_cache_rmsnorm_gb300 import ops

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    pkv.build()
    return pkv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("pkv_qknorm_rope_store", "pkv_attn_prefill", "pkv_attn_decode"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"{n} missing from libpkv.so"
        assert n in ops.SIGNATURES, f"{n} has no ctypes signature in the binding"


def test_version_and_empty_error(lib):
    assert lib.pkv_version() >= 100
    assert isinstance(lib.pkv_last_error(), bytes)


FAKE = 0x10000  # a 16-byte-aligned address that is never dereferenced (host checks fail first)


def test_store_rejects_null_and_bad_shapes(lib):
    rc = lib.pkv_qknorm_rope_store(None, 4096, FAKE, 1024, FAKE, 1024, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, None)
    assert rc == -1 and b"NULL" in lib.pkv_last_error()
    rc = lib.pkv_qknorm_rope_store(FAKE, 4096, FAKE, 1024, FAKE, 1024, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, -1, 8, None)
    assert rc == -2
    rc = lib.pkv_qknorm_rope_store(FAKE, 4000, FAKE, 1024, FAKE, 1024, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, None)
    assert rc == -2
    rc = lib.pkv_qknorm_rope_store(FAKE, 4100, FAKE, 1024, FAKE, 1024, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, None)
    assert rc == -7
    rc = lib.pkv_qknorm_rope_store(FAKE + 2, 4096, FAKE, 1024, FAKE, 1024, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8,
                                   None)
    assert rc == -7
    rc = lib.pkv_qknorm_rope_store(FAKE, 4096, FAKE, 1024, FAKE, 1024, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 0, None)
    assert rc == -2
    # zero tokens is a no-op that needs no device
    rc = lib.pkv_qknorm_rope_store(FAKE, 4096, FAKE, 1024, FAKE, 1024, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 8, None)
    assert rc == 0


def test_empty_calls_read_no_pointer(lib):
    # nothing to do: PKV_OK before any pointer is looked at, so empty tensors may have NULL data
    N = None
    assert lib.pkv_qknorm_rope_store(N, 4096, N, 1024, N, 1024, N, N, N, N, N, N, 0, 0, None) == 0
    assert lib.pkv_attn_decode(N, N, N, N, N, 0, 0, 0, 0, 0.088, N, N, 0, None) == 0
    assert lib.pkv_attn_prefill(N, N, N, N, N, N, 0, 0, 0, 0, 0, 0, 0.088, N, None) == 0
    assert lib.pkv_attn_prefill(N, N, N, N, N, N, 3, 0, 0, 0, 0, 0, 0.088, N, None) == 0  # sequences, no queries
    assert lib.pkv_add_rmsnorm(N, N, N, N, 0, 4096, 1e-6, None) == 0
    assert lib.pkv_qkv_rope_store(N, N, N, N, N, N, N, N, N, 0, 0, None) == 0
    assert lib.pkv_attn_decode_noalloc(N, N, N, N, N, 0, 0, 0, 0, 0.088, N, N, None) == 0
    # negative sizes are still errors
    assert lib.pkv_qknorm_rope_store(N, 4096, N, 1024, N, 1024, N, N, N, N, N, N, -1, 0, None) == -2
    assert lib.pkv_attn_decode(N, N, N, N, N, -1, 0, 0, 0, 0.088, N, N, 0, None) == -2


def test_decode_rejects_bad_arguments(lib):
    args = dict(q=FAKE, kc=FAKE, vc=FAKE, cl=FAKE, bt=FAKE, B=4, mb=1, nb=8, mc=256, sc=0.088, out=FAKE, ws=None, wsb=0)

    def call(**kw):
        a = {**args, **kw}
        return lib.pkv_attn_decode(a["q"], a["kc"], a["vc"], a["cl"], a["bt"], a["B"], a["mb"], a["nb"], a["mc"],
                                   a["sc"], a["out"], a["ws"], a["wsb"], None)

    assert call(q=None) == -1
    assert call(B=-1) == -2
    assert call(B=70000) == -3
    assert call(mc=257) == -2  # more than one block of context with a 1-entry table
    assert call(sc=float("nan")) == -2
    assert call(out=FAKE + 8) == -7
    assert call(B=0) == 0
    # a split decode needs a workspace
    need = lib.pkv_attn_decode_workspace_size(1, 40960)
    assert need > 0
    assert call(B=1, mb=160, mc=40960) == -8
    assert call(B=1, mb=160, mc=40960, ws=FAKE, wsb=need - 1) == -8
    assert call(B=1, mb=160, mc=40960, ws=FAKE + 16, wsb=need) == -7


def test_decode_workspace_sizes(lib):
    assert lib.pkv_attn_decode_workspace_size(0, 100) == 0
    assert lib.pkv_attn_decode_workspace_size(4, 256) == 0  # short contexts are not split
    for B in (1, 8, 64):  # long contexts are split (one resident wave of CTAs, or four per SM at B = 64)
        size = lib.pkv_attn_decode_workspace_size(B, 40960)
        assert size > 0 and size % 256 == 0
    assert lib.pkv_attn_decode_workspace_size(32, 40960) == 0  # 256 (sequence, KV head) pairs already fill the GPU


def test_decode_workspace_never_exceeds_the_no_alloc_scratch(lib):
    # every batch up to 700 sequences (beyond it no context is split) at contexts up to 40960
    f = lib.pkv_attn_decode_workspace_size
    largest = max(f(B, mc) for B in range(1, 701) for mc in (512, 1024, 2048, 4096, 8192, 16384, 20000, 40960))
    assert largest <= int(4.4 * 2 ** 20) < 8 << 20
    assert all(f(B, 40960) == 0 for B in (1000, 4096, 65535))


def test_prefill_rejects_bad_arguments(lib):
    def call(S=2, mb=4, nb=8, tq=10, mq=8, mk=8, q=FAKE, out=FAKE, sc=0.088):
        return lib.pkv_attn_prefill(q, FAKE, FAKE, FAKE, FAKE, FAKE, S, mb, nb, tq, mq, mk, sc, out, None)

    assert call(q=None) == -1
    assert call(S=-1) == -2
    assert call(mq=9, mk=8) == -2
    assert call(mk=2000, mb=4) == -2
    assert call(nb=0) == -2
    assert call(out=FAKE + 4) == -7
    assert call(S=0) == 0
    assert call(tq=0) == 0


def test_add_rmsnorm_rejects_bad_arguments(lib):
    def call(x=FAKE, r=FAKE + 65536, w=FAKE + 131072, out=FAKE + 196608, T=4, hidden=4096, eps=1e-6):
        return lib.pkv_add_rmsnorm(x, r, w, out, T, hidden, eps, None)

    assert call(x=None) == -1
    assert call(w=None) == -1
    assert call(out=None) == -1
    assert call(T=-1) == -2
    assert call(hidden=4095) == -3
    assert call(hidden=2048) == -3
    assert call(eps=-1.0) == -2
    assert call(eps=float("nan")) == -2
    assert call(out=FAKE + 8) == -7
    assert call(r=FAKE + 4) == -7
    assert call(r=FAKE) == -2          # residual aliases x
    assert call(r=FAKE + 196608) == -2  # residual aliases out
    assert call(T=0) == 0
    assert call(T=0, r=None) == 0


def test_binding_refuses_cpu_tensors():
    import torch

    q = torch.zeros(2, 32, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkv.attn_decode(q, q, q, torch.zeros(2, dtype=torch.int32), torch.zeros(2, 1, dtype=torch.int32), 1, 0.1)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        ops.load_library(str(tmp_path / "libpkv.so"))


def test_noalloc_decode_host_checks_and_scratch_bound(lib):
    rc = lib.pkv_attn_decode_noalloc(None, FAKE, FAKE, FAKE, FAKE, 4, 1, 8, 256, 0.088, FAKE, None, None)
    assert rc == -1
    rc = lib.pkv_attn_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 1, 8, 257, 0.088, FAKE, None, None)
    assert rc == -2
    assert lib.pkv_attn_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1, 8, 256, 0.088, FAKE, None, None) == 0
    # every valid (batch, max_context) fits the 8 MiB static scratch
    worst = max(lib.pkv_attn_decode_workspace_size(b, c)
                for b in list(range(1, 130)) + [256, 1024, 65535]
                for c in (256, 1000, 4096, 9000, 20000, 32768, 40960))
    assert 0 < worst <= 8 << 20
