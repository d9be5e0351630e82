"""The C ABI on the host, no GPU: the library builds, loads, exports every declared entry
point, and rejects bad arguments with the documented status before touching the device."""
import ctypes
import os
import re
import shutil

import pytest

import paged_kv_attention_store_gb300 as nv
from paged_kv_attention_store_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NV_ERR_NULL, NV_ERR_SHAPE, NV_ERR_ALIGN, NV_ERR_UNSUPPORTED, NV_ERR_WORKSPACE, NV_ERR_CUDA = -1, -2, -3, -4, -5, -6
FAKE = 0x10000          # a 16-byte-aligned address that is never dereferenced (validation fails first)
MISALIGNED = 0x10008


def declared_entry_points():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(nv_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("no CUDA toolkit to build the library")
    B.build()
    return nv.load_library()


def test_exports_every_declared_symbol(lib):
    names = declared_entry_points()
    assert {"nv_store_kvcache", "nv_paged_decode_attn", "nv_paged_prefill_attn"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(nv.EXPORTED) <= set(names)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.nv_status_string(code)
    assert b"unknown" in lib.nv_status_string(42)


def _store(lib, k=FAKE, v=FAKE, sm=FAKE, n=4, kc=FAKE, vc=FAKE, ks=1024, vs=1024, hkv=8, d=128, slots=1024):
    return lib.nv_store_kvcache(k, ks, v, vs, sm, n, kc, vc, slots, hkv, d, None, None)


def test_store_validation(lib):
    assert _store(lib, n=0, k=None) == 0                  # nothing to do, nothing read
    assert _store(lib, n=-1) == NV_ERR_SHAPE
    assert _store(lib, k=None) == NV_ERR_NULL
    assert _store(lib, sm=None) == NV_ERR_NULL
    assert _store(lib, ks=512) == NV_ERR_SHAPE            # row stride below Hkv*D
    assert _store(lib, vs=1028) == NV_ERR_ALIGN           # not a multiple of 8 elements
    assert _store(lib, k=MISALIGNED) == NV_ERR_ALIGN
    assert _store(lib, kc=MISALIGNED) == NV_ERR_ALIGN
    assert _store(lib, hkv=1, d=4, ks=8, vs=8) == NV_ERR_UNSUPPORTED   # row of 4 values


def _decode(lib, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, bts=16, cl=FAKE, B=4, hq=32, hkv=8, d=128, bs=256, nb=64,
            maxc=4096, out=FAKE, ws=None, wsb=0):
    return lib.nv_paged_decode_attn(q, kc, vc, bt, bts, cl, B, hq, hkv, d, bs, nb, maxc, 0.088, out, ws, wsb,
                                    None, None)


def test_decode_validation(lib):
    assert _decode(lib, B=0, q=None) == 0
    assert _decode(lib, q=None) == NV_ERR_NULL
    assert _decode(lib, cl=None) == NV_ERR_NULL
    assert _decode(lib, d=64) == NV_ERR_UNSUPPORTED
    assert _decode(lib, hq=12) == NV_ERR_SHAPE            # not a multiple of Hkv
    assert _decode(lib, hq=24, hkv=8) == NV_ERR_UNSUPPORTED   # group 3
    assert _decode(lib, bs=8) == NV_ERR_UNSUPPORTED
    assert _decode(lib, bs=48) == NV_ERR_UNSUPPORTED
    assert _decode(lib, out=MISALIGNED) == NV_ERR_ALIGN
    need = lib.nv_paged_decode_workspace_size(4, 32, 128, 4096)
    assert need > 0
    assert _decode(lib) == NV_ERR_WORKSPACE
    assert _decode(lib, ws=FAKE, wsb=need - 16) == NV_ERR_WORKSPACE
    # one split: no partials, but room for the tile kernel's work list (groups of 8 and 16) after the
    # 256 KiB of counters (64 bytes + 32 per sequence)
    assert lib.nv_paged_decode_workspace_size(4, 32, 128, 64) == 256 * 1024 + 64 + 32 * 4
    assert _decode(lib, hq=128, hkv=8) == NV_ERR_WORKSPACE     # group 16: the tile kernel, needs the list
    assert _decode(lib, hq=128, hkv=8, maxc=64, ws=FAKE, wsb=256 * 1024 + 64) == NV_ERR_WORKSPACE
    assert _decode(lib, hq=256, hkv=8) == NV_ERR_UNSUPPORTED   # group 32


def test_decode_workspace_size_follows_the_split_rule(lib):
    """256 KiB of split counters, then num_seqs x splits x Hq x (128 + 2) floats of partials, then a
    tile-kernel work list of 64 bytes + 32 per (sequence, split); the split is 512 positions halved
    while the batch has fewer than 1200 units, stopping at 256 once it has 600 (and at 64 at the
    least)."""
    def size(B, L, hq=32):
        return lib.nv_paged_decode_workspace_size(B, hq, 128, L)
    part = lambda B, splits, hq=32: 256 * 1024 + B * splits * hq * 130 * 4 + 64 + 32 * B * splits
    assert size(512, 4096) == part(512, 8)        # 4096 units at 512 positions
    assert size(256, 2048, 16) == part(256, 8, 16)  # 1024 units at 512 -> 2048 at 256
    assert size(64, 4096) == part(64, 16)         # 512 -> 1024 units at 256: stop (>= 600)
    assert size(4, 4096) == part(4, 64)           # a tiny batch goes down to 64 positions


def _fused(lib, q=FAKE, k=FAKE, ks=1024, v=FAKE, vs=1024, sm=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, bts=16, cl=FAKE, B=4,
           hq=32, hkv=8, d=128, bs=256, nb=64, maxc=256, out=FAKE):
    return lib.nv_store_decode_attn(q, k, ks, v, vs, sm, kc, vc, bt, bts, cl, B, hq, hkv, d, bs, nb, maxc, 0.088, out,
                                    None, 0, None, None)


def test_fused_store_decode_validation(lib):
    assert _fused(lib, B=0, q=None) == 0
    assert _fused(lib, hq=128, hkv=8) == NV_ERR_WORKSPACE      # group 16: store + tile kernel, needs the list
    assert _fused(lib, hq=256, hkv=8) == NV_ERR_UNSUPPORTED    # group 32
    assert _fused(lib, k=None) == NV_ERR_NULL
    assert _fused(lib, sm=None) == NV_ERR_NULL
    assert _fused(lib, q=None) == NV_ERR_NULL
    assert _fused(lib, ks=512) == NV_ERR_SHAPE              # row stride below Hkv*D
    assert _fused(lib, vs=1028) == NV_ERR_ALIGN             # not a multiple of 8 elements
    assert _fused(lib, v=MISALIGNED) == NV_ERR_ALIGN
    assert _fused(lib, d=64) == NV_ERR_UNSUPPORTED
    assert _fused(lib, maxc=4096) == NV_ERR_WORKSPACE       # several splits need a workspace


def _prologue(lib, qkv=FAKE, rs=4096, pos=FAKE, qw=FAKE, kw=FAKE, sm=FAKE, n=4, hq=16, hkv=8, d=128, qo=FAKE,
              kc=FAKE, vc=FAKE, slots=64, eps=1e-6, theta=1e6):
    return lib.nv_qk_norm_rope_store(qkv, rs, pos, qw, kw, eps, theta, sm, n, hq, hkv, d, qo, kc, vc, slots, None, None)


def test_prologue_validation(lib):
    assert _prologue(lib, n=0, qkv=None) == 0
    assert _prologue(lib, qkv=None) == NV_ERR_NULL
    assert _prologue(lib, kw=None) == NV_ERR_NULL
    assert _prologue(lib, d=64, rs=2048) == NV_ERR_UNSUPPORTED
    assert _prologue(lib, rs=4088) == NV_ERR_SHAPE           # row shorter than q | k | v
    assert _prologue(lib, rs=4100) == NV_ERR_ALIGN           # not a multiple of 8 elements
    assert _prologue(lib, qo=MISALIGNED) == NV_ERR_ALIGN
    assert _prologue(lib, theta=1.0) == NV_ERR_SHAPE
    assert _prologue(lib, eps=-1.0) == NV_ERR_SHAPE


def test_prepare_validation(lib):
    assert lib.nv_prepare_decode(FAKE, FAKE, 4, 0, 0, 256, 8, FAKE, FAKE, FAKE, None, None) == 0
    assert lib.nv_prepare_decode(FAKE, FAKE, 4, 3, 2, 256, 8, FAKE, FAKE, FAKE, None, None) == NV_ERR_SHAPE  # pad < n
    assert lib.nv_prepare_decode(None, FAKE, 4, 3, 3, 256, 8, FAKE, FAKE, FAKE, None, None) == NV_ERR_NULL
    assert lib.nv_prepare_decode(FAKE, FAKE, 4, 3, 3, 48, 8, FAKE, FAKE, FAKE, None, None) == NV_ERR_UNSUPPORTED
    assert lib.nv_prepare_prefill(FAKE, FAKE, FAKE, 4, 0, 0, 256, 8, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == 0
    assert lib.nv_prepare_prefill(FAKE, None, FAKE, 4, 2, 5, 256, 8, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == NV_ERR_NULL
    assert lib.nv_prepare_prefill(FAKE, FAKE, FAKE, 4, 2, 5, 100, 8, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                  None) == NV_ERR_UNSUPPORTED


def test_sampler_validation(lib):
    assert lib.nv_sample_workspace_size(512, 151936) > 0
    args = dict(lg=FAKE, ls=1024, t=FAKE, e=FAKE, es=1024, B=4, V=1000, tok=FAKE, ws=FAKE, wsb=1 << 20)

    def call(**kw):
        a = {**args, **kw}
        return lib.nv_sample_exponential_race(a["lg"], a["ls"], a["t"], a["e"], a["es"], a["B"], a["V"], a["tok"],
                                              a["ws"], a["wsb"], None, None)
    assert call(B=0, lg=None) == 0
    assert call(lg=None) == NV_ERR_NULL
    assert call(ls=999) == NV_ERR_SHAPE                    # stride shorter than the vocabulary
    assert call(ls=1004) == NV_ERR_ALIGN                   # not a multiple of 8 entries
    assert call(e=MISALIGNED) == NV_ERR_ALIGN
    assert call(ws=None) == NV_ERR_WORKSPACE


def _prefill(lib, q=FAKE, kc=FAKE, vc=FAKE, cq=FAKE, ck=FAKE, bt=FAKE, bts=8, B=2, tq=100, mq=80, hq=16, hkv=8,
             d=128, bs=256, nb=16, out=FAKE, ws=FAKE, wsb=256):
    return lib.nv_paged_prefill_attn(q, kc, vc, cq, ck, bt, bts, B, tq, mq, hq, hkv, d, bs, nb, 0.088, out, ws, wsb,
                                     None, None)


def test_prefill_validation(lib):
    assert _prefill(lib, tq=0, q=None) == 0
    assert _prefill(lib, cq=None) == NV_ERR_NULL
    assert _prefill(lib, d=256) == NV_ERR_UNSUPPORTED
    assert _prefill(lib, hq=24) == NV_ERR_UNSUPPORTED      # group 3
    assert _prefill(lib, hq=20) == NV_ERR_SHAPE
    assert _prefill(lib, bs=512) == NV_ERR_UNSUPPORTED
    assert _prefill(lib, kc=MISALIGNED) == NV_ERR_ALIGN
    assert _prefill(lib, nb=0) == NV_ERR_SHAPE
    assert _prefill(lib, ws=None) == NV_ERR_WORKSPACE
    need = lib.nv_paged_prefill_workspace_size(2, 100, 80, 16, 8)
    assert need == 64 + 32 * 4                               # min(ceil(100/64) + 2, 2 * ceil(80/64)) tiles
    assert _prefill(lib, wsb=need - 16) == NV_ERR_WORKSPACE
    assert _prefill(lib, ws=MISALIGNED) == NV_ERR_WORKSPACE


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="checks the no-GPU path only")
def test_valid_call_without_gpu_reports_cuda_error(lib):
    """With no GPU the runtime cannot launch: the entry point says so instead of crashing."""
    assert _store(lib) == NV_ERR_CUDA


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        nv.load_library(str(tmp_path / "missing.so"))


def test_header_shape_limits(lib):
    """Every shape limit the header's conventions state, at both sides of each bound.  An accepted
    shape gets as far as the workspace check (none is passed), which comes before any device work."""
    # decode: groups 1, 2, 4 (split-KV kernel) and 8, 16 (tile kernel) accepted; 32 and 3 refused
    for hq, hkv in ((8, 8), (16, 8), (32, 8), (64, 8), (128, 8), (32, 16), (256, 16)):
        assert _decode(lib, hq=hq, hkv=hkv) == NV_ERR_WORKSPACE, (hq, hkv)
    for hq, hkv in ((256, 8), (24, 8), (12, 4)):
        assert _decode(lib, hq=hq, hkv=hkv) == NV_ERR_UNSUPPORTED, (hq, hkv)
    assert _decode(lib, hq=32, hkv=32) == NV_ERR_UNSUPPORTED      # num_kv_heads above 16
    assert _decode(lib, hq=20, hkv=8) == NV_ERR_SHAPE             # not a multiple
    for bs in (16, 32, 64, 128, 256):
        assert _decode(lib, bs=bs) == NV_ERR_WORKSPACE, bs
    for bs in (8, 24, 512):
        assert _decode(lib, bs=bs) == NV_ERR_UNSUPPORTED, bs
    assert _decode(lib, d=256) == NV_ERR_UNSUPPORTED
    # decode on the tile kernel (G = 8, 16): num_seqs <= 65535, num_blocks * block_size < 2^31
    assert _decode(lib, hq=64, hkv=8, B=65535) == NV_ERR_WORKSPACE
    assert _decode(lib, hq=64, hkv=8, B=65536) == NV_ERR_UNSUPPORTED
    assert _decode(lib, hq=8, hkv=1, nb=(1 << 23) - 1) == NV_ERR_WORKSPACE
    assert _decode(lib, hq=8, hkv=1, nb=1 << 23) == NV_ERR_UNSUPPORTED
    # decode: a pool of fewer than 2^40 values per tensor (2^30 slots of 8 x 128 values)
    assert _decode(lib, bs=256, nb=(1 << 22) - 1) == NV_ERR_WORKSPACE
    assert _decode(lib, bs=256, nb=1 << 22) == NV_ERR_UNSUPPORTED
    # prefill: the same groups, block sizes and head_dim; num_seqs <= 65535
    for hq, hkv in ((8, 8), (16, 8), (32, 8), (64, 8), (128, 8)):
        assert _prefill(lib, hq=hq, hkv=hkv, ws=None) == NV_ERR_WORKSPACE, (hq, hkv)
    assert _prefill(lib, hq=256, hkv=8) == NV_ERR_UNSUPPORTED
    assert _prefill(lib, hq=24, hkv=8) == NV_ERR_UNSUPPORTED
    for bs in (16, 256):
        assert _prefill(lib, bs=bs, ws=None) == NV_ERR_WORKSPACE, bs
    for bs in (8, 512):
        assert _prefill(lib, bs=bs) == NV_ERR_UNSUPPORTED, bs
    assert _prefill(lib, B=65535, ws=None) == NV_ERR_WORKSPACE
    assert _prefill(lib, B=65536) == NV_ERR_UNSUPPORTED
    assert _prefill(lib, nb=(1 << 23) - 1, ws=None) == NV_ERR_WORKSPACE
    assert _prefill(lib, nb=1 << 23) == NV_ERR_UNSUPPORTED
