"""The C ABI without a GPU: the library loads, exports every function that
include/pkv.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest
import torch

import paged_kv_attention_22_gb300 as pkv
from paged_kv_attention_22_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def L():
    pkv_build.build()
    return pkv.lib()


def _declared_functions():
    names = set()
    for path in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names.update(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for must in ("pkv_kv_store", "pkv_paged_decode_attn", "pkv_paged_prefill_attn",
                 "pkv_decode_workspace_size", "pkv_prefill_workspace_size",
                 "pkv_check_device_errors", "pkv_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), f"libpkv.so does not export {name}"


def test_error_bits_match_header():
    text = open(HEADER).read()
    for name, val in [("SLOT", pkv.DEVERR_SLOT), ("BLOCK", pkv.DEVERR_BLOCK),
                      ("CONTEXT", pkv.DEVERR_CONTEXT), ("SEQLENS", pkv.DEVERR_SEQLENS),
                      ("TIMEOUT", pkv.DEVERR_TIMEOUT)]:
        m = re.search(r"#define PKV_DEVERR_%s (0x[0-9a-fA-F]+)u" % name, text)
        assert m and int(m.group(1), 16) == val


def test_status_strings(L):
    assert pkv.status_string(0) == "PKV_OK"
    assert pkv.status_string(3) == "PKV_ERR_WORKSPACE_TOO_SMALL"
    assert pkv.status_string(5) == "PKV_ERR_OUT_OF_BLOCKS"
    assert pkv.status_string(99) == "PKV_ERR_UNKNOWN"


FAKE = ctypes.c_void_p(0x10000)  # a non-null, 16-byte aligned value never dereferenced


def _decode(L, **kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mb=4, cl=FAKE, mcl=64, S=2, Hq=16, Hkv=8, D=128,
             bs=16, NB=64, scale=0.088, win=0, out=FAKE, lse=None, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    return L.pkv_paged_decode_attn(a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["cl"], a["mcl"],
                                   a["S"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"],
                                   a["scale"], a["win"], a["out"], a["lse"], a["ws"], a["wsb"],
                                   None)


def test_decode_argument_checks(L):
    assert _decode(L, q=None) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(L, S=0) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(L, mcl=0) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(L, D=64) == pkv.PKV_ERR_UNSUPPORTED
    assert _decode(L, Hq=12, Hkv=8) == pkv.PKV_ERR_UNSUPPORTED
    assert _decode(L, Hq=64, Hkv=8) == pkv.PKV_ERR_UNSUPPORTED
    assert _decode(L, bs=24) == pkv.PKV_ERR_UNSUPPORTED
    assert _decode(L, scale=float("nan")) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(L, win=-1) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(L, ws=None) == pkv.PKV_ERR_WORKSPACE_TOO_SMALL
    assert _decode(L, S=2048) == pkv.PKV_ERR_UNSUPPORTED
    assert _decode(L, out=ctypes.c_void_p(0x10008)) == pkv.PKV_ERR_INVALID_ARG


def test_decode_workspace_size(L):
    assert L.pkv_decode_workspace_size(0, 16, 8, 128, 640) == 0
    assert L.pkv_decode_workspace_size(64, 12, 8, 128, 640) == 0
    a = L.pkv_decode_workspace_size(64, 16, 8, 128, 640)
    if torch.cuda.is_available():
        # two partial-result slots per persistent CTA: the size follows the SM
        # count and the head counts, neither the sequence count nor the context
        assert a > 0
        assert a == L.pkv_decode_workspace_size(128, 16, 8, 128, 640)
        assert a == L.pkv_decode_workspace_size(1, 16, 8, 128, 640)
        assert a == L.pkv_decode_workspace_size(64, 16, 8, 128, 8193)
        assert a < L.pkv_decode_workspace_size(64, 32, 8, 128, 640)  # G = 4 query heads per KV head
    else:
        assert a == 0  # the size depends on the device's SM count


def test_prefill_argument_checks(L):
    def call(**kw):
        a = dict(q=FAKE, kc=FAKE, vc=FAKE, cq=FAKE, ck=FAKE, bt=FAKE, mb=4, S=2, T=100, mq=64,
                 mk=64, Hq=16, Hkv=8, D=128, bs=16, NB=64, scale=0.088, win=0, out=FAKE)
        a.update(kw)
        return L.pkv_paged_prefill_attn(a["q"], a["kc"], a["vc"], a["cq"], a["ck"], a["bt"],
                                        a["mb"], a["S"], a["T"], a["mq"], a["mk"], a["Hq"],
                                        a["Hkv"], a["D"], a["bs"], a["NB"], a["scale"], a["win"],
                                        a["out"], None, None, 0, None)
    assert call(cq=None) == pkv.PKV_ERR_INVALID_ARG
    assert call(mq=65, mk=64) == pkv.PKV_ERR_INVALID_ARG
    assert call(D=256) == pkv.PKV_ERR_UNSUPPORTED
    assert call(win=-5) == pkv.PKV_ERR_INVALID_ARG
    assert call(NB=1 << 28, bs=16) == pkv.PKV_ERR_UNSUPPORTED
    # nothing to do: returns OK without touching the device
    assert call(T=0, q=None, out=None) == pkv.PKV_OK
    assert call(S=0) == pkv.PKV_OK


def test_kv_store_argument_checks(L):
    def call(**kw):
        a = dict(k=FAKE, v=FAKE, kc=FAKE, vc=FAKE, sm=FAKE, T=4, H=8, D=128, bs=16, NB=64)
        a.update(kw)
        return L.pkv_kv_store(a["k"], a["v"], a["kc"], a["vc"], a["sm"], a["T"], a["H"], a["D"],
                              a["bs"], a["NB"], None)
    assert call(k=None) == pkv.PKV_ERR_INVALID_ARG
    assert call(T=-1) == pkv.PKV_ERR_INVALID_ARG
    assert call(H=1, D=4) == pkv.PKV_ERR_UNSUPPORTED  # 8-byte rows
    assert call(T=0, k=None, v=None, sm=None) == pkv.PKV_OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
def test_valid_call_without_gpu_reports_cuda_error(L):
    assert _decode(L) == pkv.PKV_ERR_CUDA
    assert L.pkv_last_cuda_error() != b""
    flags = ctypes.c_uint32(7)
    assert L.pkv_check_device_errors(None, ctypes.byref(flags)) == pkv.PKV_ERR_CUDA
