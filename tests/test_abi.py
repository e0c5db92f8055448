"""The C ABI without a GPU: the library builds and loads, exports every symbol
include/attn.h declares, and rejects bad arguments before any CUDA call."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    from exact_attention_43_gb300 import build, binding

    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_prefill_and_decode_entry_points():
    names = declared_functions()
    assert "attn_fwd" in names and "attn_decode" in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in attn.h but not exported"
    from exact_attention_43_gb300 import binding
    assert set(binding.EXPORTS) == set(declared_functions())


def test_version_and_status_strings(lib):
    assert lib.attn_version() >= 100
    for code, text in [(0, "ok"), (1, "invalid argument"), (4, "device wait timed out")]:
        assert lib.attn_status_string(code).decode() == text
    assert lib.attn_status_string(99).decode() == "unknown status"


FAKE = 0x10000  # never dereferenced: validation returns first


def fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=4, Hkv=4, Sq=8, Skv=8, D=64,
        causal=0, scale=0.125, dtype=0):
    return lib.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, causal, scale, dtype, None)


def test_fwd_argument_errors(lib):
    assert fwd(lib, q=None) == 1
    assert fwd(lib, o=None) == 1
    assert fwd(lib, k=None) == 1
    assert fwd(lib, Hkv=3) == 1            # Hq % Hkv != 0
    assert fwd(lib, Hkv=0) == 1
    assert fwd(lib, B=-1) == 1
    assert fwd(lib, Sq=-5) == 1
    assert fwd(lib, q=FAKE + 8) == 1       # misaligned
    assert fwd(lib, lse=FAKE + 2) == 1
    assert fwd(lib, scale=float("nan")) == 1
    assert fwd(lib, scale=float("inf")) == 1
    assert fwd(lib, D=96) == 2
    assert fwd(lib, D=256) == 2
    assert fwd(lib, dtype=7) == 2
    assert fwd(lib, B=70000) == 2


def test_fwd_empty_work_is_a_no_op(lib):
    assert fwd(lib, Sq=0) == 0
    assert fwd(lib, B=0) == 0
    assert fwd(lib, Hq=0, q=None, o=None) == 0


def dec(lib, q=FAKE, k=FAKE, v=FAKE, lens=FAKE, o=FAKE, B=2, Hq=8, Hkv=2, max_S=64, D=128,
        splits=0, dtype=0):
    return lib.attn_decode(q, k, v, lens, o, B, Hq, Hkv, max_S, D, splits, dtype, None)


def test_decode_argument_errors(lib):
    assert dec(lib, lens=None) == 1
    assert dec(lib, k=None) == 1
    assert dec(lib, Hkv=3) == 1
    assert dec(lib, splits=-1) == 1
    assert dec(lib, max_S=-1) == 1
    assert dec(lib, o=FAKE + 4) == 1
    assert dec(lib, lens=FAKE + 2) == 1
    assert dec(lib, D=32) == 2
    assert dec(lib, dtype=2) == 2
    assert dec(lib, B=0) == 0


def test_varlen_and_packed_argument_errors(lib):
    def vl(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, cq=FAKE, ck=FAKE, B=2, Hq=8, Hkv=2,
                 tq=100, tk=100, mq=64, mk=64, D=128, causal=1, wl=-1, wr=-1, scale=0.1, dtype=0)
        a.update(kw)
        return lib.attn_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cq"], a["ck"], a["B"],
                                   a["Hq"], a["Hkv"], a["tq"], a["tk"], a["mq"], a["mk"], a["D"],
                                   a["causal"], a["wl"], a["wr"], a["scale"], a["dtype"], None)

    assert vl(cq=None) == 1
    assert vl(k=None) == 1
    assert vl(k=None, v=None, tk=0, wl=-2) == 1        # a window bound below -1
    assert vl(Hkv=3) == 1
    assert vl(lse=FAKE + 2) == 1
    assert vl(scale=float("inf")) == 1
    assert vl(D=96) == 2
    assert vl(mq=1 << 29, mk=1 << 29) == 2              # key indices would leave an int
    assert vl(B=0) == 0 and vl(tq=0) == 0 and vl(mq=0) == 0

    def pk(**kw):
        a = dict(qkv=FAKE, o=FAKE, lse=FAKE, B=2, S=100, H=4, D=64, causal=1, wl=-1, wr=-1,
                 scale=0.1, dtype=1)
        a.update(kw)
        return lib.attn_fwd_qkvpacked(a["qkv"], a["o"], a["lse"], a["B"], a["S"], a["H"], a["D"],
                                      a["causal"], a["wl"], a["wr"], a["scale"], a["dtype"], None)

    assert pk(qkv=None) == 1
    assert pk(o=FAKE + 8) == 1
    assert pk(wr=-3) == 1
    assert pk(dtype=5) == 2
    assert pk(S=0) == 0


def test_backward_argument_errors(lib):
    def bw(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, do=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=2,
                 Hq=8, Hkv=2, Sq=64, Skv=64, D=128, causal=1, scale=0.1, dtype=0)
        a.update(kw)
        return lib.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"],
                            a["dv"], a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Skv"], a["D"],
                            a["causal"], a["scale"], a["dtype"], None)

    assert bw(lse=None) == 1
    assert bw(dk=None) == 1
    assert bw(dq=FAKE + 8) == 1
    assert bw(Hkv=3) == 1
    assert bw(scale=float("nan")) == 1
    assert bw(D=32) == 2 and bw(dtype=7) == 2
    assert bw(B=0) == 0 and bw(Sq=0, Skv=0) == 0
    # fp32 row terms, plus alignment slack
    assert lib.attn_bwd_workspace_bytes(2, 8, 64, 128) == 2 * 8 * 64 * 4 + 256
    assert lib.attn_bwd_workspace_bytes(-1, 8, 64, 128) == 0


def test_backward_token_major_argument_errors(lib):
    def vb(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, do=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
                 cq=FAKE, ck=FAKE, B=2, Hq=8, Hkv=2, tq=100, tk=120, mq=60, mk=70, D=128, causal=1,
                 wl=-1, wr=-1, scale=0.1, dtype=0)
        a.update(kw)
        return lib.attn_bwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"],
                                   a["dk"], a["dv"], a["cq"], a["ck"], a["B"], a["Hq"], a["Hkv"],
                                   a["tq"], a["tk"], a["mq"], a["mk"], a["D"], a["causal"], a["wl"],
                                   a["wr"], a["scale"], a["dtype"], None)

    assert vb(cq=None) == 1 and vb(ck=None) == 1
    assert vb(lse=None) == 1 and vb(dv=None) == 1
    assert vb(dk=FAKE + 8) == 1 and vb(cq=FAKE + 2) == 1
    assert vb(Hkv=3) == 1 and vb(wl=-2) == 1 and vb(tq=-1) == 1
    assert vb(scale=float("inf")) == 1
    assert vb(D=96) == 2 and vb(dtype=4) == 2
    assert vb(B=0) == 0 and vb(tq=0, tk=0) == 0

    def pk(**kw):
        a = dict(qkv=FAKE, o=FAKE, lse=FAKE, do=FAKE, dqkv=FAKE, B=2, S=64, H=4, D=64, causal=1,
                 wl=-1, wr=-1, scale=0.1, dtype=1)
        a.update(kw)
        return lib.attn_bwd_qkvpacked(a["qkv"], a["o"], a["lse"], a["do"], a["dqkv"], a["B"],
                                      a["S"], a["H"], a["D"], a["causal"], a["wl"], a["wr"],
                                      a["scale"], a["dtype"], None)

    assert pk(dqkv=None) == 1 and pk(lse=None) == 1
    assert pk(do=FAKE + 8) == 1 and pk(wr=-5) == 1
    assert pk(D=80) == 2
    assert pk(S=0) == 0


def test_fused_decode_argument_errors(lib):
    def fused(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, lens=FAKE, o=FAKE, B=2, Hq=8, Hkv=2, max_S=64, D=128,
                 splits=0, dtype=0)
        a.update(kw)
        return lib.attn_decode_fused(a["q"], a["k"], a["v"], a["lens"], a["o"], a["B"], a["Hq"],
                                     a["Hkv"], a["max_S"], a["D"], a["splits"], a["dtype"], None)

    assert fused(lens=None) == 1
    assert fused(Hkv=3) == 1
    assert fused(o=FAKE + 4) == 1
    assert fused(D=32) == 2
    assert fused(B=0) == 0
    # more (sequence, query head) pairs than merge counters: refused before any CUDA call
    assert fused(B=32769, Hq=32, Hkv=8) == 2


def paged(lib, q=FAKE, kp=FAKE, vp=FAKE, bt=FAKE, lens=FAKE, o=FAKE, B=2, Hq=8, Hkv=2, num_pages=4,
          page_size=16, max_pages=4, D=128, splits=0, dtype=0):
    return lib.attn_decode_paged(q, kp, vp, bt, lens, o, B, Hq, Hkv, num_pages, page_size, max_pages,
                                 D, splits, dtype, None)


def test_paged_decode_argument_errors(lib):
    assert paged(lib, bt=None) == 1             # pages but no block table
    assert paged(lib, num_pages=0) == 1         # block table into an empty pool
    assert paged(lib, page_size=0) == 1
    assert paged(lib, max_pages=-1) == 1
    assert paged(lib, bt=FAKE + 2) == 1         # int32 table not 4-byte aligned
    assert paged(lib, kp=FAKE + 8) == 1         # pages not 16-byte aligned
    assert paged(lib, Hkv=3) == 1
    assert paged(lib, D=96) == 2
    assert paged(lib, page_size=1 << 16, max_pages=1 << 16) == 2  # positions overflow an int
    assert paged(lib, B=0) == 0


def test_noalloc_decode_refuses_oversized_partials_before_any_cuda_call(lib):
    # 64 x 32 x 64 chunks x 130 floats x 4 B = 68 MB > 16 MiB of fixed scratch
    assert lib.attn_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 64, 32, 8, 32768, 128, 64, 0,
                                   None) == 2
    assert lib.attn_decode_noalloc(FAKE, FAKE, FAKE, None, FAKE, 2, 8, 2, 64, 128, 0, 0, None) == 1
    assert lib.attn_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 8, 2, 64, 128, 0, 0, None) == 0


def test_decode_chunking_and_workspace(lib):
    assert lib.attn_decode_chunk(32768, 64) == 512
    assert lib.attn_decode_chunk(32768, 0) == 512
    assert lib.attn_decode_chunk(1000, 3) == 334
    assert lib.attn_decode_chunk(5, 64) == 1
    assert lib.attn_decode_chunk(-1, 2) == 0
    want = 64 * 32 * 64 * (128 + 2) * 4
    assert lib.attn_decode_workspace_bytes(64, 32, 32768, 128, 64) == want
    assert lib.attn_decode_workspace_bytes(2, 4, 0, 128, 8) == 0
    assert lib.attn_decode_workspace_bytes(-2, 4, 10, 128, 8) == 0


def test_debug_hook_validation(lib):
    # faults 1-3 withhold a copy in the prefill, decode and backward kernels
    for bad in (-1, 4, 5):
        assert lib.attn_debug_set(bad, 0) == 1
    for good in (1, 2, 3, 0):
        assert lib.attn_debug_set(good, 0) == 0


def test_binding_fails_loudly_without_the_library(tmp_path):
    from exact_attention_43_gb300 import binding
    with pytest.raises(binding.ExtensionMissing):
        binding._lib, saved = None, binding._lib
        try:
            binding.load(str(tmp_path / "missing.so"))
        finally:
            binding._lib = saved
