"""The C ABI without a GPU: the library builds, loads and exports every symbol
include/fa.h declares, and host-side validation rejects bad arguments before
anything is launched."""
import ctypes
import os
import re

import pytest

from flash_attention_gqa_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def clib():
    if not os.path.exists(binding.LIB_PATH):
        from flash_attention_gqa_gb300 import build
        build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)


def test_every_declared_symbol_is_exported(clib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(clib, n), n
        assert n in binding.SIGNATURES, f"binding lacks {n}"


def test_status_strings(clib):
    for code in range(5):
        assert binding.status_string(code)
    assert binding.status_string(99) == "unknown status"


def _split_part(B, K, S, H, sms):
    """Bytes of the Q-range split part: counters and 4 fp32 partial dK/dV tiles
    per dK/dV CTA, for the KV tile sizes (64, and 128 at H <= 128) whose grid is
    smaller than the GPU; the largest over them.  H = 64 runs the H = 128
    kernels, so its partial tiles have 128 head dims."""
    up = lambda x: (x + 255) // 256 * 256
    cnt = part = 0
    for rows in ((64, 128) if H <= 128 else (64,)):
        ctas = B * K * -(-S // rows)
        if 0 < ctas < sms:
            cnt = max(cnt, up(ctas * 4))
            part = max(part, 4 * ctas * 2 * rows * max(H, 128) * 4)
    return cnt + up(part) if part else 0


def test_workspace_size(clib):
    sms = binding.load().fa_device_sm_count()   # 0 without a GPU: no split part
    # fp32 D rows, then one (min, max) int32 pair per (b, q tile) and (b, kv tile),
    # then one segment-run byte per (b, kv tile), each part rounded up to 256 B
    n = binding.fa_bwd_workspace_size(1, 2, 8, 8192, 8192, 256)
    assert n == 2 * 8 * 8192 * 4 + (8192 // 16 + 8192 // 64) * 8 + 256 + \
        _split_part(1, 2, 8192, 256, sms)
    assert n % 256 == 0
    assert binding.fa_bwd_workspace_size(1, 1, 1, 128, 128, 128) == 512 + 256 + 256 + \
        _split_part(1, 1, 128, 128, sms)
    assert binding.fa_bwd_workspace_size(0, 1, 1, 128, 128, 128) == 0
    # ragged sizes: D rows rounded up to 256 B, then one range pair per tile
    assert binding.fa_bwd_workspace_size(1, 1, 1, 100, 130, 128) == 512 + 256 + 256 + \
        _split_part(1, 1, 130, 128, sms)
    assert binding.fa_bwd_workspace_size(1, 1, 1, 100, 128, 96) == 0      # H unsupported
    # H = 64: D rows and range table as for any H, the split part at 128 head dims
    assert binding.fa_bwd_workspace_size(2, 2, 4, 1024, 1024, 64) == 2 * 2 * 4 * 1024 * 4 + \
        256 * ((2 * (1024 // 32 + 1024 // 64) * 8 + 255) // 256) + 256 + _split_part(2, 2, 1024, 64, sms)


def test_split_part_layout():
    # a 152-SM GPU: the T=1024 shape (B2 K2) splits at both KV tile sizes,
    # the largest part being 4 x 64 CTAs x 2 x 64 x 128 fp32
    assert _split_part(2, 2, 1024, 128, 152) == 256 + 4 * 64 * 2 * 64 * 128 * 4
    assert _split_part(1, 2, 8192, 256, 152) == 0     # 256 CTAs fill the GPU
    assert _split_part(1, 1, 128, 128, 0) == 0


def _fwd(clib, *, q=16, k=16, v=16, sq=None, skv=None, causal=0, o=16, lse=16,
         B=1, K=1, G=4, T=128, S=128, H=128):
    P = ctypes.c_void_p
    return clib.fa_fwd(P(q), P(k), P(v), P(sq), P(skv), causal, P(o), P(lse),
                       B, K, G, T, S, H, None)


def test_fwd_validation(clib):
    # every call below is rejected (or has nothing to do) before any launch:
    # the pointers are fake
    assert _fwd(clib, q=0) == binding.FA_ERR_INVALID_ARG
    assert _fwd(clib, q=8) == binding.FA_ERR_INVALID_ARG            # misaligned
    assert _fwd(clib, sq=16) == binding.FA_ERR_INVALID_ARG           # one seg pointer
    assert _fwd(clib, B=-1) == binding.FA_ERR_INVALID_ARG
    assert _fwd(clib, H=96) == binding.FA_ERR_UNSUPPORTED
    assert _fwd(clib, G=3) == binding.FA_ERR_UNSUPPORTED
    assert _fwd(clib, G=256) == binding.FA_ERR_UNSUPPORTED
    assert _fwd(clib, S=256 * 1024) == binding.FA_ERR_UNSUPPORTED
    assert _fwd(clib, T=0) == binding.FA_OK                          # nothing to do


def test_bwd_validation(clib):
    P = ctypes.c_void_p

    def call(ws=256, ws_bytes=1 << 20, H=128, dq=16):
        return clib.fa_bwd(P(16), P(16), P(16), P(16), P(16), P(16), None, None, 1,
                           P(dq), P(16), P(16), P(ws), ws_bytes, 1, 1, 4, 128, 128, H, None)

    assert call(dq=0) == binding.FA_ERR_INVALID_ARG
    assert call(ws=0) == binding.FA_ERR_INVALID_ARG
    assert call(ws=272) == binding.FA_ERR_INVALID_ARG                 # not 256-aligned
    assert call(ws_bytes=16) == binding.FA_ERR_INVALID_ARG
    assert call(H=96) == binding.FA_ERR_UNSUPPORTED


def test_splitkv_host_side(clib):
    assert binding.fa_fwd_splitkv_workspace_size(1, 2, 8, 1, 4096, 128, 4) == \
        ((4 * 16 * 128 * 4 + 255) // 256) * 256 + 256
    assert binding.fa_fwd_splitkv_workspace_size(1, 2, 8, 1, 4096, 128, 0) == 0
    P = ctypes.c_void_p
    rc = clib.fa_fwd_splitkv(P(16), P(16), P(16), None, None, 0, P(16), P(16), 0, P(256), 1 << 20,
                             1, 1, 8, 1, 256, 128, None)
    assert rc == binding.FA_ERR_INVALID_ARG          # n_splits must be >= 1
    rc = clib.fa_fwd_splitkv(P(16), P(16), P(16), None, None, 0, P(16), P(16), 4, P(256), 16,
                             1, 1, 8, 1, 256, 128, None)
    assert rc == binding.FA_ERR_INVALID_ARG          # workspace too small


def test_wait_limit_setter(clib):
    assert binding.fa_set_wait_limit_ns(0) == binding.FA_ERR_INVALID_ARG
    assert binding.fa_set_wait_limit_ns(2_000_000_000) == binding.FA_OK


def test_bwd_kv_rows_setter(clib):
    for bad in (-1, 1, 32, 96, 256):
        assert binding.fa_set_bwd_kv_rows(bad) == binding.FA_ERR_INVALID_ARG
    for ok in (64, 128, 0):
        assert binding.fa_set_bwd_kv_rows(ok) == binding.FA_OK


def test_bwd_q_splits_setter(clib):
    for bad in (-1, 5, 64):
        assert binding.fa_set_bwd_q_splits(bad) == binding.FA_ERR_INVALID_ARG
    for ok in (1, 2, 3, 4, 0):
        assert binding.fa_set_bwd_q_splits(ok) == binding.FA_OK


def test_fwd_schedule_setter(clib):
    for bad in (-1, 3, 100):
        assert binding.fa_set_fwd_schedule(bad) == binding.FA_ERR_INVALID_ARG
    for ok in (1, 2, 0):
        assert binding.fa_set_fwd_schedule(ok) == binding.FA_OK


def test_bwd_plan(clib):
    """The backward's grid plan on a 152-SM GPU (host logic, no device)."""
    plan = lambda *a: binding.fa_bwd_plan(*a)
    OK = binding.FA_OK
    # T=1024 (B2 K2 G4 H128): 32 dK/dV CTAs at 128 keys -> 64-key tiles, 64 CTAs;
    # H <= 128 takes the largest split count that stays within one wave: 2 (128 CTAs)
    assert plan(2, 2, 4, 1024, 1024, 128, 1, 0, 152) == (OK, 64, 2)
    assert plan(2, 2, 4, 1024, 1024, 128, 0, 0, 152) == (OK, 64, 2)
    assert plan(2, 2, 4, 1024, 1024, 128, 0, 1, 152) == (OK, 64, 2)
    assert plan(1, 1, 4, 1024, 1024, 128, 1, 0, 152) == (OK, 64, 4)   # 16 CTAs: 4 fit
    assert plan(1, 5, 4, 2048, 2048, 128, 1, 0, 152) == (OK, 64, 1)   # 160 CTAs: full
    # H=256 T=2048 (B1 K2): 64 CTAs of 64 keys; waves/splits 1, 1/2, 2/3, 2/4 -> causal ties to 4
    assert plan(1, 2, 8, 2048, 2048, 256, 1, 0, 152) == (OK, 64, 4)
    assert plan(1, 2, 8, 2048, 2048, 256, 0, 0, 152) == (OK, 64, 2)
    # H=256 T=8192 (B1 K2): 256 CTAs of 64 keys fill the GPU
    assert plan(1, 2, 8, 8192, 8192, 256, 1, 0, 152) == (OK, 64, 1)
    # packed documents (B4 K8 H128 T=4096): 1024 CTAs of 128 keys
    assert plan(4, 8, 4, 4096, 4096, 128, 1, 1, 152) == (OK, 128, 1)
    # 140 CTAs: every split count gives one wave per split -> 1 unless uneven
    assert plan(1, 140, 1, 64, 64, 256, 0, 0, 152) == (OK, 64, 1)
    assert plan(1, 140, 1, 64, 64, 256, 1, 0, 152) == (OK, 64, 4)
    # no SMs reported: nothing is split, H=128 keeps 128-key tiles
    assert plan(1, 1, 4, 128, 128, 128, 1, 0, 0) == (OK, 128, 1)
    # H = 64 follows the H = 128 rule (it runs the H = 128 kernels)
    assert plan(2, 2, 4, 1024, 1024, 64, 1, 0, 152) == (OK, 64, 2)
    assert plan(4, 8, 4, 4096, 4096, 64, 1, 1, 152) == (OK, 128, 1)
    assert plan(1, 1, 4, 128, 128, 96, 1, 0, 152)[0] == binding.FA_ERR_UNSUPPORTED
    assert plan(1, 1, 4, 128, 128, 128, 1, 0, -1)[0] == binding.FA_ERR_INVALID_ARG
