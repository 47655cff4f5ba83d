"""The C-ABI library: it builds, loads, exports every entry point include/longstraw.h
declares, and rejects bad arguments on the host before touching CUDA (runs without a GPU)."""
import ctypes
import os
import re

import pytest

from long_context_grpo_gb300 import build as lsbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "longstraw.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ls_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    path = lsbuild.build()
    from long_context_grpo_gb300 import _lib
    return _lib._lib()


def test_header_declares_the_hot_path():
    names = declared_functions()
    for need in ("ls_prefix_prepare", "ls_replay_fwd", "ls_replay_bwd", "ls_grpo_loss",
                 "ls_prefix_grad_finalize"):
        assert need in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert L.ls_version() == b"0.1.0"
    assert L.ls_status_string(0) == b"ok"
    assert L.ls_status_string(3) == b"prefix handle not prepared"


def test_invalid_arguments_return_before_cuda(L):
    from long_context_grpo_gb300._lib import PrefixDesc
    h = ctypes.c_void_p()
    assert L.ls_prefix_prepare(None, ctypes.byref(h), None) == 1
    # D outside {64, 128}
    d = PrefixDesc(16, 4, 2, 96, 0.0, 0x1000, 0x2000, 0x3000, 0x4000)
    assert L.ls_prefix_prepare(ctypes.byref(d), ctypes.byref(h), None) == 2
    # Hq not a multiple of Hkv
    d = PrefixDesc(16, 3, 2, 64, 0.0, 0x1000, 0x2000, 0x3000, 0x4000)
    assert L.ls_prefix_prepare(ctypes.byref(d), ctypes.byref(h), None) == 2
    # group larger than 16
    d = PrefixDesc(16, 34, 2, 64, 0.0, 0x1000, 0x2000, 0x3000, 0x4000)
    assert L.ls_prefix_prepare(ctypes.byref(d), ctypes.byref(h), None) == 2
    # P = 0
    d = PrefixDesc(0, 4, 2, 64, 0.0, 0x1000, 0x2000, 0x3000, 0x4000)
    assert L.ls_prefix_prepare(ctypes.byref(d), ctypes.byref(h), None) == 1
    # misaligned prompt keys
    d = PrefixDesc(16, 4, 2, 64, 0.0, 0x1008, 0x2000, 0x3000, 0x4000)
    assert L.ls_prefix_prepare(ctypes.byref(d), ctypes.byref(h), None) == 4
    assert h.value is None


def test_calls_without_a_handle(L):
    assert L.ls_replay_fwd(None, 4, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, None) == 3
    assert L.ls_replay_bwd(None, 4, *([0x1000] * 9), 0x1000, 1 << 20, None) == 3
    assert L.ls_prefix_grad_finalize(None, 1.0, None, None, 0, 0, None) == 3
    assert L.ls_prefix_grad_finalize_rows(None, 0, 4, 1.0, None, None, 0, 0, None) == 3
    assert L.ls_block_replay_fwd(None, 16, 4, 0x1000, 0x1000, 0x1000, None) == 3
    assert L.ls_block_replay_bwd(None, 16, 4, *([0x1000] * 6), 1 << 20, None) == 3
    cu = (ctypes.c_int64 * 3)(0, 2, 5)
    assert L.ls_replay_fwd_packed(None, 2, cu, *([0x1000] * 5), None) == 3
    assert L.ls_replay_bwd_packed(None, 2, cu, *([0x1000] * 10), 1 << 20, None) == 3
    assert L.ls_replay_bwd_packed_workspace_bytes(None, 2, cu) == 0
    assert L.ls_replay_fwd_prompt_only(None, 4, 0x1000, 0x1000, 0x1000, None) == 3
    assert L.ls_replay_bwd_prompt_only(None, 4, *([0x1000] * 6), 1 << 20, None) == 3


def test_merge_and_sum_argument_checks(L):
    parts = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    lses = (ctypes.c_void_p * 2)(0x3000, 0x4000)
    assert L.ls_attn_merge(0, 4, 2, 64, parts, lses, 0x5000, 0x6000, None) == 1     # n < 1
    assert L.ls_attn_merge(17, 4, 2, 64, parts, lses, 0x5000, 0x6000, None) == 2    # n > 16
    assert L.ls_attn_merge(2, 4, 2, 60, parts, lses, 0x5000, 0x6000, None) == 2     # D % 8
    assert L.ls_attn_merge(2, 4, 2, 64, None, lses, 0x5000, 0x6000, None) == 1
    bad = (ctypes.c_void_p * 2)(0x1008, 0x2000)
    assert L.ls_attn_merge(2, 4, 2, 64, bad, lses, 0x5000, 0x6000, None) == 4       # misaligned
    assert L.ls_sum_bf16(2, 12, parts, 0x5000, None) == 2                           # count % 8
    assert L.ls_sum_bf16(2, 16, None, 0x5000, None) == 1
    assert L.ls_replay_bwd_workspace_bytes(None, 4) == 0
    assert L.ls_prefix_destroy(None) == 0


def test_loss_argument_checks(L):
    ws = L.ls_grpo_loss_workspace_bytes(100)
    assert ws >= 800 and ws % 256 == 0
    ok = dict(R=100, V=64, G=4, logits=0x1000, ids=0x2000, old=0x3000, A=1.0, eps=0.2,
              loss=0x4000, dl=0x5000, mask=0x6000, logp=0x7000, ws=0x8000, wsb=ws)

    def call(**kw):
        a = dict(ok, **kw)
        return L.ls_grpo_loss(a["R"], a["V"], a["G"], a["logits"], a["ids"], a["old"], a["A"],
                              a["eps"], a["loss"], a["dl"], a["mask"], a["logp"], a["ws"],
                              a["wsb"], None)

    assert call(logits=None) == 1
    assert call(R=0) == 1
    assert call(G=0) == 1
    assert call(eps=1.0) == 1
    assert call(eps=-0.1) == 1
    assert call(A=float("nan")) == 1
    assert call(wsb=ws - 8) == 8
    assert call(ws=None) == 8
    assert call(ids=0x2002) == 4
    assert call(loss=0x4004) == 4


def test_no_gpu_means_a_cuda_error_not_a_fallback(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    ws = L.ls_grpo_loss_workspace_bytes(8)
    st = L.ls_grpo_loss(8, 64, 1, 0x1000, 0x2000, 0x3000, 1.0, 0.2, 0x4000, 0x5000, 0x6000,
                        0x7000, 0x8000, ws, None)
    assert st == 5
