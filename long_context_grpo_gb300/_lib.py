"""Thin ctypes binding over the C ABI in include/longstraw.h.

Argument marshalling only: tensors are checked (device, dtype, shape, contiguity) and
passed as raw pointers with torch's current CUDA stream; every step of the replay runs in
the CUDA library.  PyTorch provides device memory and streams.  There is no fallback: if
the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

library_path = _build.LIB

LS_OK = 0
STATUS_NAMES = {
    0: "LS_OK", 1: "LS_ERR_INVALID_ARGUMENT", 2: "LS_ERR_UNSUPPORTED", 3: "LS_ERR_NOT_PREPARED",
    4: "LS_ERR_MISALIGNED", 5: "LS_ERR_CUDA", 6: "LS_ERR_TIMEOUT", 7: "LS_ERR_DEVICE_STATUS",
    8: "LS_ERR_WORKSPACE", 9: "LS_ERR_WRONG_DEVICE",
}


class LongStrawError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = "%s failed: %s" % (where, STATUS_NAMES.get(status, str(status)))
        if status == 5 and lib is not None:
            msg += " (%s)" % lib.ls_last_error().decode()
        super().__init__(msg)


class PrefixDesc(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int64), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("D", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
                ("k_prefix", ctypes.c_void_p), ("v_prefix", ctypes.c_void_p),
                ("dk_acc", ctypes.c_void_p), ("dv_acc", ctypes.c_void_p)]


def _load():
    if not os.path.exists(library_path):
        raise RuntimeError("liblongstraw.so is not built (run long_context_grpo_gb300/build.py); "
                           "there is no non-CUDA implementation")
    L = ctypes.CDLL(library_path)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    sig = {
        "ls_prefix_prepare": (ctypes.c_int, [ctypes.POINTER(PrefixDesc), ctypes.POINTER(vp), vp]),
        "ls_prefix_destroy": (ctypes.c_int, [vp]),
        "ls_replay_fwd": (ctypes.c_int, [vp, i64, vp, vp, vp, vp, vp, vp]),
        "ls_replay_bwd_workspace_bytes": (sz, [vp, i64]),
        "ls_replay_bwd": (ctypes.c_int, [vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "ls_grpo_loss_workspace_bytes": (sz, [i64]),
        "ls_grpo_loss": (ctypes.c_int, [i64, i64, i32, vp, vp, vp, ctypes.c_double,
                                        ctypes.c_double, vp, vp, vp, vp, vp, sz, vp]),
        "ls_token_logp": (ctypes.c_int, [i64, i64, vp, vp, vp, vp]),
        "ls_grpo_loss_noalloc": (ctypes.c_int, [i64, i64, i32, vp, vp, vp, ctypes.c_double,
                                                ctypes.c_double, vp, vp, vp, vp, vp]),
        "ls_grpo_loss_noalloc_max_rows": (i64, []),
        "ls_prefix_grad_finalize": (ctypes.c_int, [vp, ctypes.c_float, vp, vp, ctypes.c_int,
                                                   ctypes.c_int, vp]),
        "ls_prefix_grad_finalize_rows": (ctypes.c_int, [vp, i64, i64, ctypes.c_float, vp, vp,
                                                        ctypes.c_int, ctypes.c_int, vp]),
        "ls_block_replay_fwd": (ctypes.c_int, [vp, i64, i64, vp, vp, vp, vp]),
        "ls_replay_fwd_packed": (ctypes.c_int, [vp, i32, vp, vp, vp, vp, vp, vp, vp]),
        "ls_replay_fwd_prompt_only": (ctypes.c_int, [vp, i64, vp, vp, vp, vp]),
        "ls_replay_bwd_prompt_only": (ctypes.c_int, [vp, i64, vp, vp, vp, vp, vp, vp, sz, vp]),
        "ls_attn_merge": (ctypes.c_int, [i32, i64, i32, i32, vp, vp, vp, vp, vp]),
        "ls_sum_bf16": (ctypes.c_int, [i32, i64, vp, vp, vp]),
        "ls_bf16_to_f32": (ctypes.c_int, [i64, vp, vp, vp]),
        "ls_f32_to_bf16": (ctypes.c_int, [i64, vp, vp, vp]),
        "ls_replay_bwd_packed_workspace_bytes": (sz, [vp, i32, vp]),
        "ls_replay_bwd_packed": (ctypes.c_int, [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                vp, sz, vp]),
        "ls_block_replay_bwd": (ctypes.c_int, [vp, i64, i64, vp, vp, vp, vp, vp, vp, sz, vp]),
        "ls_get_device_status": (ctypes.c_int, [vp, ctypes.POINTER(ctypes.c_uint32)]),
        "ls_timing_enable": (ctypes.c_int, [ctypes.c_int]),
        "ls_debug_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, vp]),
        "ls_debug_fail_launch": (ctypes.c_int, [i64]),
        "ls_debug_fail_launch_pending": (i64, []),
        "ls_timing_read": (ctypes.c_int, [ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(ctypes.c_int64), ctypes.c_int]),
        "ls_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "ls_last_error": (ctypes.c_char_p, []),
        "ls_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = None


def _lib():
    global lib
    if lib is None:
        lib = _load()
    return lib


def _check(st: int, where: str):
    if st != LS_OK:
        raise LongStrawError(st, where)


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t, name, dtype, shape=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t.data_ptr()


class Prefix:
    """Resident prompt K/V of one attention layer and its fp32 gradient accumulators.

    The tensors are borrowed: they must outlive the handle, and k/v are never written.
    Creating the handle zeroes dk_acc / dv_acc on the current stream.
    """

    def __init__(self, k_prefix, v_prefix, dk_acc, dv_acc, Hq: int, softmax_scale: float = 0.0):
        L = _lib()
        P, Hkv, D = k_prefix.shape
        self.P, self.Hq, self.Hkv, self.D = P, Hq, Hkv, D
        self._keep = (k_prefix, v_prefix, dk_acc, dv_acc)
        d = PrefixDesc(P, Hq, Hkv, D, softmax_scale,
                       _ptr(k_prefix, "k_prefix", torch.bfloat16, (P, Hkv, D)),
                       _ptr(v_prefix, "v_prefix", torch.bfloat16, (P, Hkv, D)),
                       _ptr(dk_acc, "dk_acc", torch.float32, (P, Hkv, D)),
                       _ptr(dv_acc, "dv_acc", torch.float32, (P, Hkv, D)))
        h = ctypes.c_void_p()
        _check(L.ls_prefix_prepare(ctypes.byref(d), ctypes.byref(h), _stream()), "ls_prefix_prepare")
        self._h = h
        self.dk_acc, self.dv_acc = dk_acc, dv_acc

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value is not None:
            _check(_lib().ls_prefix_destroy(self._h), "ls_prefix_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def fwd(self, q, k_suffix, v_suffix, o=None, lse=None):
        R = q.shape[0]
        if o is None:
            o = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((R, self.Hq), dtype=torch.float32, device=q.device)
        _check(_lib().ls_replay_fwd(
            self._h, R,
            _ptr(q, "q", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(k_suffix, "k_suffix", torch.bfloat16, (R, self.Hkv, self.D)),
            _ptr(v_suffix, "v_suffix", torch.bfloat16, (R, self.Hkv, self.D)),
            _ptr(o, "o", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(lse, "lse", torch.float32, (R, self.Hq)), _stream()), "ls_replay_fwd")
        return o, lse

    def bwd_workspace_bytes(self, R: int) -> int:
        return int(_lib().ls_replay_bwd_workspace_bytes(self._h, R))

    def bwd(self, q, k_suffix, v_suffix, o, lse, d_out, dq=None, dk_suffix=None,
            dv_suffix=None, workspace=None):
        R = q.shape[0]
        dq = torch.empty_like(q) if dq is None else dq
        dk_suffix = torch.empty_like(k_suffix) if dk_suffix is None else dk_suffix
        dv_suffix = torch.empty_like(v_suffix) if dv_suffix is None else dv_suffix
        need = self.bwd_workspace_bytes(R)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        _check(_lib().ls_replay_bwd(
            self._h, R,
            _ptr(q, "q", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(k_suffix, "k_suffix", torch.bfloat16, (R, self.Hkv, self.D)),
            _ptr(v_suffix, "v_suffix", torch.bfloat16, (R, self.Hkv, self.D)),
            _ptr(o, "o", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(lse, "lse", torch.float32, (R, self.Hq)),
            _ptr(d_out, "d_out", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(dq, "dq", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(dk_suffix, "dk_suffix", torch.bfloat16, (R, self.Hkv, self.D)),
            _ptr(dv_suffix, "dv_suffix", torch.bfloat16, (R, self.Hkv, self.D)),
            _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream()),
            "ls_replay_bwd")
        return dq, dk_suffix, dv_suffix

    @staticmethod
    def _cu(cu_seqlens):
        cu = [int(x) for x in cu_seqlens]
        return len(cu) - 1, (ctypes.c_int64 * len(cu))(*cu), cu[-1]

    def fwd_packed(self, cu_seqlens, q, k_suffix, v_suffix, o=None, lse=None):
        """One launch for G responses packed along the token axis: response b owns rows
        cu_seqlens[b] .. cu_seqlens[b+1]-1 and sees the prompt and, causally, itself."""
        G, cu, T = self._cu(cu_seqlens)
        if o is None:
            o = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((T, self.Hq), dtype=torch.float32, device=q.device)
        _check(_lib().ls_replay_fwd_packed(
            self._h, G, ctypes.cast(cu, ctypes.c_void_p),
            _ptr(q, "q", torch.bfloat16, (T, self.Hq, self.D)),
            _ptr(k_suffix, "k_suffix", torch.bfloat16, (T, self.Hkv, self.D)),
            _ptr(v_suffix, "v_suffix", torch.bfloat16, (T, self.Hkv, self.D)),
            _ptr(o, "o", torch.bfloat16, (T, self.Hq, self.D)),
            _ptr(lse, "lse", torch.float32, (T, self.Hq)), _stream()), "ls_replay_fwd_packed")
        return o, lse

    def bwd_packed_workspace_bytes(self, cu_seqlens) -> int:
        G, cu, _ = self._cu(cu_seqlens)
        return int(_lib().ls_replay_bwd_packed_workspace_bytes(self._h, G, ctypes.cast(cu, ctypes.c_void_p)))

    def bwd_packed(self, cu_seqlens, q, k_suffix, v_suffix, o, lse, d_out, dq=None,
                   dk_suffix=None, dv_suffix=None, workspace=None):
        G, cu, T = self._cu(cu_seqlens)
        dq = torch.empty_like(q) if dq is None else dq
        dk_suffix = torch.empty_like(k_suffix) if dk_suffix is None else dk_suffix
        dv_suffix = torch.empty_like(v_suffix) if dv_suffix is None else dv_suffix
        if workspace is None:
            workspace = torch.empty(max(self.bwd_packed_workspace_bytes(cu_seqlens), 16),
                                    dtype=torch.uint8, device=q.device)
        _check(_lib().ls_replay_bwd_packed(
            self._h, G, ctypes.cast(cu, ctypes.c_void_p),
            _ptr(q, "q", torch.bfloat16, (T, self.Hq, self.D)),
            _ptr(k_suffix, "k_suffix", torch.bfloat16, (T, self.Hkv, self.D)),
            _ptr(v_suffix, "v_suffix", torch.bfloat16, (T, self.Hkv, self.D)),
            _ptr(o, "o", torch.bfloat16, (T, self.Hq, self.D)),
            _ptr(lse, "lse", torch.float32, (T, self.Hq)),
            _ptr(d_out, "d_out", torch.bfloat16, (T, self.Hq, self.D)),
            _ptr(dq, "dq", torch.bfloat16, (T, self.Hq, self.D)),
            _ptr(dk_suffix, "dk_suffix", torch.bfloat16, (T, self.Hkv, self.D)),
            _ptr(dv_suffix, "dv_suffix", torch.bfloat16, (T, self.Hkv, self.D)),
            _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream()),
            "ls_replay_bwd_packed")
        return dq, dk_suffix, dv_suffix

    def fwd_prompt_only(self, q, o=None, lse=None):
        """Partial attention of q over this handle's prompt keys only (one prompt shard)."""
        R = q.shape[0]
        o = torch.empty_like(q) if o is None else o
        if lse is None:
            lse = torch.empty((R, self.Hq), dtype=torch.float32, device=q.device)
        _check(_lib().ls_replay_fwd_prompt_only(
            self._h, R, _ptr(q, "q", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(o, "o", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(lse, "lse", torch.float32, (R, self.Hq)), _stream()), "ls_replay_fwd_prompt_only")
        return o, lse

    def bwd_prompt_only(self, q, o, lse, d_out, dq=None, workspace=None):
        """Backward over this handle's prompt keys only, with the merged (global) o and lse:
        this shard's part of dq; its key/value gradients go into its accumulators."""
        R = q.shape[0]
        dq = torch.empty_like(q) if dq is None else dq
        if workspace is None:
            workspace = torch.empty(max(self.bwd_workspace_bytes(R), 16), dtype=torch.uint8,
                                    device=q.device)
        _check(_lib().ls_replay_bwd_prompt_only(
            self._h, R, _ptr(q, "q", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(o, "o", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(lse, "lse", torch.float32, (R, self.Hq)),
            _ptr(d_out, "d_out", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(dq, "dq", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream()),
            "ls_replay_bwd_prompt_only")
        return dq

    def block_fwd(self, prefix_len: int, q, o=None, lse=None):
        """Blockwise replay forward: the block's keys/values are rows prefix_len .. of the
        handle's K/V buffers; its queries see rows 0 .. prefix_len-1 and, causally, its own."""
        R = q.shape[0]
        if o is None:
            o = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((R, self.Hq), dtype=torch.float32, device=q.device)
        _check(_lib().ls_block_replay_fwd(
            self._h, prefix_len, R,
            _ptr(q, "q", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(o, "o", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(lse, "lse", torch.float32, (R, self.Hq)), _stream()), "ls_block_replay_fwd")
        return o, lse

    def block_bwd(self, prefix_len: int, q, o, lse, d_out, dq=None, workspace=None):
        """Blockwise replay backward: dq of the block; key/value gradients of rows
        0 .. prefix_len+R-1 added into the accumulators."""
        R = q.shape[0]
        dq = torch.empty_like(q) if dq is None else dq
        need = self.bwd_workspace_bytes(R)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        _check(_lib().ls_block_replay_bwd(
            self._h, prefix_len, R,
            _ptr(q, "q", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(o, "o", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(lse, "lse", torch.float32, (R, self.Hq)),
            _ptr(d_out, "d_out", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(dq, "dq", torch.bfloat16, (R, self.Hq, self.D)),
            _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream()),
            "ls_block_replay_bwd")
        return dq

    def finalize_rows(self, row0: int, nrows: int, scale: float = 1.0, dk_out=None, dv_out=None,
                      out_fp32=False, reset=False):
        shp = (nrows, self.Hkv, self.D)
        dt = torch.float32 if out_fp32 else torch.bfloat16
        _check(_lib().ls_prefix_grad_finalize_rows(
            self._h, row0, nrows, scale, _ptr(dk_out, "dk_out", dt, shp),
            _ptr(dv_out, "dv_out", dt, shp), 1 if out_fp32 else 0, 1 if reset else 0, _stream()),
            "ls_prefix_grad_finalize_rows")
        return dk_out, dv_out

    def finalize(self, scale: float = 1.0, dk_out=None, dv_out=None, out_fp32=False, reset=False):
        shp = (self.P, self.Hkv, self.D)
        dt = torch.float32 if out_fp32 else torch.bfloat16
        _check(_lib().ls_prefix_grad_finalize(
            self._h, scale, _ptr(dk_out, "dk_out", dt, shp), _ptr(dv_out, "dv_out", dt, shp),
            1 if out_fp32 else 0, 1 if reset else 0, _stream()), "ls_prefix_grad_finalize")
        return dk_out, dv_out


def attn_merge(o_parts, lse_parts, o=None, lse=None):
    """Merge per-shard partial attention results: lse = logsumexp_r lse_r,
    o = sum_r exp(lse_r - lse) o_r (bf16 [R, Hq, D] parts, fp32 [R, Hq] lse)."""
    n = len(o_parts)
    R, Hq, D = o_parts[0].shape
    o = torch.empty_like(o_parts[0]) if o is None else o
    lse = torch.empty_like(lse_parts[0]) if lse is None else lse
    op = (ctypes.c_void_p * n)(*[_ptr(t, "o_part", torch.bfloat16, (R, Hq, D)) for t in o_parts])
    lp = (ctypes.c_void_p * n)(*[_ptr(t, "lse_part", torch.float32, (R, Hq)) for t in lse_parts])
    _check(_lib().ls_attn_merge(n, R, Hq, D, ctypes.cast(op, ctypes.c_void_p),
                                ctypes.cast(lp, ctypes.c_void_p),
                                _ptr(o, "o", torch.bfloat16, (R, Hq, D)),
                                _ptr(lse, "lse", torch.float32, (R, Hq)), _stream()), "ls_attn_merge")
    return o, lse


def sum_bf16(parts, out=None):
    """out = bf16(sum of the bf16 parts), fp32 accumulation."""
    n = len(parts)
    out = torch.empty_like(parts[0]) if out is None else out
    pp = (ctypes.c_void_p * n)(*[_ptr(t, "part", torch.bfloat16, tuple(parts[0].shape)) for t in parts])
    _check(_lib().ls_sum_bf16(n, parts[0].numel(), ctypes.cast(pp, ctypes.c_void_p),
                              _ptr(out, "out", torch.bfloat16, tuple(parts[0].shape)), _stream()),
           "ls_sum_bf16")
    return out


def bf16_to_f32(x, out=None):
    """Exact widening of a bf16 tensor to fp32 (numel a multiple of 8)."""
    out = torch.empty(x.shape, dtype=torch.float32, device=x.device) if out is None else out
    _check(_lib().ls_bf16_to_f32(x.numel(), _ptr(x, "x", torch.bfloat16),
                                 _ptr(out, "out", torch.float32, tuple(x.shape)), _stream()),
           "ls_bf16_to_f32")
    return out


def f32_to_bf16(x, out=None):
    """fp32 -> bf16, round to nearest, ties to even (numel a multiple of 8)."""
    out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device) if out is None else out
    _check(_lib().ls_f32_to_bf16(x.numel(), _ptr(x, "x", torch.float32),
                                 _ptr(out, "out", torch.bfloat16, tuple(x.shape)), _stream()),
           "ls_f32_to_bf16")
    return out


def grpo_loss_workspace_bytes(R: int) -> int:
    return int(_lib().ls_grpo_loss_workspace_bytes(R))


def grpo_loss(logits, ids, logp_old, advantage: float, eps: float, G: int, loss_accum,
              dlogits=None, clip_mask=None, logp_out=None, workspace=None):
    """Adds this response's clipped-surrogate loss into loss_accum (fp64 [1]) and returns
    (dlogits bf16 [R,V], clip_mask uint8 [R], logp fp32 [R])."""
    R, V = logits.shape
    dlogits = torch.empty_like(logits) if dlogits is None else dlogits
    clip_mask = torch.empty((R,), dtype=torch.uint8, device=logits.device) if clip_mask is None else clip_mask
    logp_out = torch.empty((R,), dtype=torch.float32, device=logits.device) if logp_out is None else logp_out
    need = grpo_loss_workspace_bytes(R)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=logits.device)
    _check(_lib().ls_grpo_loss(
        R, V, G, _ptr(logits, "logits", torch.bfloat16, (R, V)),
        _ptr(ids, "ids", torch.int32, (R,)), _ptr(logp_old, "logp_old", torch.float32, (R,)),
        float(advantage), float(eps), _ptr(loss_accum, "loss_accum", torch.float64, (1,)),
        _ptr(dlogits, "dlogits", torch.bfloat16, (R, V)),
        _ptr(clip_mask, "clip_mask", torch.uint8, (R,)),
        _ptr(logp_out, "logp_out", torch.float32, (R,)),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream()), "ls_grpo_loss")
    return dlogits, clip_mask, logp_out


KERNEL_NAMES = ("zero", "replay_fwd", "bwd_prep", "bwd_dkdv", "bwd_dq", "grpo_loss", "finalize",
                "token_logp", "merge", "sum", "cast")


def timing_enable(on: bool = True):
    _check(_lib().ls_timing_enable(1 if on else 0), "ls_timing_enable")


def timing_read():
    """{kernel name: (total ms, launches)} since the previous read."""
    n = len(KERNEL_NAMES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _check(_lib().ls_timing_read(ms, cnt, n), "ls_timing_read")
    return {KERNEL_NAMES[i]: (ms[i], cnt[i]) for i in range(n)}


def token_logp(logits, ids, logp_out=None):
    """Scoring without gradients: fp32 log softmax(logits)[ids] per row."""
    R, V = logits.shape
    logp_out = torch.empty((R,), dtype=torch.float32, device=logits.device) if logp_out is None else logp_out
    _check(_lib().ls_token_logp(R, V, _ptr(logits, "logits", torch.bfloat16, (R, V)),
                                _ptr(ids, "ids", torch.int32, (R,)),
                                _ptr(logp_out, "logp_out", torch.float32, (R,)), _stream()),
           "ls_token_logp")
    return logp_out


def device_status():
    """(status, bits) of the device status word; reading it clears it."""
    bits = ctypes.c_uint32(0)
    st = _lib().ls_get_device_status(_stream(), ctypes.byref(bits))
    return st, bits.value
