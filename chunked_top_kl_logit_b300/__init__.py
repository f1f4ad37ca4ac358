"""Python binding of libkdtopk.so: the fused, chunked top-K KL distillation loss.

Argument marshalling only.  Every step of the loss runs in the library's CUDA
kernels; PyTorch supplies device memory and the current stream.  There is no
fallback: if the library is missing or the device is not an sm_103a GPU, the
calls raise.

The functions keep the C ABI's names (see include/kd_topk_kl.h):

    kd_topk_kl_workspace_size(T, V, d, K, chunk) -> (fwd_bytes, bwd_bytes)
    kd_topk_kl_forward(h, W, teacher_idx, teacher_logits, valid, tau, chunk,
                       loss, lse, row_kl=None, gathered_idx=None, ws=..., dev_status=...)
    kd_topk_kl_backward(h, W, teacher_idx, teacher_logits, valid, tau, chunk,
                        lse, grad_loss, dh, dW, ws=..., dev_status=...)
    kd_gemm_bf16_diag(A, B, C, M, N, Kd, a_mn, b_mn, dev_status=...)

plus `TopKKL`, a small helper that allocates outputs and workspace with torch
and runs forward + backward.
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "KD_OK", "KDError", "lib", "library_path", "status_string",
    "kd_topk_kl_workspace_size", "kd_topk_kl_launch_count", "kd_topk_kl_forward",
    "kd_topk_kl_forward_backward_workspace_size",
    "kd_topk_kl_forward_noalloc", "kd_topk_kl_backward", "kd_topk_kl_forward_backward",
    "KD_ACCUMULATE_DW", "KD_VALID_ROWS_ONLY", "kd_entropy_filter_workspace_size",
    "kd_entropy_filter",
    "kd_topk_kl_forward_residual", "kd_topk_kl_backward_residual",
    "kd_topk_kl_forward_backward_residual",
    "kd_teacher_topk_workspace_size", "kd_teacher_topk", "PRODUCER_KERNELS",
    "kd_gemm_bf16_diag", "kd_gemm_bf16_diag_pair", "kd_pipeline_wait_selftest", "check_device_status", "TopKKL",
    "KERNELS", "SWEEP_KERNELS", "kd_timing_start", "kd_timing_stop", "kd_timing_query", "kd_timing_release",
    "topk_kl_loss",
]

# contraction kernel ids of the diagnostic timing interface
KERNELS = {"logits_fwd": 0, "logits_bwd": 1, "dh": 3, "dW": 4}
# the single sweep's cached-column pass (a SIMT kernel), timed the same way
SWEEP_KERNELS = {"sweep_fix": 7}
PRODUCER_KERNELS = {"topk_pass1": 5, "topk_scan": 6}

KD_OK = 0
KD_ACCUMULATE_DW = 1
KD_VALID_ROWS_ONLY = 2
_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def library_path() -> str:
    return os.path.join(_HERE, "libkdtopk.so")


class KDError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (code {code})")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libkdtopk.so (built by __graft_entry__.build() / _build.py)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing; build it with python -m chunked_top_kl_logit_b300._build")
        L = ctypes.CDLL(path)
        i64, i32, f32, vp, sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
        L.kd_topk_kl_workspace_size.argtypes = [i64, i64, i64, i32, i64, ctypes.POINTER(sz), ctypes.POINTER(sz)]
        L.kd_topk_kl_workspace_size.restype = ctypes.c_int
        L.kd_topk_kl_launch_count.argtypes = [i64, i64, i64, i32, i64, ctypes.POINTER(i32),
                                               ctypes.POINTER(i32)]
        L.kd_topk_kl_launch_count.restype = ctypes.c_int
        L.kd_topk_kl_forward_backward_workspace_size.argtypes = [i64, i64, i64, i32, i64,
                                                                 ctypes.POINTER(sz),
                                                                 ctypes.POINTER(i32)]
        L.kd_topk_kl_forward_backward_workspace_size.restype = ctypes.c_int
        L.kd_topk_kl_forward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, f32, i64,
                                         vp, vp, vp, vp, vp, sz, vp, vp]
        L.kd_topk_kl_forward.restype = ctypes.c_int
        L.kd_topk_kl_backward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, f32, i64,
                                          vp, f32, vp, vp, vp, sz, vp, vp]
        L.kd_topk_kl_backward.restype = ctypes.c_int
        L.kd_topk_kl_forward_backward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, f32, i64,
                                                  f32, ctypes.c_uint32, vp, vp, vp, vp, vp, vp,
                                                  sz, vp, vp]
        L.kd_topk_kl_forward_backward.restype = ctypes.c_int
        L.kd_topk_kl_forward_residual.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, f32,
                                                  i64, vp, vp, vp, vp, vp, sz, vp, vp]
        L.kd_topk_kl_forward_residual.restype = ctypes.c_int
        L.kd_topk_kl_backward_residual.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, f32,
                                                   i64, vp, vp, f32, vp, vp, vp, sz, vp, vp]
        L.kd_topk_kl_backward_residual.restype = ctypes.c_int
        L.kd_topk_kl_forward_backward_residual.argtypes = [
            vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, f32, i64, f32, ctypes.c_uint32, vp, vp, vp,
            vp, vp, vp, vp, sz, vp, vp]
        L.kd_topk_kl_forward_backward_residual.restype = ctypes.c_int
        L.kd_teacher_topk_workspace_size.argtypes = [i64, i64, i64, i32, i64, ctypes.POINTER(sz)]
        L.kd_teacher_topk_workspace_size.restype = ctypes.c_int
        L.kd_teacher_topk.argtypes = [vp, vp, i64, i64, i64, i32, f32, i64, vp, vp, vp, vp, sz, vp,
                                      vp]
        L.kd_teacher_topk.restype = ctypes.c_int
        L.kd_entropy_filter_workspace_size.argtypes = [i64, ctypes.POINTER(sz)]
        L.kd_entropy_filter_workspace_size.restype = ctypes.c_int
        L.kd_entropy_filter.argtypes = [vp, vp, i64, i32, f32, i32, i32, vp, vp, vp, sz, vp, vp]
        L.kd_entropy_filter.restype = ctypes.c_int
        L.kd_topk_kl_status_string.argtypes = [ctypes.c_int]
        L.kd_topk_kl_status_string.restype = ctypes.c_char_p
        L.kd_topk_kl_forward_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, f32,
                                                 vp, vp, vp, vp, vp, vp]
        L.kd_topk_kl_forward_noalloc.restype = ctypes.c_int
        L.kd_gemm_bf16_diag.argtypes = [vp, vp, vp, i64, i64, i64, i32, i32, vp, vp]
        L.kd_gemm_bf16_diag.restype = ctypes.c_int
        L.kd_gemm_bf16_diag_pair.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp]
        L.kd_gemm_bf16_diag_pair.restype = ctypes.c_int
        L.kd_pipeline_wait_selftest.argtypes = [ctypes.c_uint64, vp, vp]
        L.kd_pipeline_wait_selftest.restype = ctypes.c_int
        L.kd_timing_start.argtypes = [i32]
        L.kd_timing_start.restype = ctypes.c_int
        L.kd_timing_stop.argtypes = []
        L.kd_timing_stop.restype = ctypes.c_int
        L.kd_timing_query.argtypes = [i32, ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_double)]
        L.kd_timing_query.restype = ctypes.c_int
        L.kd_timing_release.argtypes = []
        L.kd_timing_release.restype = ctypes.c_int
        _LIB = L
    return _LIB


def status_string(code: int) -> str:
    return lib().kd_topk_kl_status_string(int(code)).decode()


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, *tensors):
    """Handle of the stream the library enqueues on (`stream`, else torch's
    current stream).  The library takes its launch configuration and tensor
    maps from the current device, so every tensor and the stream must live on
    the current device; anything else raises before a call is made."""
    cur = torch.cuda.current_device()
    if stream is None:
        stream = torch.cuda.current_stream()
    if stream.device.index != cur:
        raise ValueError(f"the stream is on {stream.device} but the current device is cuda:{cur}")
    for t in tensors:
        if t is not None and (t.device.type != "cuda" or t.device.index != cur):
            raise ValueError(f"a tensor is on {t.device} but the current device is cuda:{cur}; "
                             f"run the call inside torch.cuda.device(...) of its tensors")
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, where: str):
    if rc != KD_OK:
        raise KDError(rc, where)


def kd_topk_kl_workspace_size(T: int, V: int, d: int, K: int, chunk: int):
    f, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib().kd_topk_kl_workspace_size(T, V, d, K, chunk, ctypes.byref(f), ctypes.byref(b)),
           "kd_topk_kl_workspace_size")
    return f.value, b.value


def kd_topk_kl_launch_count(T: int, V: int, d: int, K: int, chunk: int):
    f, b = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib().kd_topk_kl_launch_count(T, V, d, K, chunk, ctypes.byref(f), ctypes.byref(b)),
           "kd_topk_kl_launch_count")
    return f.value, b.value


def kd_topk_kl_forward_backward_workspace_size(T: int, V: int, d: int, K: int, chunk: int):
    """(workspace bytes, kernel launches) of kd_topk_kl_forward_backward."""
    b, n = ctypes.c_size_t(0), ctypes.c_int32(0)
    _check(lib().kd_topk_kl_forward_backward_workspace_size(T, V, d, K, chunk, ctypes.byref(b),
                                                            ctypes.byref(n)),
           "kd_topk_kl_forward_backward_workspace_size")
    return b.value, n.value


def kd_topk_kl_forward(h, W, teacher_idx, teacher_logits, valid, tau, chunk, loss, lse,
                       row_kl=None, gathered_idx=None, *, ws, dev_status, stream=None):
    T, d = h.shape
    V = W.shape[0]
    K = teacher_idx.shape[1]
    st = _stream(stream, h, W, teacher_idx, teacher_logits, valid, loss, lse, row_kl,
                 gathered_idx, ws, dev_status)
    rc = lib().kd_topk_kl_forward(_ptr(h), _ptr(W), _ptr(teacher_idx), _ptr(teacher_logits),
                                  _ptr(valid), T, V, d, K, float(tau), int(chunk), _ptr(loss),
                                  _ptr(lse), _ptr(row_kl), _ptr(gathered_idx), _ptr(ws),
                                  ws.numel() * ws.element_size(), _ptr(dev_status), st)
    _check(rc, "kd_topk_kl_forward")


def kd_topk_kl_forward_noalloc(h, W, teacher_idx, teacher_logits, valid, tau, loss, lse,
                               row_kl=None, gathered_idx=None, *, dev_status, stream=None):
    """Forward on the library's built-in 32 MiB scratch (no workspace argument)."""
    T, d = h.shape
    V = W.shape[0]
    K = teacher_idx.shape[1]
    st = _stream(stream, h, W, teacher_idx, teacher_logits, valid, loss, lse, row_kl,
                 gathered_idx, dev_status)
    rc = lib().kd_topk_kl_forward_noalloc(_ptr(h), _ptr(W), _ptr(teacher_idx),
                                          _ptr(teacher_logits), _ptr(valid), T, V, d, K,
                                          float(tau), _ptr(loss), _ptr(lse), _ptr(row_kl),
                                          _ptr(gathered_idx), _ptr(dev_status), st)
    _check(rc, "kd_topk_kl_forward_noalloc")


def kd_topk_kl_backward(h, W, teacher_idx, teacher_logits, valid, tau, chunk, lse, grad_loss,
                        dh, dW, *, ws, dev_status, stream=None):
    T, d = h.shape
    V = W.shape[0]
    K = teacher_idx.shape[1]
    st = _stream(stream, h, W, teacher_idx, teacher_logits, valid, lse, dh, dW, ws, dev_status)
    rc = lib().kd_topk_kl_backward(_ptr(h), _ptr(W), _ptr(teacher_idx), _ptr(teacher_logits),
                                   _ptr(valid), T, V, d, K, float(tau), int(chunk), _ptr(lse),
                                   float(grad_loss), _ptr(dh), _ptr(dW), _ptr(ws),
                                   ws.numel() * ws.element_size(), _ptr(dev_status), st)
    _check(rc, "kd_topk_kl_backward")


def kd_topk_kl_forward_backward(h, W, teacher_idx, teacher_logits, valid, tau, chunk, grad_loss,
                                loss, lse, dh, dW, row_kl=None, *, flags=0, ws, dev_status,
                                stream=None):
    """Forward + backward in one call (one teacher prep); flags: KD_ACCUMULATE_DW,
    KD_VALID_ROWS_ONLY."""
    T, d = h.shape
    V = W.shape[0]
    K = teacher_idx.shape[1]
    st = _stream(stream, h, W, teacher_idx, teacher_logits, valid, loss, lse, row_kl, dh, dW,
                 ws, dev_status)
    rc = lib().kd_topk_kl_forward_backward(
        _ptr(h), _ptr(W), _ptr(teacher_idx), _ptr(teacher_logits), _ptr(valid), T, V, d, K,
        float(tau), int(chunk), float(grad_loss), int(flags), _ptr(loss), _ptr(lse), _ptr(row_kl),
        _ptr(dh), _ptr(dW), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status), st)
    _check(rc, "kd_topk_kl_forward_backward")


def kd_topk_kl_forward_backward_residual(h, W, teacher_idx, teacher_logits, teacher_lse, valid,
                                         tau, chunk, grad_loss, loss, lse, outside_mass, dh, dW,
                                         row_kl=None, *, flags=0, ws, dev_status, stream=None):
    """The residual-mass variant's forward + backward in one call (the single
    sweep); flags: KD_ACCUMULATE_DW, KD_VALID_ROWS_ONLY."""
    T, d = h.shape
    V = W.shape[0]
    K = teacher_idx.shape[1]
    st = _stream(stream, h, W, teacher_idx, teacher_logits, teacher_lse, valid, loss, lse,
                 outside_mass, row_kl, dh, dW, ws, dev_status)
    rc = lib().kd_topk_kl_forward_backward_residual(
        _ptr(h), _ptr(W), _ptr(teacher_idx), _ptr(teacher_logits), _ptr(teacher_lse), _ptr(valid),
        T, V, d, K, float(tau), int(chunk), float(grad_loss), int(flags), _ptr(loss), _ptr(lse),
        _ptr(row_kl), _ptr(outside_mass), _ptr(dh), _ptr(dW), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(dev_status), st)
    _check(rc, "kd_topk_kl_forward_backward_residual")


def kd_topk_kl_forward_residual(h, W, teacher_idx, teacher_logits, teacher_lse, valid, tau, chunk,
                                loss, lse, row_kl=None, outside_mass=None, *, ws, dev_status,
                                stream=None):
    """Forward of the residual-mass variant (teacher full-vocabulary normaliser);
    outside_mass receives the student's mass outside the cached entries."""
    T, d = h.shape
    V = W.shape[0]
    K = teacher_idx.shape[1]
    st = _stream(stream, h, W, teacher_idx, teacher_logits, teacher_lse, valid, loss, lse,
                 row_kl, outside_mass, ws, dev_status)
    rc = lib().kd_topk_kl_forward_residual(
        _ptr(h), _ptr(W), _ptr(teacher_idx), _ptr(teacher_logits), _ptr(teacher_lse), _ptr(valid),
        T, V, d, K, float(tau), int(chunk), _ptr(loss), _ptr(lse), _ptr(row_kl),
        _ptr(outside_mass), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status), st)
    _check(rc, "kd_topk_kl_forward_residual")


def kd_topk_kl_backward_residual(h, W, teacher_idx, teacher_logits, teacher_lse, valid, tau,
                                 chunk, lse, outside_mass, grad_loss, dh, dW, *, ws, dev_status,
                                 stream=None):
    """Backward of the residual-mass variant; lse and outside_mass from its forward."""
    T, d = h.shape
    V = W.shape[0]
    K = teacher_idx.shape[1]
    st = _stream(stream, h, W, teacher_idx, teacher_logits, teacher_lse, valid, lse,
                 outside_mass, dh, dW, ws, dev_status)
    rc = lib().kd_topk_kl_backward_residual(
        _ptr(h), _ptr(W), _ptr(teacher_idx), _ptr(teacher_logits), _ptr(teacher_lse), _ptr(valid),
        T, V, d, K, float(tau), int(chunk), _ptr(lse), _ptr(outside_mass), float(grad_loss),
        _ptr(dh), _ptr(dW), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status), st)
    _check(rc, "kd_topk_kl_backward_residual")


def kd_teacher_topk_workspace_size(T: int, V: int, d: int, K: int, chunk: int) -> int:
    b = ctypes.c_size_t(0)
    _check(lib().kd_teacher_topk_workspace_size(T, V, d, K, chunk, ctypes.byref(b)),
           "kd_teacher_topk_workspace_size")
    return b.value


def kd_teacher_topk(h, W, K, tau, chunk, topk_idx, topk_logits, full_lse=None, *, ws, dev_status,
                    stream=None):
    """Per row the K largest logits of h W^T (descending, ties by lower index),
    their indices, and optionally the full-vocabulary lse of z / tau."""
    T, d = h.shape
    V = W.shape[0]
    st = _stream(stream, h, W, topk_idx, topk_logits, full_lse, ws, dev_status)
    rc = lib().kd_teacher_topk(_ptr(h), _ptr(W), T, V, d, int(K), float(tau), int(chunk),
                               _ptr(topk_idx), _ptr(topk_logits), _ptr(full_lse), _ptr(ws),
                               ws.numel() * ws.element_size(), _ptr(dev_status), st)
    _check(rc, "kd_teacher_topk")


def kd_entropy_filter_workspace_size(T: int) -> int:
    b = ctypes.c_size_t(0)
    _check(lib().kd_entropy_filter_workspace_size(T, ctypes.byref(b)),
           "kd_entropy_filter_workspace_size")
    return b.value


def kd_entropy_filter(teacher_logits, valid_in, tau, keep_num, keep_den, valid_out,
                      entropy=None, *, ws, dev_status, stream=None):
    """Keep the ceil(N_in * keep_num / keep_den) highest-entropy valid rows."""
    T, K = teacher_logits.shape
    st = _stream(stream, teacher_logits, valid_in, valid_out, entropy, ws, dev_status)
    rc = lib().kd_entropy_filter(_ptr(teacher_logits), _ptr(valid_in), T, K, float(tau),
                                 int(keep_num), int(keep_den), _ptr(valid_out), _ptr(entropy),
                                 _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status), st)
    _check(rc, "kd_entropy_filter")


def kd_gemm_bf16_diag(A, B, C, M, N, Kd, a_mn, b_mn, *, dev_status, stream=None):
    st = _stream(stream, A, B, C, dev_status)
    rc = lib().kd_gemm_bf16_diag(_ptr(A), _ptr(B), _ptr(C), M, N, Kd, int(a_mn), int(b_mn),
                                 _ptr(dev_status), st)
    _check(rc, "kd_gemm_bf16_diag")


def kd_gemm_bf16_diag_pair(A, B, C, M, N, Kd, *, dev_status, stream=None):
    """C = A B^T on the CTA-pair (cta_group::2) pipeline; A [M, Kd], B [N, Kd] bf16."""
    st = _stream(stream, A, B, C, dev_status)
    rc = lib().kd_gemm_bf16_diag_pair(_ptr(A), _ptr(B), _ptr(C), M, N, Kd, _ptr(dev_status), st)
    _check(rc, "kd_gemm_bf16_diag_pair")


def kd_pipeline_wait_selftest(limit_ns, *, dev_status, stream=None):
    st = _stream(stream, dev_status)
    rc = lib().kd_pipeline_wait_selftest(int(limit_ns), _ptr(dev_status), st)
    _check(rc, "kd_pipeline_wait_selftest")


def kd_timing_start(capacity: int):
    """Start bracketing each contraction launch with CUDA events (diagnostic)."""
    _check(lib().kd_timing_start(int(capacity)), "kd_timing_start")


def kd_timing_stop():
    _check(lib().kd_timing_stop(), "kd_timing_stop")


def kd_timing_query(kernel: int):
    """(launches, total milliseconds) of the recorded launches of one kernel id."""
    n, ms = ctypes.c_int32(0), ctypes.c_double(0.0)
    _check(lib().kd_timing_query(int(kernel), ctypes.byref(n), ctypes.byref(ms)),
           "kd_timing_query")
    return n.value, ms.value


def kd_timing_release():
    _check(lib().kd_timing_release(), "kd_timing_release")


def check_device_status(dev_status, where: str = "device"):
    """Synchronise-read the device status word and raise if it holds an error."""
    code = int(dev_status.item())
    if code != KD_OK:
        raise KDError(code, where)


class _TopKKLFunction(torch.autograd.Function):
    """Autograd adapter: the forward runs kd_topk_kl_forward, the backward
    kd_topk_kl_backward with the upstream gradient as grad_loss.  Workspaces are
    allocated per call from torch's caching allocator."""

    @staticmethod
    def forward(ctx, h, W, teacher_idx, teacher_logits, valid, tau, chunk):
        T, d = h.shape
        V = W.shape[0]
        K = teacher_idx.shape[1]
        fwd, _ = kd_topk_kl_workspace_size(T, V, d, K, chunk)
        dev = h.device
        ws = torch.empty(fwd, dtype=torch.uint8, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        loss = torch.empty(1, dtype=torch.float32, device=dev)
        lse = torch.empty(T, dtype=torch.float32, device=dev)
        kd_topk_kl_forward(h, W, teacher_idx, teacher_logits, valid, tau, chunk, loss, lse,
                           ws=ws, dev_status=status)
        ctx.save_for_backward(h, W, teacher_idx, teacher_logits, valid, lse, status)
        ctx.tau, ctx.chunk = float(tau), int(chunk)
        return loss.view(())

    @staticmethod
    def backward(ctx, grad):
        h, W, teacher_idx, teacher_logits, valid, lse, status = ctx.saved_tensors
        with torch.cuda.device(h.device):
            return _TopKKLFunction._backward(ctx, grad, h, W, teacher_idx, teacher_logits, valid,
                                             lse, status)

    @staticmethod
    def _backward(ctx, grad, h, W, teacher_idx, teacher_logits, valid, lse, status):
        check_device_status(status, "kd_topk_kl_forward")
        T, d = h.shape
        V = W.shape[0]
        K = teacher_idx.shape[1]
        _, bwd = kd_topk_kl_workspace_size(T, V, d, K, ctx.chunk)
        ws = torch.empty(bwd, dtype=torch.uint8, device=h.device)
        dh = torch.empty(T, d, dtype=torch.float32, device=h.device)
        dW = torch.empty(V, d, dtype=torch.float32, device=h.device)
        kd_topk_kl_backward(h, W, teacher_idx, teacher_logits, valid, ctx.tau, ctx.chunk, lse,
                            float(grad), dh, dW, ws=ws, dev_status=status)
        check_device_status(status, "kd_topk_kl_backward")
        return dh, dW, None, None, None, None, None


def topk_kl_loss(h, W, teacher_idx, teacher_logits, valid, tau, chunk=4096):
    """The fused top-K KL distillation loss as a differentiable torch function.

    h bf16 [T, d] and W bf16 [V, d] (the student's final hidden states and LM
    head), teacher_idx int32 [T, K], teacher_logits fp32 [T, K], valid uint8 [T],
    all contiguous on one CUDA device (checked; the call runs with that device
    current).  Returns the scalar loss (fp32); its
    backward gives dh and dW from the library (fp32; autograd casts them to the
    parameters' dtype).  The backward reads the upstream gradient and the status
    word on the host (two synchronisations) and raises KDError on a device error.
    """
    args = ((h, torch.bfloat16, "h"), (W, torch.bfloat16, "W"),
            (teacher_idx, torch.int32, "teacher_idx"),
            (teacher_logits, torch.float32, "teacher_logits"), (valid, torch.uint8, "valid"))
    for t, dt, name in args:
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
    for t, _, name in args:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.device != h.device:
            raise ValueError(f"{name} is on {t.device} but h is on {h.device}: all inputs must "
                             f"be on one CUDA device")
    # the library launches on the current device: make it the inputs' device
    with torch.cuda.device(h.device):
        return _TopKKLFunction.apply(h, W, teacher_idx, teacher_logits, valid, tau, chunk)


class TopKKL:
    """Allocates outputs and one workspace (torch) for a fixed shape and runs
    the library's forward and backward on the current stream.  fused=True sizes
    the workspace for the one-call training step (forward_backward) as well;
    otherwise its first forward_backward call allocates that workspace."""

    def __init__(self, T, V, d, K, chunk, device="cuda", fused=False):
        self.T, self.V, self.d, self.K, self.chunk = T, V, d, K, chunk
        fwd, bwd = kd_topk_kl_workspace_size(T, V, d, K, chunk)
        self.sweep_bytes = kd_topk_kl_forward_backward_workspace_size(T, V, d, K, chunk)[0]
        dev = torch.device(device)
        nbytes = max(fwd, bwd, self.sweep_bytes) if fused else max(fwd, bwd)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self._ws_sweep = None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.loss = torch.empty(1, dtype=torch.float32, device=dev)
        self.lse = torch.empty(T, dtype=torch.float32, device=dev)
        self.row_kl = torch.empty(T, dtype=torch.float32, device=dev)
        self.dh = torch.empty(T, d, dtype=torch.float32, device=dev)
        self.dW = torch.empty(V, d, dtype=torch.float32, device=dev)

    def forward(self, h, W, idx, tl, valid, tau, gathered_idx=None, row_kl=True, stream=None):
        kd_topk_kl_forward(h, W, idx, tl, valid, tau, self.chunk, self.loss, self.lse,
                           self.row_kl if row_kl else None, gathered_idx, ws=self.ws,
                           dev_status=self.status, stream=stream)
        return self.loss

    def _sweep_ws(self):
        if self.ws.numel() >= self.sweep_bytes:
            return self.ws
        if self._ws_sweep is None:
            self._ws_sweep = torch.empty(self.sweep_bytes, dtype=torch.uint8,
                                         device=self.ws.device)
        return self._ws_sweep

    def forward_backward(self, h, W, idx, tl, valid, tau, grad_loss=1.0, accumulate_dW=False,
                         row_kl=True, stream=None, valid_rows_only=False):
        kd_topk_kl_forward_backward(h, W, idx, tl, valid, tau, self.chunk, grad_loss, self.loss,
                                    self.lse, self.dh, self.dW,
                                    self.row_kl if row_kl else None,
                                    flags=(KD_ACCUMULATE_DW if accumulate_dW else 0)
                                    | (KD_VALID_ROWS_ONLY if valid_rows_only else 0),
                                    ws=self._sweep_ws(), dev_status=self.status, stream=stream)
        return self.loss, self.dh, self.dW

    def forward_backward_residual(self, h, W, idx, tl, teacher_lse, valid, tau, grad_loss=1.0,
                                  accumulate_dW=False, row_kl=True, stream=None,
                                  valid_rows_only=False):
        """The residual-mass variant's training step; the student's mass outside
        the cache lands in self.outside_mass."""
        if getattr(self, "outside_mass", None) is None:
            self.outside_mass = torch.empty_like(self.lse)
        kd_topk_kl_forward_backward_residual(
            h, W, idx, tl, teacher_lse, valid, tau, self.chunk, grad_loss, self.loss, self.lse,
            self.outside_mass, self.dh, self.dW, self.row_kl if row_kl else None,
            flags=(KD_ACCUMULATE_DW if accumulate_dW else 0)
            | (KD_VALID_ROWS_ONLY if valid_rows_only else 0),
            ws=self._sweep_ws(), dev_status=self.status, stream=stream)
        return self.loss, self.dh, self.dW

    def backward(self, h, W, idx, tl, valid, tau, grad_loss=1.0, stream=None):
        kd_topk_kl_backward(h, W, idx, tl, valid, tau, self.chunk, self.lse, grad_loss,
                            self.dh, self.dW, ws=self.ws, dev_status=self.status, stream=stream)
        return self.dh, self.dW
