"""The C ABI without a GPU: the library loads, exports every function the
public header declares, and rejects bad arguments synchronously with a
kd_status code before touching CUDA.  The device pointers below are fake,
16-byte-aligned addresses: the library never dereferences a device pointer on
the host, and every case here returns before any CUDA call."""

import ctypes
import os
import re

import pytest

import chunked_top_kl_logit_b300 as kd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kd_topk_kl.h")

OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA, RANGE, TIMEOUT = range(7)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kd_\w+)\s*\(", text)))


def test_header_symbols_exported():
    names = declared_functions()
    assert "kd_topk_kl_forward" in names and "kd_topk_kl_backward" in names
    L = kd.lib()
    for n in names:
        assert hasattr(L, n), n
        getattr(L, n)  # resolves the symbol


def test_status_strings():
    for code in range(10):
        s = kd.status_string(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert kd.status_string(99) == "unknown status"


def test_workspace_sizes():
    f, b = kd.kd_topk_kl_workspace_size(32768, 201088, 2880, 100, 8192)
    # forward: one fp32 lse partial per (row, 256-wide vocab tile) dominates
    assert f >= 32768 * ((201088 + 255) // 256) * 4
    # backward: the bf16 gradient chunk dominates, bounded by chunk x V
    assert 8192 * 201088 * 2 <= b < 8192 * 201088 * 2 + 32768 * 100 * 20 + 8192 * 2880 * 4 * 8
    f1, b1 = kd.kd_topk_kl_workspace_size(32768, 201088, 2880, 100, 2048)
    assert b1 < b and f1 == f


@pytest.mark.parametrize("shape,code", [
    ((0, 1024, 64, 4, 16), INVALID), ((16, 0, 64, 4, 16), INVALID),
    ((16, 1024, 0, 4, 16), INVALID), ((16, 1024, 64, 0, 16), INVALID),
    ((16, 1024, 64, 4, 0), INVALID), ((16, 1020, 64, 4, 16), UNSUPPORTED),
    ((16, 1024, 96, 4, 16), UNSUPPORTED), ((16, 1024, 64, 1025, 16), UNSUPPORTED),
    ((16, 65536, 64, 40000, 16), UNSUPPORTED), ((16, 1024, 64, 4, 16), OK)])
def test_shape_checks(shape, code):
    f, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert kd.lib().kd_topk_kl_workspace_size(*shape, ctypes.byref(f), ctypes.byref(b)) == code


def test_launch_count():
    fl, bl = kd.kd_topk_kl_launch_count(32768, 201088, 2880, 100, 8192)
    # backward: prep + row compaction, then per chunk gather (plain and
    # transposed), recompute, dh, [split reduce], dW
    assert fl == 4 and bl in (2 + 4 * 5, 2 + 4 * 6)


A = 0x10000  # fake, aligned device addresses


def fwd(**kw):
    a = dict(h=A, W=A, idx=A, tl=A, valid=A, T=16, V=1024, d=64, K=4, tau=1.0, chunk=16,
             loss=A, lse=A, row_kl=None, gidx=None, ws=A, ws_bytes=1 << 40, status=A, stream=None)
    a.update(kw)
    vp = ctypes.c_void_p
    return kd.lib().kd_topk_kl_forward(
        vp(a["h"]), vp(a["W"]), vp(a["idx"]), vp(a["tl"]), vp(a["valid"]), a["T"], a["V"], a["d"],
        a["K"], a["tau"], a["chunk"], vp(a["loss"]), vp(a["lse"]), vp(a["row_kl"]),
        vp(a["gidx"]), vp(a["ws"]), a["ws_bytes"], vp(a["status"]), vp(a["stream"]))


def bwd(**kw):
    a = dict(h=A, W=A, idx=A, tl=A, valid=A, T=16, V=1024, d=64, K=4, tau=1.0, chunk=16,
             lse=A, g=1.0, dh=A, dW=A, ws=A, ws_bytes=1 << 40, status=A, stream=None)
    a.update(kw)
    vp = ctypes.c_void_p
    return kd.lib().kd_topk_kl_backward(
        vp(a["h"]), vp(a["W"]), vp(a["idx"]), vp(a["tl"]), vp(a["valid"]), a["T"], a["V"], a["d"],
        a["K"], a["tau"], a["chunk"], vp(a["lse"]), a["g"], vp(a["dh"]), vp(a["dW"]), vp(a["ws"]),
        a["ws_bytes"], vp(a["status"]), vp(a["stream"]))


@pytest.mark.parametrize("kw", [dict(h=None), dict(W=None), dict(idx=None), dict(tl=None),
                                dict(valid=None), dict(ws=None), dict(status=None),
                                dict(loss=None), dict(tau=0.0),
                                dict(tau=-1.0), dict(tau=float("inf")), dict(tau=float("nan")),
                                dict(h=A + 8), dict(W=A + 2), dict(ws=A + 4), dict(idx=A + 2),
                                dict(T=0), dict(K=0)])
def test_forward_invalid_args(kw):
    assert fwd(**kw) == INVALID


@pytest.mark.parametrize("kw", [dict(lse=None), dict(dh=None), dict(dW=None), dict(dh=A + 4),
                                dict(g=float("nan")), dict(tau=0.0), dict(h=None)])
def test_backward_invalid_args(kw):
    assert bwd(**kw) == INVALID


def test_shape_limits_reported_as_unsupported():
    assert fwd(V=1020) == UNSUPPORTED
    assert fwd(d=100) == UNSUPPORTED
    assert bwd(K=2000) == UNSUPPORTED


def test_workspace_too_small():
    f, b = kd.kd_topk_kl_workspace_size(16, 1024, 64, 4, 16)
    assert fwd(ws_bytes=f - 1) == WORKSPACE
    assert bwd(ws_bytes=b - 1) == WORKSPACE


def test_diag_and_selftest_arg_checks():
    vp = ctypes.c_void_p
    L = kd.lib()
    assert L.kd_gemm_bf16_diag(None, vp(A), vp(A), 8, 8, 8, 0, 0, vp(A), None) == INVALID
    assert L.kd_gemm_bf16_diag(vp(A), vp(A), vp(A), 8, 8, 8, 2, 0, vp(A), None) == INVALID
    assert L.kd_gemm_bf16_diag(vp(A), vp(A), vp(A), 12, 8, 8, 0, 0, vp(A), None) == UNSUPPORTED
    assert L.kd_pipeline_wait_selftest(0, vp(A), None) == INVALID
    assert L.kd_pipeline_wait_selftest(2_000_000_000, vp(A), None) == INVALID
    assert L.kd_pipeline_wait_selftest(1000, None, None) == INVALID


def test_timing_interface_without_records():
    """Querying before anything was recorded returns zero launches and makes no
    CUDA call; a bad capacity is rejected before any CUDA call."""
    assert kd.lib().kd_timing_start(0) == INVALID
    assert kd.lib().kd_timing_stop() == OK
    for kernel in kd.KERNELS.values():
        assert kd.kd_timing_query(kernel) == (0, 0.0)
    assert kd.lib().kd_timing_release() == OK


def test_forward_backward_argument_checks():
    """The fused entry rejects bad flags, a missing lse and a small workspace
    before any CUDA call."""
    A = ctypes.c_void_p(0x10000)
    T, V, d, K, chunk = 64, 1024, 64, 8, 64
    f, b = kd.kd_topk_kl_workspace_size(T, V, d, K, chunk)
    L = kd.lib()
    args = lambda flags, lse, ws_bytes: (A, A, A, A, A, T, V, d, K, 1.0, chunk, 1.0, flags,
                                         A, lse, None, A, A, A, ws_bytes, A, None)
    sw, _ = kd.kd_topk_kl_forward_backward_workspace_size(T, V, d, K, chunk)
    assert L.kd_topk_kl_forward_backward(*args(4, A, sw)) == INVALID
    assert L.kd_topk_kl_forward_backward(*args(0, None, sw)) == INVALID
    assert L.kd_topk_kl_forward_backward(*args(0, A, sw - 1)) == WORKSPACE


def test_forward_backward_workspace_and_launch_count():
    """The single sweep needs the backward's buffers (its bf16 G chunk holds
    the forward's stored logits first) plus the gathered logits and the row
    tables (T x K and T floats), one chunk's lse partials, three floats per
    chunk row (offsets and scales) and one flag per chunk, and makes
    2 + chunks x (8 or 9) + 2 launches."""
    T, V, d, K = 32768, 201088, 2880, 100
    for chunk in (4096, 8192):
        f, b = kd.kd_topk_kl_workspace_size(T, V, d, K, chunk)
        sw, n = kd.kd_topk_kl_forward_backward_workspace_size(T, V, d, K, chunk)
        extra = sw - b
        tables = T * K * 4 + 786 * chunk * 4 + T * 4 + 3 * chunk * 4
        assert tables <= extra <= tables + 4096
        chunks = -(-T // chunk)
        assert n in (2 + chunks * 8 + 2, 2 + chunks * 9 + 2)
    with pytest.raises(kd.KDError):
        kd.kd_topk_kl_forward_backward_workspace_size(0, V, d, K, 64)
    with pytest.raises(kd.KDError):
        kd.kd_topk_kl_forward_backward_workspace_size(T, 1020, d, K, 64)


def test_residual_entry_argument_checks():
    """The residual-mass entries need teacher_lse (and the backward outside_mass)
    and reject their absence before any CUDA call."""
    vp = ctypes.c_void_p
    L = kd.lib()
    T, V, d, K, chunk = 16, 1024, 64, 4, 16
    f, b = kd.kd_topk_kl_workspace_size(T, V, d, K, chunk)
    assert L.kd_topk_kl_forward_residual(vp(A), vp(A), vp(A), vp(A), None, vp(A), T, V, d, K, 1.0,
                                         chunk, vp(A), vp(A), None, None, vp(A), f, vp(A),
                                         None) == INVALID
    assert L.kd_topk_kl_forward_residual(vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), T, V, d, K,
                                         1.0, chunk, vp(A), vp(A), None, None, vp(A), f - 1,
                                         vp(A), None) == WORKSPACE
    assert L.kd_topk_kl_backward_residual(vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), T, V, d, K,
                                          1.0, chunk, vp(A), None, 1.0, vp(A), vp(A), vp(A), b,
                                          vp(A), None) == INVALID
    assert L.kd_topk_kl_backward_residual(vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), T, V, d, K,
                                          1.0, chunk, vp(A), vp(A), 1.0, vp(A), vp(A), vp(A),
                                          b - 1, vp(A), None) == WORKSPACE


def test_teacher_topk_workspace_and_argument_checks():
    """The producer's workspace holds one chunk's fp32 logits (chunk x V x 4 B)
    and its candidates (at most (K - 1) * 256 + 1 keys of 8 B per row, or the
    whole row when it has fewer than K vocabulary tiles); bad arguments and a
    short workspace are rejected before any CUDA call."""
    T, V, d, K = 32768, 201088, 2880, 100
    cap = (K - 1) * 256 + 1
    sizes = [kd.kd_teacher_topk_workspace_size(T, V, d, K, c) for c in (1024, 4096, 8192)]
    for c, b in zip((1024, 4096, 8192), sizes):
        assert c * V * 4 + c * cap * 8 <= b < c * V * 4 + c * cap * 8 + c * 786 * 12 + (1 << 22)
    assert sizes[0] < sizes[1] < sizes[2]
    # fewer vocabulary tiles than K: every logit of the row is a candidate
    b = kd.kd_teacher_topk_workspace_size(64, 1024, 64, 8, 64)
    assert 64 * 1024 * 4 + 64 * 1024 * 8 <= b
    vp = ctypes.c_void_p
    L = kd.lib()
    T, V, d, K, chunk = 64, 1024, 64, 8, 64
    b = kd.kd_teacher_topk_workspace_size(T, V, d, K, chunk)

    def call(**kw):
        a = dict(h=A, W=A, tau=1.0, idx=A, val=A, lse=None, ws=A, ws_bytes=b, status=A, d=d, V=V)
        a.update(kw)
        return L.kd_teacher_topk(vp(a["h"]), vp(a["W"]), T, a["V"], a["d"], K, a["tau"], chunk,
                                 vp(a["idx"]), vp(a["val"]), vp(a["lse"]), vp(a["ws"]),
                                 a["ws_bytes"], vp(a["status"]), None)

    for kw in (dict(h=None), dict(W=None), dict(idx=None), dict(val=None), dict(ws=None),
               dict(status=None), dict(tau=0.0), dict(tau=float("nan")), dict(h=A + 8),
               dict(ws=A + 4), dict(idx=A + 2), dict(lse=A + 2)):
        assert call(**kw) == INVALID, kw
    assert call(ws_bytes=b - 1) == WORKSPACE
    assert call(V=1020) == UNSUPPORTED and call(d=96) == UNSUPPORTED


def test_autograd_adapter_checks_inputs_before_any_call():
    """topk_kl_loss rejects wrong dtypes and host tensors before touching the
    library."""
    import torch
    h = torch.zeros(4, 64, dtype=torch.bfloat16)
    W = torch.zeros(1024, 64, dtype=torch.bfloat16)
    idx = torch.zeros(4, 2, dtype=torch.int32)
    tl = torch.zeros(4, 2, dtype=torch.float32)
    valid = torch.ones(4, dtype=torch.uint8)
    with pytest.raises(TypeError):
        kd.topk_kl_loss(h.float(), W, idx, tl, valid, 1.0, 4)
    with pytest.raises(TypeError):
        kd.topk_kl_loss(h, W, idx.long(), tl, valid, 1.0, 4)
    with pytest.raises(ValueError):
        kd.topk_kl_loss(h, W, idx, tl, valid, 1.0, 4)  # host tensors


class _FakeCuda:
    """Stands in for a CUDA tensor on device `index` (shape, dtype and device
    only); the checks below must reject it before anything reaches the library."""

    def __init__(self, shape, dtype, index):
        import torch
        self.shape, self.dtype, self.is_cuda = shape, dtype, True
        self.device = torch.device("cuda", index)


def test_autograd_adapter_rejects_inputs_on_two_devices():
    import torch
    T, V, d, K = 4, 1024, 64, 2
    args = [_FakeCuda((T, d), torch.bfloat16, 0), _FakeCuda((V, d), torch.bfloat16, 0),
            _FakeCuda((T, K), torch.int32, 0), _FakeCuda((T, K), torch.float32, 0),
            _FakeCuda((T,), torch.uint8, 0)]
    for i in range(1, 5):
        a = list(args)
        a[i] = _FakeCuda(a[i].shape, a[i].dtype, 1)
        with pytest.raises(ValueError, match="one CUDA device"):
            kd.topk_kl_loss(*a, 1.0, 4)


def test_wrappers_reject_tensors_off_the_current_device(monkeypatch):
    """Every wrapper checks that its tensors and stream are on the current
    device (the library launches there) before calling into the library."""
    import torch

    class _Stream:
        device = torch.device("cuda", 0)
        cuda_stream = 0

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: _Stream())
    T, V, d, K = 4, 1024, 64, 2
    on0 = dict(h=_FakeCuda((T, d), torch.bfloat16, 0), W=_FakeCuda((V, d), torch.bfloat16, 0),
               teacher_idx=_FakeCuda((T, K), torch.int32, 0),
               teacher_logits=_FakeCuda((T, K), torch.float32, 0),
               valid=_FakeCuda((T,), torch.uint8, 0))
    out = dict(loss=_FakeCuda((1,), torch.float32, 0), lse=_FakeCuda((T,), torch.float32, 0))
    for name in list(on0) + ["loss", "ws"]:
        kw = dict(on0, **out)
        ws = _FakeCuda((64,), torch.uint8, 0)
        if name == "ws":
            ws = _FakeCuda((64,), torch.uint8, 1)
        else:
            kw[name] = _FakeCuda(kw[name].shape, kw[name].dtype, 1)
        with pytest.raises(ValueError, match="current device"):
            kd.kd_topk_kl_forward(kw["h"], kw["W"], kw["teacher_idx"], kw["teacher_logits"],
                                  kw["valid"], 1.0, 4, kw["loss"], kw["lse"], ws=ws,
                                  dev_status=_FakeCuda((1,), torch.int32, 0))


def test_residual_forward_backward_argument_checks():
    """The residual training step needs teacher_lse and outside_mass, takes the
    same flags as kd_topk_kl_forward_backward and the same workspace."""
    vp = ctypes.c_void_p
    L = kd.lib()
    T, V, d, K, chunk = 64, 1024, 64, 8, 64
    sw, _ = kd.kd_topk_kl_forward_backward_workspace_size(T, V, d, K, chunk)

    def call(tlse=A, mass=A, flags=0, ws_bytes=sw):
        return L.kd_topk_kl_forward_backward_residual(
            vp(A), vp(A), vp(A), vp(A), vp(tlse), vp(A), T, V, d, K, 1.0, chunk, 1.0, flags,
            vp(A), vp(A), None, vp(mass), vp(A), vp(A), vp(A), ws_bytes, vp(A), None)
    assert call(tlse=None) == INVALID
    assert call(mass=None) == INVALID
    assert call(flags=4) == INVALID
    assert call(ws_bytes=sw - 1) == WORKSPACE
