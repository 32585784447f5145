"""Host-side failure injection: a CUDA launch that fails is reported, and cleaned up after.

The entry points return MT_ERR_CUDA when a CUDA call fails, and mt_last_cuda_error()
returns the failing call's cudaError_t. The allocating backwards (and the norm + GEMV)
take stream-ordered scratch; on a failed launch they must still free it. These tests
make a launch fail on the host, without touching the GPU: a test build of the library
(libmt_norm_hooks.so, api.cu compiled with -DMT_TEST_HOOKS, every kernel object shared
with the product library) has mt_test_fail_launch(skip, err), which makes the launch
after `skip` more launches return `err` instead of launching. The product library has
no such hook.
"""
import ctypes

import pytest
import torch

import row_wise_rmsnorm_gb300 as mt
from row_wise_rmsnorm_gb300 import _binding
from row_wise_rmsnorm_gb300 import build

ERR = 701  # cudaErrorLaunchOutOfResources: what a refused launch would report


def _hooks():
    lib = ctypes.CDLL(build.build_test_hooks())
    for name, args in _binding._SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.mt_test_fail_launch.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.mt_test_fail_launch.restype = None
    lib.mt_test_failure_armed.restype = ctypes.c_int
    lib.mt_test_pool_used_bytes.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_ulonglong)]
    lib.mt_test_pool_used_bytes.restype = ctypes.c_int
    return lib


def test_product_library_has_no_hook():
    build.build()
    lib = ctypes.CDLL(build.LIB)
    for name in ("mt_test_fail_launch", "mt_test_failure_armed", "mt_test_pool_used_bytes"):
        assert not hasattr(lib, name), name
    h = _hooks()
    for name in ("mt_test_fail_launch", "mt_test_failure_armed", "mt_test_pool_used_bytes"):
        assert hasattr(h, name), name


def test_injected_launch_failure_is_reported_without_a_gpu():
    """The forwards make no CUDA call before their launch (vector path: D % 8 == 0,
    16-byte aligned addresses), so with the failure armed each returns MT_ERR_CUDA with
    the injected code, and the hook is consumed. The addresses are never dereferenced."""
    h = _hooks()
    N, D = 8, 64
    a = [0x100000 * (i + 1) for i in range(10)]  # disjoint, 16-byte aligned, 1 KB each
    calls = {
        "mt_rmsnorm_forward": lambda: h.mt_rmsnorm_forward(a[0], a[1], a[2], a[3], N, D, 1e-5, None),
        "mt_layernorm_forward": lambda: h.mt_layernorm_forward(a[0], a[1], a[4], a[2], a[5], a[3],
                                                               N, D, 1e-5, None),
        "mt_add_rmsnorm_forward": lambda: h.mt_add_rmsnorm_forward(a[0], a[6], a[1], a[7], a[2],
                                                                   a[3], N, D, 1e-5, None),
        "mt_norm_forward_ex": lambda: h.mt_norm_forward_ex(mt.MT_OP_RMSNORM, mt.MT_DTYPE_BF16,
                                                           mt.MT_DTYPE_F32, a[0], None, a[1],
                                                           None, None, a[2], None, a[3], N, D,
                                                           1e-5, None),
        "mt_softmax_forward": lambda: h.mt_softmax_forward(mt.MT_DTYPE_F16, a[0], a[2], N, D, 0,
                                                           None),
        "mt_softmax_backward": lambda: h.mt_softmax_backward(mt.MT_DTYPE_F16, a[0], a[1], a[2],
                                                             N, D, 1, None),
        "mt_cross_entropy_forward": lambda: h.mt_cross_entropy_forward(
            mt.MT_DTYPE_BF16, a[0], a[1], N, D, -100, 0.0, 0.0, mt.MT_REDUCTION_NONE, a[2], a[3],
            None, None, None),
    }
    for name, call in calls.items():
        h.mt_test_fail_launch(0, ERR)
        assert h.mt_test_failure_armed() == 1
        assert call() == mt.MT_ERR_CUDA, name
        assert h.mt_last_cuda_error() == ERR, name
        assert h.mt_test_failure_armed() == 0, name


# ------------------------------------------------------------------- GPU ---

def _pool_used(h):
    v = ctypes.c_ulonglong(0)
    assert h.mt_test_pool_used_bytes(torch.cuda.current_device(), ctypes.byref(v)) == 0
    return v.value


def _p(t):
    return None if t is None else t.data_ptr()


@pytest.mark.gpu
@pytest.mark.parametrize("skip", [0, 1])
def test_failed_launch_frees_stream_ordered_workspace(skip):
    """skip = 0 fails an entry point's first launch (the row kernel, or the statistics
    kernel of the norm + GEMV), skip = 1 its second (the parameter reduction, launched
    after the row kernel). Every allocating backward, the no-alloc backward and the norm +
    GEMV return MT_ERR_CUDA with the injected code, and once the stream has drained the
    memory pool is back at its previous use: the scratch was freed on the error path.
    Then the same calls, unarmed, give the product library's results bit for bit."""
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the -m gpu tests")
    h = _hooks()
    prod = mt.load()
    dev = "cuda:0"
    torch.manual_seed(0)
    N, D = 600, 4096
    X = torch.randn(N, D, device=dev).half()
    R = torch.randn(N, D, device=dev).half()
    g = (1 + 0.1 * torch.randn(D, device=dev)).half()
    b = (0.1 * torch.randn(D, device=dev)).half()
    dY = torch.randn(N, D, device=dev).half()
    _, mean, rstd = mt.layernorm_forward(X, g, b)
    S, _, rstd2 = mt.add_rmsnorm_forward(X, R, g)
    _, rstd_r = mt.rmsnorm_forward(X, g)
    W = (torch.randn(D, 1024, device=dev) / 64).half()
    xg = X[:4].contiguous()
    stream = torch.cuda.current_stream().cuda_stream

    def grads():
        return torch.empty_like(X), torch.empty(D, device=dev), torch.empty(D, device=dev)

    def rms(lib):
        dX, dg, _ = grads()
        st = lib.mt_rmsnorm_backward(_p(X), _p(g), _p(dY), _p(rstd_r), _p(dX), _p(dg), N, D,
                                     stream)
        return st, (dX, dg)

    def layer(lib):
        dX, dg, db = grads()
        st = lib.mt_layernorm_backward(_p(X), _p(g), _p(dY), _p(mean), _p(rstd), _p(dX), _p(dg),
                                       _p(db), N, D, stream)
        return st, (dX, dg, db)

    def add(lib):
        dX, dg, _ = grads()
        st = lib.mt_add_rmsnorm_backward(_p(S), _p(g), _p(dY), _p(dY), _p(rstd2), _p(dX), _p(dg),
                                         N, D, stream)
        return st, (dX, dg)

    def ex(lib):
        dX, dg, _ = grads()
        st = lib.mt_norm_backward_ex(mt.MT_OP_RMSNORM, mt.MT_DTYPE_F16, mt.MT_DTYPE_F16,
                                     mt.MT_DTYPE_F16, _p(X), _p(g), _p(dY), None, None,
                                     _p(rstd_r), _p(dX), _p(dg), None, N, D, None, 0, stream)
        return st, (dX, dg)

    def noalloc(lib):
        dX, dg, _ = grads()
        st = lib.mt_rmsnorm_backward_noalloc(_p(X), _p(g), _p(dY), _p(rstd_r), _p(dX), _p(dg),
                                             N, D, stream)
        return st, (dX, dg)

    def gemv(lib):
        yg = torch.empty(4, 1024, dtype=torch.float16, device=dev)
        st = lib.mt_fused_rmsnorm_gemv(_p(xg), _p(g), _p(W), _p(yg), 4, 1024, D, 1e-5, stream)
        return st, (yg,)

    calls = dict(rms=rms, layer=layer, add=add, ex=ex, noalloc=noalloc, gemv=gemv)
    torch.cuda.synchronize()
    before = _pool_used(h)
    for name, call in calls.items():
        h.mt_test_fail_launch(skip, ERR)
        st, _ = call(h)
        assert st == mt.MT_ERR_CUDA, name
        assert h.mt_last_cuda_error() == ERR, name
        assert h.mt_test_failure_armed() == 0, name
        torch.cuda.synchronize()
        assert _pool_used(h) == before, f"{name}: scratch not freed after a failed launch"
    # unarmed: the hook library computes exactly what the product library does
    for name, call in calls.items():
        st_h, got = call(h)
        st_p, want = call(prod)
        torch.cuda.synchronize()
        assert st_h == mt.MT_OK and st_p == mt.MT_OK, name
        for a_, b_ in zip(got, want):
            assert torch.equal(a_, b_), name
    assert _pool_used(h) == before
