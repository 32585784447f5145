"""The backward's scratch needs no clearing, and separate scratch on separate streams works.

The vectorised backward writes each CTA's dgamma (and dbeta) partial row into the scratch
before the fixed-order reduction reads it, so whatever the scratch held before must not
matter. These tests fill it with zeros, all-ones bytes, random bytes and an earlier call's
leftovers and require the allocating form's results bit for bit each time; then run two
backwards on two streams at once, each with its own scratch. The device's wait-error
word must stay 0 throughout (the split-row case exchanges row sums between the CTAs of a
cluster with bounded waits).
"""
import pytest
import torch

import row_wise_rmsnorm_gb300 as mt

DEV = "cuda:0"

# (op, N, D): one row group per CTA and several, one- and two-array partials, split rows
# (2- and 4-CTA clusters: one partial row per cluster) and many small rows.
CASES = [("rms", 600, 4096), ("layer", 300, 16384), ("add", 400, 2048),
         ("rms", 200, 24576), ("layer", 5000, 512), ("add", 64, 65536)]


def _inputs(op, N, D, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    X = torch.randn(N, D, generator=g).half().to(DEV)
    dY = torch.randn(N, D, generator=g).half().to(DEV)
    dS = torch.randn(N, D, generator=g).half().to(DEV)
    gamma = (1 + 0.1 * torch.randn(D, generator=g)).half().to(DEV)
    beta = (0.1 * torch.randn(D, generator=g)).half().to(DEV)
    if op == "layer":
        _, mean, rstd = mt.layernorm_forward(X, gamma, beta)
        return dict(X=X, dY=dY, gamma=gamma, mean=mean, rstd=rstd)
    _, rstd = mt.rmsnorm_forward(X, gamma)
    return dict(X=X, dY=dY, dS=dS, gamma=gamma, rstd=rstd)


def _code(op):
    return {"rms": mt.MT_OP_RMSNORM, "layer": mt.MT_OP_LAYERNORM, "add": mt.MT_OP_ADD_RMSNORM}[op]


def _run(op, t, ws=None, stream=None):
    """The backward with the given scratch (None: the allocating form)."""
    N, D = t["X"].shape
    dX = torch.empty_like(t["X"])
    dg = torch.empty(D, dtype=torch.float32, device=DEV)
    db = torch.empty(D, dtype=torch.float32, device=DEV)
    s = None if stream is None else stream.cuda_stream
    if op == "rms":
        if ws is None:
            mt.mt_rmsnorm_backward(t["X"], t["gamma"], t["dY"], t["rstd"], dX, dg, N, D, s)
        else:
            mt.mt_rmsnorm_backward_ws(t["X"], t["gamma"], t["dY"], t["rstd"], dX, dg, N, D, ws,
                                      ws.numel(), s)
        return dX, dg
    if op == "layer":
        if ws is None:
            mt.mt_layernorm_backward(t["X"], t["gamma"], t["dY"], t["mean"], t["rstd"], dX, dg, db,
                                     N, D, s)
        else:
            mt.mt_layernorm_backward_ws(t["X"], t["gamma"], t["dY"], t["mean"], t["rstd"], dX, dg,
                                        db, N, D, ws, ws.numel(), s)
        return dX, dg, db
    if ws is None:
        mt.mt_add_rmsnorm_backward(t["X"], t["gamma"], t["dY"], t["dS"], t["rstd"], dX, dg, N, D, s)
    else:
        mt.mt_add_rmsnorm_backward_ws(t["X"], t["gamma"], t["dY"], t["dS"], t["rstd"], dX, dg, N,
                                      D, ws, ws.numel(), s)
    return dX, dg


def _same(got, want, what):
    for a, b in zip(got, want):
        assert torch.equal(a, b), what


@pytest.mark.gpu
@pytest.mark.parametrize("op,N,D", CASES)
def test_scratch_contents_do_not_matter(op, N, D):
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the -m gpu tests")
    mt.mt_device_wait_errors(0, clear=True)
    t = _inputs(op, N, D, seed=N + D)
    want = _run(op, t)
    need = mt.mt_norm_backward_workspace_size(_code(op), N, D, 0)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    g = torch.Generator(device="cpu").manual_seed(7)
    fills = {
        "zeros": lambda: ws.zero_(),
        "ones": lambda: ws.fill_(0xFF),
        "random": lambda: ws.copy_(torch.randint(0, 256, (need,), generator=g, dtype=torch.uint8)),
        "leftovers": lambda: None,  # what the previous call left behind
    }
    for name, fill in fills.items():
        fill()
        got = _run(op, t, ws)
        torch.cuda.synchronize()
        _same(got, want, f"{op} {N}x{D}, scratch {name}")
    got = _run(op, t, ws)
    again = _run(op, t, ws)  # enqueued straight after, on the same scratch
    torch.cuda.synchronize()
    _same(got, want, f"{op} {N}x{D}, reused scratch")
    _same(again, want, f"{op} {N}x{D}, reused scratch twice")
    assert mt.mt_device_wait_errors(0) == 0


@pytest.mark.gpu
def test_two_streams_at_once():
    """Two backwards on two streams, each with its own scratch, enqueued before either is
    waited for: each gives what it gives alone."""
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the -m gpu tests")
    mt.mt_device_wait_errors(0, clear=True)
    ta = _inputs("rms", 4096, 4096, seed=1)
    tb = _inputs("layer", 1024, 8192, seed=2)
    want_a, want_b = _run("rms", ta), _run("layer", tb)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    wa = torch.empty(mt.mt_norm_backward_workspace_size(mt.MT_OP_RMSNORM, 4096, 4096, 0),
                     dtype=torch.uint8, device=DEV)
    wb = torch.empty(mt.mt_norm_backward_workspace_size(mt.MT_OP_LAYERNORM, 1024, 8192, 0),
                     dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(3):
        outs.append((_run("rms", ta, wa, sa), _run("layer", tb, wb, sb)))
    torch.cuda.synchronize()
    for ga, gb in outs:
        _same(ga, want_a, "rms on stream a")
        _same(gb, want_b, "layer on stream b")
    assert mt.mt_device_wait_errors(0) == 0
