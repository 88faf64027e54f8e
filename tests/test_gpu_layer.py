"""GPU parity of dense_layer_int4 (gate/up SwiGLU pair, then the down projection, in one call)
against the fp64 oracle and against the same layer made of separate calls, and of the two ways
the GEMV kernel brings x on chip (one bulk copy for x of up to 128 groups, the threads' own loads
beyond) at the boundary between them."""
import numpy as np
import pytest

import oracle
from conftest import Guarded, assert_within, assert_within_bound, dense_layer_reference
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _dense(hidden, inter, out, seed=0):
    g = I.int4_weight(seed, I.TID_GATE, inter, hidden)
    u = I.int4_weight(seed, I.TID_UP, inter, hidden)
    d = I.int4_weight(seed, I.TID_DOWN, out, inter)
    return g, u, d


@pytest.fixture(scope="module")
def dense_full():
    """The dense decode layer at full size: hidden 5120, FFN 17408."""
    return _dense(5120, 17408, 5120)


def _run_dense(qg, ws, x):
    """dense_layer_int4 with y and the workspace (h) guarded on both sides; returns y, h."""
    import torch

    G, U, D = (qg.Int4Weight.from_numpy(w) for w in ws)
    wsb = Guarded(qg.qg_workspace_bytes(qg.QG_OP_LAYER, D, 0), torch.uint8)
    yb = Guarded(D.out, torch.float32)
    qg.dense_layer_int4(G, U, D, qg.to_device(x), y=yb.t, workspace=wsb.t)
    torch.cuda.synchronize()
    assert wsb.intact() and yb.intact(), "a kernel wrote outside y or the workspace"
    h = qg.to_numpy(wsb.t[:4 * D.in_dim].view(torch.float32)).astype(np.float64)
    return qg.to_numpy(yb.t).astype(np.float64), h


def _check_dense(ws, x, y, h):
    """End to end against the oracle's fp64 chain x -> g, u -> h (fp64) -> y: every row of h and of
    y, y within the bound propagated through SwiGLU and the down projection (conftest)."""
    y_ref, y_bound, h_ref, h_bound = dense_layer_reference(*ws, x)
    assert_within(h, h_ref, h_bound, what="h")
    assert_within(y, y_ref, y_bound, what="y")


@pytest.mark.parametrize("hidden,inter,out", [(128, 64, 128), (576, 192, 576), (1024, 4160, 700), (2048, 2048, 64)])
def test_dense_layer_small_shapes(qg, hidden, inter, out):
    ws = _dense(hidden, inter, out, seed=hidden + inter)
    x = I.bf16_normal(hidden, I.TID_X, hidden)
    y, h = _run_dense(qg, ws, x)
    _check_dense(ws, x, y, h)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("xkind", ["bf16", "f32"])
def test_dense_layer_full_size(qg, dense_full, xkind):
    """hidden 5120, FFN 17408, in the launch configuration the benchmark times (PDL on): all 17408
    rows of h and all 5120 rows of y against the fp64 chain."""
    x = I.bf16_normal(0, I.TID_X, 5120) if xkind == "bf16" else I.f32_normal(0, I.TID_X, 5120)
    prev = qg.qg_set_pdl(True)
    try:
        y, h = _run_dense(qg, dense_full, x)
    finally:
        qg.qg_set_pdl(prev)
    _check_dense(dense_full, x, y, h)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("xkind", ["bf16", "f32"])
def test_dense_layer_equals_separate_calls(qg, dense_full, xkind):
    x = I.bf16_normal(1, I.TID_X, 5120) if xkind == "bf16" else I.f32_normal(1, I.TID_X, 5120)
    y1, h1 = _run_dense(qg, dense_full, x)
    G, U, D = (qg.Int4Weight.from_numpy(w) for w in dense_full)
    h2 = qg.qgemv_int4_multi([G, U], qg.to_device(x), epilogue="swiglu")
    y2 = qg.qgemv_int4(D, h2)
    np.testing.assert_array_equal(h1, qg.to_numpy(h2).astype(np.float64))
    np.testing.assert_array_equal(y1, qg.to_numpy(y2).astype(np.float64))
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("in_dim", [8192, 8256])
@pytest.mark.parametrize("xkind", ["bf16", "f32"])
def test_x_staging_boundary(qg, in_dim, xkind):
    """x of 128 groups arrives by bulk copy, of 129 groups by the threads' loads: both within the
    bound, with PDL on as well as off."""
    d = I.int4_weight(9, I.TID_W, 1000, in_dim)
    x = I.bf16_normal(9, I.TID_X, in_dim) if xkind == "bf16" else I.f32_normal(9, I.TID_X, in_dim)
    w = qg.Int4Weight.from_numpy(d)
    xd = qg.to_device(x)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x)
    for pdl in (False, True):
        prev = qg.qg_set_pdl(pdl)
        try:
            y = qg.to_numpy(qg.qgemv_int4(w, xd)).astype(np.float64)
        finally:
            qg.qg_set_pdl(prev)
        assert_within_bound(y, y_ref, a, what=f"pdl={pdl}")
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("xkind", ["bf16", "f32"])
def test_dense_layer_host_buffers(qg, xkind):
    """dense_layer_int4_host (x read from and y written to page-locked host memory by the kernels)
    gives bit for bit the device-buffer call's y, over repeated calls with changing x and PDL on."""
    import torch

    ws = _dense(2048, 4096, 2048, seed=11)
    G, U, D = (qg.Int4Weight.from_numpy(w) for w in ws)
    xs = [I.bf16_normal(s, I.TID_X, 2048) if xkind == "bf16" else I.f32_normal(s, I.TID_X, 2048) for s in (11, 12)]
    y_host = torch.empty(2048, dtype=torch.float32).pin_memory()
    wsp = torch.empty(qg.qg_workspace_bytes(qg.QG_OP_LAYER_HOST, D, 2048), dtype=torch.uint8, device="cuda")
    prev = qg.qg_set_pdl(True)
    try:
        for i in range(6):
            x = xs[i % 2]
            x_host = qg.to_device(x, "cpu").pin_memory()
            qg.dense_layer_int4_host(G, U, D, x_host, y_host, workspace=wsp)
            torch.cuda.synchronize()
            y_dev = qg.dense_layer_int4(G, U, D, qg.to_device(x))
            np.testing.assert_array_equal(y_host.numpy(), qg.to_numpy(y_dev))
    finally:
        qg.qg_set_pdl(prev)
    y_ref, y_bound, _, _ = dense_layer_reference(*ws, xs[(6 - 1) % 2])
    assert_within(y_host.numpy().astype(np.float64), y_ref, y_bound)
    assert qg.qg_device_status() == 0


def test_dense_layer_host_rejects_pageable_memory(qg):
    """Pageable host tensors are refused before any launch (QG_EINVAL)."""
    import torch

    ws = _dense(128, 64, 128, seed=13)
    G, U, D = (qg.Int4Weight.from_numpy(w) for w in ws)
    x_host = qg.to_device(I.bf16_normal(13, I.TID_X, 128), "cpu")  # not pinned
    y_host = torch.empty(128, dtype=torch.float32).pin_memory()
    with pytest.raises(qg.QGError) as e:
        qg.dense_layer_int4_host(G, U, D, x_host, y_host)
    assert e.value.code == qg.QG_EINVAL
    x_pinned = x_host.pin_memory()
    with pytest.raises(qg.QGError) as e:
        qg.dense_layer_int4_host(G, U, D, x_pinned, torch.empty(128, dtype=torch.float32))
    assert e.value.code == qg.QG_EINVAL
    assert qg.qg_device_status() == 0
