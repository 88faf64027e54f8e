"""GPU parity of dense_layer_int4 (gate/up SwiGLU pair, then the down projection, in one call)
against the fp64 oracle and against the same layer made of separate calls, and of the two ways
the GEMV kernel brings x on chip (one bulk copy for x of up to 128 groups, the threads' own loads
beyond) at the boundary between them."""
import numpy as np
import pytest

import oracle
from conftest import assert_within_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _silu_bound(g, u, ag, au):
    """First-order propagation of the GEMV bounds on g and u into h = silu(g) * u."""
    s = 1.0 / (1.0 + np.exp(-g))
    dsilu = s * (1.0 + g * (1.0 - s))
    return np.abs(dsilu * u) * ag + np.abs(g * s) * au


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
    import torch

    G, U, D = (qg.Int4Weight.from_numpy(w) for w in ws)
    workspace = torch.empty(qg.qg_workspace_bytes(qg.QG_OP_LAYER, D, 0), dtype=torch.uint8, device="cuda")
    y = qg.dense_layer_int4(G, U, D, qg.to_device(x), workspace=workspace)
    h = qg.to_numpy(workspace[:4 * D.in_dim].view(torch.float32)).astype(np.float64)
    return qg.to_numpy(y).astype(np.float64), h


def _check_dense(ws, x, y, h, h_rows):
    g, u, d = ws
    r0, r1 = h_rows
    gr, ag = oracle.qgemv(g["packed"], g["scales"], g["biases"], x, rows=h_rows)
    ur, au = oracle.qgemv(u["packed"], u["scales"], u["biases"], x, rows=h_rows)
    h_ref = oracle.swiglu(gr, ur)
    assert_within_bound(h[r0:r1], h_ref, _silu_bound(gr, ur, ag, au) + np.abs(h_ref) * 1e-3, what="h")
    # y against the oracle's GEMV of the GPU's own h (fp32, as the kernel reads it)
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], h.astype(np.float32))
    assert_within_bound(y, y_ref, a, what="y")


@pytest.mark.parametrize("hidden,inter,out", [(128, 64, 128), (576, 192, 576), (1024, 4160, 700), (2048, 2048, 64)])
def test_dense_layer_small_shapes(qg, hidden, inter, out):
    ws = _dense(hidden, inter, out, seed=hidden + inter)
    x = I.bf16_normal(hidden, I.TID_X, hidden)
    y, h = _run_dense(qg, ws, x)
    _check_dense(ws, x, y, h, (0, inter))
    assert qg.qg_device_status() == 0


def test_dense_layer_full_size(qg, dense_full):
    """hidden 5120, FFN 17408: h on its first and last 700 rows, y on all 5120 rows."""
    x = I.bf16_normal(0, I.TID_X, 5120)
    y, h = _run_dense(qg, dense_full, x)
    _check_dense(dense_full, x, y, h, (0, 700))
    _check_dense(dense_full, x, y, h, (17408 - 700, 17408))
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
    y_ref, a = oracle.qgemv(ws[2]["packed"], ws[2]["scales"], ws[2]["biases"],
                            qg.to_numpy(wsp[:4 * 4096].view(torch.float32)))
    assert_within_bound(y_host.numpy().astype(np.float64), y_ref, a)
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
