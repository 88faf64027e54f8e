"""The GEMV planner's K split across a thread-block cluster (qg_tune_gemv_split): every cluster size
the planner can choose, forced on the shapes where it applies, against the fp64 oracle; results
repeat bit for bit; outputs stay inside their guard regions.  The split changes the order in which
a row's partial sums are added, so split and unsplit results differ in rounding only."""
import numpy as np
import pytest

import oracle
from conftest import ABS, ORACLE_THREADS, REL, Guarded, assert_within, assert_within_bound, swiglu_bound
from moe_int4_affine_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture
def split(qg):
    def set_(k):
        qg.qg_tune_gemv_split(k)
    yield set_
    qg.qg_tune_gemv_split(0)


@pytest.mark.parametrize("kcl", [1, 2, 3, 4])
@pytest.mark.parametrize("out,in_dim,xkind", [(5120, 17408, "bf16"), (5120, 17408, "f32"), (1000, 4160, "bf16"),
                                              (129, 2112, "f32"), (3, 8192, "bf16"), (2048, 6144, "f32")])
def test_split_qgemv(qg, split, kcl, out, in_dim, xkind):
    d = I.int4_weight(out + kcl, I.TID_W, out, in_dim)
    x = I.bf16_normal(out, I.TID_X, in_dim) if xkind == "bf16" else I.f32_normal(out, I.TID_X, in_dim)
    split(kcl)
    W = qg.Int4Weight.from_numpy(d)
    xd = qg.to_device(x)
    import torch

    yb = Guarded(out, torch.float32)
    prev = qg.qg_set_pdl(True)
    try:
        qg.qgemv_int4(W, xd, y=yb.t)
        y2 = qg.to_numpy(qg.qgemv_int4(W, xd))
    finally:
        qg.qg_set_pdl(prev)
    torch.cuda.synchronize()
    assert yb.intact()
    y = qg.to_numpy(yb.t)
    np.testing.assert_array_equal(y, y2)  # deterministic
    y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x, threads=ORACLE_THREADS)
    assert_within_bound(y.astype(np.float64), y_ref, a)
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("kcl", [2, 3, 4])
def test_split_multi_and_pair(qg, split, kcl):
    """Four projections sharing x of 8192 (four chunks of K), and the gate/up SwiGLU pair at
    17408 x 5120 (three chunks)."""
    split(kcl)
    outs = (4096, 1000, 32, 7)
    ds = [I.int4_weight(kcl, I.TID_MULTI + i, o, 8192) for i, o in enumerate(outs)]
    x = I.bf16_normal(kcl, I.TID_X, 8192)
    ys = qg.qgemv_int4_multi([qg.Int4Weight.from_numpy(d) for d in ds], qg.to_device(x))
    for d, y in zip(ds, ys):
        y_ref, a = oracle.qgemv(d["packed"], d["scales"], d["biases"], x, threads=ORACLE_THREADS)
        assert_within_bound(qg.to_numpy(y).astype(np.float64), y_ref, a)
    gd, ud = I.int4_weight(0, I.TID_GATE, 17408, 5120), I.int4_weight(0, I.TID_UP, 17408, 5120)
    x = I.bf16_normal(0, I.TID_X, 5120)
    h = qg.qgemv_int4_multi([qg.Int4Weight.from_numpy(gd), qg.Int4Weight.from_numpy(ud)], qg.to_device(x),
                            epilogue="swiglu")
    g, ag = oracle.qgemv(gd["packed"], gd["scales"], gd["biases"], x, threads=ORACLE_THREADS)
    u, au = oracle.qgemv(ud["packed"], ud["scales"], ud["biases"], x, threads=ORACLE_THREADS)
    assert_within(qg.to_numpy(h).astype(np.float64), oracle.swiglu(g, u),
                  swiglu_bound(g, u, REL * ag + ABS, REL * au + ABS))
    assert qg.qg_device_status() == 0


@pytest.mark.parametrize("kcl", [2, 3])
@pytest.mark.parametrize("bits", [4, 2])
def test_split_moe(qg, split, kcl, bits):
    """The MoE step (128 experts, hidden 2048, intermediate 768, top 8): the down projection's
    eight 768-column segments (three chunks of K) split across the cluster."""
    split(kcl)
    E, hidden, inter, k = 128, 2048, 768, 8
    gen = I.int4_weight if bits == 4 else I.int2_weight
    gate, up = gen(kcl, I.TID_GATE, inter, hidden, n_mat=E), gen(kcl, I.TID_UP, inter, hidden, n_mat=E)
    down = gen(kcl, I.TID_DOWN, hidden, inter, n_mat=E)
    logits = I.f32_normal(kcl, I.TID_LOGITS, E)
    x, r = I.bf16_normal(kcl, I.TID_X, hidden), I.bf16_normal(kcl, I.TID_RESID, hidden)
    t = qg.to_device

    def W(d, out, in_dim):
        return qg.Int4Weight(t(d["packed"]), t(d["scales"]), t(d["biases"]), out, in_dim, n_mat=E, bits=bits)

    G, U, D = W(gate, inter, hidden), W(up, inter, hidden), W(down, hidden, inter)
    y, idx, p = qg.moe_layer_int4(t(logits), G, U, D, t(x), t(r), k=k, bits=bits)
    i_ref, p_ref = oracle.router_topk(logits, k)
    assert qg.to_numpy(idx).astype(np.uint32).tolist() == i_ref.tolist()
    tt = lambda d: (d["packed"], d["scales"], d["biases"])  # noqa: E731
    fn = oracle.moe if bits == 4 else oracle.moe2
    y_ref, a, _ = fn(tt(gate), tt(up), tt(down), i_ref, p_ref, x, r)
    g1 = oracle.qgemv if bits == 4 else oracle.qgemv2
    gdx = oracle.qgemv_f64x if bits == 4 else oracle.qgemv2_f64x
    extra = np.zeros_like(a)
    for s_, e in enumerate(i_ref.tolist()):
        ex = lambda d: tuple(np.ascontiguousarray(v[e]) for v in tt(d))  # noqa: E731
        gr, ag = g1(*ex(gate), x)
        ur, au = g1(*ex(up), x)
        _, dab = gdx(*ex(down), swiglu_bound(gr, ur, REL * ag + ABS, REL * au + ABS))
        extra += abs(p_ref[s_]) * dab
    assert_within(qg.to_numpy(y).astype(np.float64), y_ref, REL * (a + extra) + ABS + extra)
    assert qg.qg_device_status() == 0


def test_split_refused_values(qg):
    with pytest.raises(qg.QGError):
        qg.qg_tune_gemv_split(5)
    with pytest.raises(qg.QGError):
        qg.qg_tune_gemv_split(-1)
