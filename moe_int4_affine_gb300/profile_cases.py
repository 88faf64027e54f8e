"""Small, fixed invocations of the library's kernels for profilers (ncu) and quick timing.

    python -m moe_int4_affine_gb300.profile_cases layer      # gate/up SwiGLU pair + down, 17408 x 5120
    python -m moe_int4_affine_gb300.profile_cases down_bf16  # the M = 1 GEMV 5120 x 17408, bf16 x
    python -m moe_int4_affine_gb300.profile_cases moe        # router + MoE gather (128 experts, top 8)
    python -m moe_int4_affine_gb300.profile_cases qgemm T    # dequant-GEMM 17408 x 5120, T tokens
    python -m moe_int4_affine_gb300.profile_cases quant B K  # encode 17408 x 5120 weights (K = bf16 | f32) to B bits
    python -m moe_int4_affine_gb300.profile_cases moe_prefill T  # MoE layer for T tokens (128 experts, top 8)

Each case builds its seeded synthetic inputs (a few hundred MB at most on the device), runs the
calls three times and prints "ok <device status>".  Nothing is timed here.
"""
from __future__ import annotations

import sys


def main(argv=None) -> int:
    argv = sys.argv[1:] if argv is None else argv
    case = argv[0] if argv else "layer"
    import torch

    from . import build

    build.build()
    from . import inputs as I
    from . import qg

    reps = 3
    if case == "layer":
        g = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_GATE, 17408, 5120))
        u = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_UP, 17408, 5120))
        d = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_DOWN, 5120, 17408))
        x = qg.to_device(I.bf16_normal(0, I.TID_X, 5120))
        h = torch.empty(17408, device="cuda")
        y = torch.empty(5120, device="cuda")
        for _ in range(reps):
            qg.qgemv_int4_multi([g, u], x, [h, None], epilogue="swiglu")
            qg.qgemv_int4(d, h, y)
    elif case == "down_bf16":
        d = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_DOWN, 5120, 17408))
        x = qg.to_device(I.bf16_normal(0, I.TID_X, 17408))
        y = torch.empty(5120, device="cuda")
        for _ in range(reps):
            qg.qgemv_int4(d, x, y)
    elif case == "moe":
        g = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_GATE, 768, 2048, n_mat=128))
        u = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_UP, 768, 2048, n_mat=128))
        d = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_DOWN, 2048, 768, n_mat=128))
        x = qg.to_device(I.bf16_normal(0, I.TID_X, 2048))
        r = qg.to_device(I.bf16_normal(0, I.TID_RESID, 2048))
        for i in range(reps):
            idx, p = qg.moe_router_topk(qg.to_device(I.f32_normal(i, I.TID_LOGITS, 128)), k=8)
            qg.moe_gather_qgemv_int4(g, u, d, idx, p, x, r)
    elif case == "qgemm":
        T = int(argv[1]) if len(argv) > 1 else 256
        w = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_W, 17408, 5120))
        X = qg.to_device(I.bf16_normal(0, I.TID_X, (T, 5120)))
        for _ in range(reps):
            qg.qgemm_int4(w, X)
    elif case == "quant":
        bits = int(argv[1]) if len(argv) > 1 else 4
        kind = argv[2] if len(argv) > 2 else "bf16"
        shape = (17408, 5120)
        w = qg.to_device(I.bf16_normal(0, I.TID_W, shape) if kind == "bf16" else I.f32_normal(0, I.TID_W, shape))
        for _ in range(reps):
            qg.quantize_affine_q64a(w, bits)
    elif case == "moe_prefill":
        T = int(argv[1]) if len(argv) > 1 else 256
        g = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_GATE, 768, 2048, n_mat=128))
        u = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_UP, 768, 2048, n_mat=128))
        d = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_DOWN, 2048, 768, n_mat=128))
        X = qg.to_device(I.bf16_normal(0, I.TID_X, (T, 2048)))
        r = qg.to_device(I.bf16_normal(0, I.TID_RESID, (T, 2048)))
        for i in range(reps):
            qg.moe_prefill_int4(qg.to_device(I.f32_normal(i, I.TID_LOGITS, (T, 128))), g, u, d, X, r, k=8)
    else:
        print(f"unknown case {case!r}", file=sys.stderr)
        return 2
    torch.cuda.synchronize()
    status = qg.qg_device_status()
    print("ok", status)
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
