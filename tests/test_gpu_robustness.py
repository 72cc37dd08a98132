"""Robustness of the tensor-core and FP32 paths beyond single-call parity.

  * Concurrent calls on two streams.  The DeepGEMM essay
    "企业官网建设流程全解析" (section 6.5, stability checks) asks for calls
    issued concurrently from several streams.  Every plan with library
    scratch is covered: tuned single-CTA split-K partials and counters (per
    stream), 3xTF32 operand splits, FP32 repacked operands, next to CTA-pair
    and cluster plans that use none.  Each result is checked against the
    oracle.
  * Guard bands.  C sits inside a larger buffer whose margins hold a known
    pattern; after the call the margins must be bit-for-bit unchanged.  This
    covers the TMA stores of FP32, FP16 and BF16 C (32x32 and 32x64 boxes)
    and the padding between the matrices of a batch with stride_c > M * N.
"""
import numpy as np
import pytest

import oracle
from dense_gemm_11_gb300 import inputs
from tests.helpers import TOL_F16, TOL_F32, assert_within, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import dense_gemm_11_gb300 as g  # noqa: E402

DEV = torch.device("cuda:0")
TORCH_T = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
BITS_T = {"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16}


def _dev(x, kind="f32"):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV).to(TORCH_T[kind])


def test_two_streams_every_scratch_plan():
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    # two tuned single-CTA split-K plans (per-stream partials and counters)
    sk1 = (256, 1024, 4096)
    sk2 = (384, 768, 2048)
    table = [dict(path=g.GEMM_PATH_TC, M=sk1[0], N=sk1[1], K=sk1[2], variant=2, bn=128, splits=4),
             dict(path=g.GEMM_PATH_TC, M=sk2[0], N=sk2[1], K=sk2[2], variant=2, bn=256, splits=3)]
    d_sk1 = inputs.make(*sk1, kind="f16", dist="normal_k", seed=501, bias=True)
    d_sk2 = inputs.make(*sk2, kind="f16", dist="normal_k", seed=502, beta=0.5)
    # 3xTF32 (operand split scratch) on both streams
    d_x1 = inputs.make(512, 520, 1000, kind="f32", dist="uniform", seed=503)
    d_x2 = inputs.make(300, 640, 768, kind="f32", dist="uniform", seed=504, beta=1.5)
    # FP32 with rows that are not 16-byte aligned and >= 2e9 multiply-adds: repacked operands
    d_rp = inputs.make(1000, 1001, 2003, kind="f32", dist="normal", seed=505)
    # a CTA-pair plan and a cluster split plan (no scratch) in between
    d_pr = inputs.make(2048, 4096, 1024, kind="f16", dist="normal_k", seed=506)
    d_cl = inputs.make(16, 4096, 4096, kind="bf16", dist="normal_k", seed=507, bias=True)

    t = {}
    for name, d, kind in (("sk1", d_sk1, "f16"), ("sk2", d_sk2, "f16"), ("x1", d_x1, "f32"), ("x2", d_x2, "f32"),
                          ("rp", d_rp, "f32"), ("pr", d_pr, "f16"), ("cl", d_cl, "bf16")):
        t[name] = dict(A=_dev(d["A"], kind), B=_dev(d["B"], kind), C0=_dev(d["C"]),
                       bias=_dev(d["bias"]) if "bias" in d else None)
    outs = {name: [torch.empty_like(v["C0"]) for _ in range(3)] for name, v in t.items()}
    torch.cuda.synchronize()
    plans = {}
    try:
        g.tune_set(table)
        for it in range(3):
            for name, stream, fn, alpha, beta in (("sk1", s1, "tc", 0.5, 0.0), ("sk2", s2, "tc", 1.0, 0.5),
                                                 ("x1", s1, "x3", 1.0, 0.0), ("x2", s2, "x3", -0.5, 1.5),
                                                 ("pr", s2, "tc", 1.0, 0.0), ("rp", s1, "f32", 0.7, 0.0),
                                                 ("cl", s2, "tc", 0.5, 0.0)):
                v, C = t[name], outs[name][it]
                with torch.cuda.stream(stream):
                    C.copy_(v["C0"])  # stream-ordered before the GEMM that reads it
                if fn == "tc":
                    g.gemm_tc(v["A"], v["B"], C, alpha=alpha, beta=beta, bias=v["bias"],
                              act=1 if v["bias"] is not None else 0, stream=stream)
                elif fn == "x3":
                    g.gemm_f32_3xtf32(v["A"], v["B"], C, alpha=alpha, beta=beta, stream=stream)
                else:
                    g.gemm_f32(v["A"], v["B"], C, alpha=alpha, beta=beta, stream=stream)
                plans[name] = g.last_plan()
        torch.cuda.synchronize()
    finally:
        g.tune_set([])
    assert g.check() == g.GEMM_OK
    assert plans["sk1"].endswith("+tuned") and plans["sk2"].endswith("+tuned"), plans
    assert "repack" in plans["rp"] and "pair" in plans["pr"] and "clusterk" in plans["cl"], plans

    checks = (("sk1", d_sk1, 0.5, 0.0, 1, TOL_F16), ("sk2", d_sk2, 1.0, 0.5, 0, TOL_F16),
              ("x1", d_x1, 1.0, 0.0, 0, TOL_F32), ("x2", d_x2, -0.5, 1.5, 0, TOL_F32),
              ("pr", d_pr, 1.0, 0.0, 0, TOL_F16), ("rp", d_rp, 0.7, 0.0, 0, TOL_F32),
              ("cl", d_cl, 0.5, 0.0, 1, TOL_F16))
    for name, d, alpha, beta, act, tol in checks:
        M = d["A"].shape[0]
        rows = sample_rows(M, seed=1) if M > 512 else None
        ref, S = oracle.gemm(d["A"], d["B"], d["C"], alpha=alpha, beta=beta, bias=d.get("bias"), act=act, rows=rows)
        for it in range(3):
            got = outs[name][it].cpu().numpy()
            assert_within(got if rows is None else got[rows], ref, S, tol, f"{name} call {it} [{plans[name]}]",
                          bias=d.get("bias"))


def _banded(numel, kind, pad=4096):
    """A buffer of numel + 2 pad elements whose every element holds a
    distinct-ish bit pattern; returns (buffer, pristine copy)."""
    buf = torch.empty(numel + 2 * pad, dtype=TORCH_T[kind], device=DEV)
    bits = buf.view(BITS_T[kind])
    bits.copy_(torch.arange(bits.numel(), device=DEV, dtype=torch.int64).mul_(2654435761).remainder_(30011)
               .add_(1).to(BITS_T[kind]))
    return buf, buf.clone()


def _margins_untouched(buf, pristine, lo, hi, what):
    a, b = buf.view(BITS_T_OF[buf.dtype]), pristine.view(BITS_T_OF[buf.dtype])
    assert torch.equal(a[:lo], b[:lo]), f"{what}: the band before C was written"
    assert torch.equal(a[hi:], b[hi:]), f"{what}: the band after C was written"


BITS_T_OF = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}


@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(300, 264, 256),     # CTA pairs, ragged M and N
                                   (1000, 4000, 264),   # pairs, 64-column 16-bit stores
                                   (100, 200, 128),     # single-CTA tiles
                                   (16, 1000, 512),     # transposed small M
                                   (128, 4096, 4096)])  # cluster split-K
def test_tensor_core_guard_bands(out, M, N, K):
    d = inputs.make(M, N, K, kind="bf16", dist="normal_k", seed=M + N, beta=0.75, bias=True)
    pad = 4096
    buf, pristine = _banded(M * N, out, pad)
    C = buf[pad:pad + M * N].view(M, N)
    C0 = d["C"] if out == "f32" else oracle.round_to(out, d["C"])
    C.copy_(_dev(C0, out))
    pristine[pad:pad + M * N].copy_(C.reshape(-1))
    g.gemm_tc(_dev(d["A"], "bf16"), _dev(d["B"], "bf16"), C, alpha=0.5, beta=0.75, bias=_dev(d["bias"]), act=3)
    torch.cuda.synchronize()
    plan = g.last_plan()
    assert g.check() == g.GEMM_OK
    _margins_untouched(buf, pristine, pad, pad + M * N, f"{out} {M}x{N}x{K} [{plan}]")
    rows = sample_rows(M, seed=2) if M > 256 else None
    ref, S = oracle.gemm(d["A"], d["B"], C0, alpha=0.5, beta=0.75, bias=d["bias"], act=3, rows=rows)
    got = C.float().cpu().numpy().astype(np.float64)
    assert_within(got if rows is None else got[rows], ref, S, TOL_F16, f"{out} {M}x{N}x{K} [{plan}]", out=out,
                  bias=d["bias"])


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("batch,M,N,K,b_trans", [(3, 300, 264, 128, False), (4, 16, 520, 256, True),
                                                 (2, 1000, 136, 64, True)])
def test_batched_padding_between_matrices_untouched(out, batch, M, N, K, b_trans):
    d = inputs.make_batched(batch, M, N, K, kind="f16", seed=batch + M, beta=0.5, b_trans=b_trans)
    gap = 1000  # elements between matrices; a multiple of 8 keeps every matrix 16-byte aligned
    stride_c = M * N + gap
    pad = 4096
    buf, pristine = _banded(batch * stride_c, out, pad)
    view = buf[pad:pad + batch * stride_c].as_strided((batch, M, N), (stride_c, N, 1))
    C0 = d["C"] if out == "f32" else oracle.round_to(out, d["C"])
    view.copy_(_dev(C0, out))
    pristine.copy_(buf)
    g.gemm_tc_batched(_dev(d["A"], "f16"), _dev(d["B"], "f16"), view, alpha=1.25, beta=0.5, act=2, b_trans=b_trans)
    torch.cuda.synchronize()
    plan = g.last_plan()
    assert g.check() == g.GEMM_OK
    bits, pbits = buf.view(BITS_T_OF[buf.dtype]), pristine.view(BITS_T_OF[buf.dtype])
    _margins_untouched(buf, pristine, pad, pad + batch * stride_c - gap, f"batched {out} [{plan}]")
    for z in range(batch):
        lo = pad + z * stride_c + M * N
        assert torch.equal(bits[lo:lo + gap], pbits[lo:lo + gap]), f"padding after matrix {z} was written [{plan}]"
    got = view.float().cpu().numpy().astype(np.float64)
    for z in range(batch):
        Bz = d["B"][z].T if b_trans else d["B"][z]
        ref, S = oracle.gemm(d["A"][z], Bz, C0[z], alpha=1.25, beta=0.5, act=2)
        assert_within(got[z], ref, S, TOL_F16, f"z={z} {out} [{plan}]", out=out)
