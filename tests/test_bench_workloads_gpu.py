"""The launches bench.py times, exactly as it makes them, against the oracle.

The bench's decode part is grouped calls over the full-size 7B-shaped decode
set (batch 1 and 8); its MoE part routes 16 tokens over 256 resident experts;
its GEMM part is the q6_K ffn_down prefill in both variants. Each is built
here through bench.py's own workload classes, run once, and compared with the
CPU oracle on sampled outputs computed one by one:
|y - y_ref| <= 1e-4 * sum_k |w_k x_k| + 1e-6 (MoE: the propagated bound)."""
import os
import sys

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import block_quantized_weight_q6_gb300 as qmm  # noqa: E402

FMT = {"Q4_0": qmm.Q4_0, "Q8_0": qmm.Q8_0, "q6_K": qmm.Q6_K}


def assert_within(got, ref, absum, what):
    err = np.abs(got.astype(np.float64) - ref)
    bound = 1e-4 * absum + 1e-6
    bad = ~(err <= bound)
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} sampled outputs out of bound; "
                             f"first #{i}: got {got[i]}, ref {ref[i]}, bound {bound[i]}")


def bf16_host(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("act", ["float", "q8"])
def test_decode_set_grouped_calls_vs_oracle(act):
    """All 18 matvecs of the decode set (batch 1 and 8), run as the grouped
    calls of the bench's step; 512 sampled outputs per matvec."""
    dev = torch.device("cuda", 0)
    dec = bench.DecodeSet(torch, dev, act=qmm.ACT_Q8 if act == "q8" else qmm.ACT_FLOAT)
    dec.y_all.fill_(float("nan"))
    dec.run()
    torch.cuda.synchronize()
    qmm.sync_check()
    for i, (name, fmt, N, K, B, Wt, xt, yt) in enumerate(dec.items):
        f = FMT[fmt]
        W = Wt.cpu().numpy()
        x = bf16_host(xt)
        y = yt.cpu().numpy()
        assert np.isfinite(y).all(), f"{name} B={B}: unwritten outputs"
        rng = np.random.default_rng(1000 + i)
        bs = rng.integers(0, B, 512)
        ns = np.concatenate([rng.integers(0, N, 508), [0, N - 1, N // 2, N - 2]])
        if act == "float":
            ref, absum = oracle.gemv_float_pairs(f, W, K, x, bs, ns)
        else:
            xq, s = oracle.quantize_q8(x)
            ref, absum = oracle.gemm_q8_pairs(f, W, K, xq, s, bs, ns)
        assert_within(y[bs, ns], ref, absum, f"{name} {fmt} {N}x{K} B={B} {act}")
    del dec
    torch.cuda.empty_cache()


def test_gemm_case_both_variants_vs_oracle():
    """The q6_K ffn_down prefill (M=512) as the bench runs it: plane and
    in-kernel outputs bitwise equal, 1024 sampled outputs against the oracle."""
    dev = torch.device("cuda", 0)
    gem = bench.GemmCase(torch, dev)
    gem.Y1.fill_(float("nan"))
    gem.Y2.fill_(float("nan"))
    gem.run_exp()
    gem.run_in_kernel()
    torch.cuda.synchronize()
    qmm.sync_check()
    assert torch.equal(gem.Y1.view(torch.int32), gem.Y2.view(torch.int32))
    W = gem.W.cpu().numpy()
    xq, s = oracle.quantize_q8(bf16_host(gem.X))
    rng = np.random.default_rng(7)
    ms = np.concatenate([rng.integers(0, gem.M, 1020), [0, gem.M - 1, 0, gem.M - 1]])
    ns = np.concatenate([rng.integers(0, gem.N, 1020), [0, gem.N - 1, gem.N - 1, 0]])
    ref, absum = oracle.gemm_q8_pairs(qmm.Q6_K, W, gem.K, xq, s, ms, ns)
    assert_within(gem.Y2.cpu().numpy()[ms, ns], ref, absum, "ffn_down prefill")
    qmm.plane_release(gem.W)
    del gem
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [1, 16])
def test_moe_case_vs_oracle(T):
    """The routed-expert FFN over the 256 resident experts as the bench runs
    it (routing on the device, then the expert FFN); sampled tokens against
    the oracle's FFN over the experts each selected, and the router's indices
    against the oracle's."""
    dev = torch.device("cuda", 0)
    wts = bench.MoeWeights(torch, dev)
    case = bench.MoeCase(torch, dev, wts, T)
    case.y.fill_(float("nan"))
    case.run()
    torch.cuda.synchronize()
    qmm.sync_check()
    idx = case.idx.cpu().numpy()
    gate = case.gate.cpu().numpy()
    ridx, _ = oracle.route_topk_softmax(case.logits.cpu().numpy(), case.k)
    assert np.array_equal(idx, ridx)
    y = case.y.cpu().numpy()
    assert np.isfinite(y).all()
    x = bf16_host(case.x)
    dummy = np.zeros(18, np.uint8)
    for t in ([0] if T == 1 else [0, 6, 15]):
        sel = set(idx[t].tolist())
        wg = [wts.g[e].cpu().numpy() if e in sel else dummy for e in range(wts.E)]
        wu = [wts.u[e].cpu().numpy() if e in sel else dummy for e in range(wts.E)]
        wd = [wts.d[e].cpu().numpy() if e in sel else dummy for e in range(wts.E)]
        ref, bound = oracle.moe_float(qmm.Q4_0, wts.H, wts.I, wg, wu, wd, idx[t:t + 1],
                                      gate[t:t + 1].astype(np.float64), x[t:t + 1])
        err = np.abs(y[t].astype(np.float64) - ref[0])
        assert (err <= bound[0]).all(), f"token {t}: max err/bound {(err / bound[0]).max()}"
    del case, wts
    torch.cuda.empty_cache()
