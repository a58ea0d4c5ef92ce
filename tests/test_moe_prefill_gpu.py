"""Expert-grouped MoE prefill (moe_prefill) on the GPU against the CPU oracle.

The oracle (orc_moe_q8) computes the expert FFN with every matmul on
activations quantized per 32, as the prefill GEMM does, and re-quantizes h.
Two bounds come with it:
  tight: holds when every code of the quantized h equals the oracle's;
  loose: holds for any h within its propagated error (each code may then be
         one step off).
Every output must be within the loose bound, and nearly all (h codes that
sit on a rounding boundary are rare) within the tight one.
Activations are N(0,1) * 1000 so that the outputs are of order 1 with the
synthetic scales (d ~ 2e-4).
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only containers
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_quantized_weight_q6_gb300 as qmm  # noqa: E402


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def x_tensor(x):
    if x.dtype == np.uint16:
        return dev(x.view(np.int16)).view(torch.bfloat16)
    return dev(x)


def experts(fmt, E, H, I, seed):
    wg = [synth.matrix(fmt, seed + e, I, H) for e in range(E)]
    wu = [synth.matrix(fmt, seed + 100 + e, I, H) for e in range(E)]
    wd = [synth.matrix(fmt, seed + 200 + e, H, I) for e in range(E)]
    return wg, wu, wd


def run(fmt, wg, wu, wd, H, I, idx, gate, x):
    T, k = idx.shape
    Wg, Wu, Wd = [dev(w) for w in wg], [dev(w) for w in wu], [dev(w) for w in wd]
    m = qmm.moe_experts(Wg, Wu, Wd, H, I, k, T)
    y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    qmm.moe_prefill(fmt, m, dev(idx.astype(np.int32)), dev(gate.astype(np.float32)), x_tensor(x), y)
    torch.cuda.synchronize()
    qmm.sync_check()
    return y.cpu().numpy()


def check(y, ref, tight, loose, what, min_tight=0.95):
    err = np.abs(y.astype(np.float64) - ref)
    assert np.isfinite(y).all(), what
    assert (err <= loose).all(), (what, float((err / loose).max()))
    frac = float((err <= tight).mean())
    assert frac >= min_tight, (what, frac, float((err / tight).max()))
    return frac


def scaled_x(seed, T, H, bf16=True):
    xf = synth.normal_f32(seed, (T, H)) * 1000.0
    return synth.to_bf16_bits(xf) if bf16 else xf


CASES = [(synth.Q4_0, 6, 512, 256), (synth.Q6_K, 5, 512, 256)]


@pytest.mark.parametrize("fmt,E,H,I", CASES)
@pytest.mark.parametrize("T,k", [(1, 1), (7, 2), (64, 4), (300, 2)])
@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_moe_prefill_vs_oracle(fmt, E, H, I, T, k, xdt):
    wg, wu, wd = experts(fmt, E, H, I, 3000 + fmt * 10)
    x = scaled_x(3100 + T, T, H, xdt == "bf16")
    idx, gate = oracle.route_topk_softmax(synth.normal_f32(3200 + T, (T, E)), k)
    gate32 = gate.astype(np.float32)
    qmm.liveness_reset()
    y = run(fmt, wg, wu, wd, H, I, idx, gate32, x)
    live = qmm.liveness()
    used = len(np.unique(idx))
    assert live["moe_prefill_plan"] == 1 and live["moe_prefill_rows"] == 2 and live["moe_prefill_silu"] == 1
    gemm_slot = "gemm_q4_0" if fmt == synth.Q4_0 else "gemm_in_kernel"
    assert live[gemm_slot] == 3 * used
    ref, tight, loose = oracle.moe_q8(fmt, H, I, wg, wu, wd, idx, gate32.astype(np.float64), x)
    check(y, ref, tight, loose, f"fmt {fmt} T={T} k={k} {xdt}")
    # the order of every sum is fixed: a second call is bitwise identical
    y2 = run(fmt, wg, wu, wd, H, I, idx, gate32, x)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


def test_moe_prefill_one_expert_takes_every_token():
    """all tokens on one expert (its GEMMs span several 128-row tiles), the
    other experts unused"""
    fmt, E, H, I, T = synth.Q4_0, 4, 1024, 512, 384
    wg, wu, wd = experts(fmt, E, H, I, 3300)
    x = scaled_x(3310, T, H)
    idx = np.full((T, 1), 2, np.int32)
    gate = np.ones((T, 1), np.float32)
    y = run(fmt, wg, wu, wd, H, I, idx, gate, x)
    ref, tight, loose = oracle.moe_q8(fmt, H, I, wg, wu, wd, idx, gate.astype(np.float64), x)
    check(y, ref, tight, loose, "one expert")


def test_moe_prefill_medium_sampled_tokens():
    """64 experts, 512 tokens top-4 (about 32 tokens per expert): 6 tokens
    against the oracle (each token's output depends only on its own row)"""
    fmt, E, H, I, T, k = synth.Q4_0, 64, 2048, 1024, 512, 4
    wg = [synth.matrix(fmt, 3400 + e, I, H) for e in range(E)]
    wu = [synth.matrix(fmt, 3500 + e, I, H) for e in range(E)]
    wd = [synth.matrix(fmt, 3600 + e, H, I) for e in range(E)]
    x = scaled_x(3700, T, H)
    idx, gate = oracle.route_topk_softmax(synth.normal_f32(3701, (T, E)), k)
    gate32 = gate.astype(np.float32)
    y = run(fmt, wg, wu, wd, H, I, idx, gate32, x)
    ts = np.array([0, 1, 77, 255, 300, T - 1])
    ref, tight, loose = oracle.moe_q8(fmt, H, I, wg, wu, wd, idx[ts], gate32[ts].astype(np.float64), x[ts])
    check(y[ts], ref, tight, loose, "medium sampled")


def test_moe_prefill_bad_index_is_an_error():
    fmt, E, H, I, T = synth.Q4_0, 4, 256, 128, 5
    wg, wu, wd = experts(fmt, E, H, I, 3800)
    x = scaled_x(3810, T, H)
    idx = np.zeros((T, 2), np.int32)
    idx[:, 1] = 1
    idx[3, 1] = E  # out of range
    m = qmm.moe_experts([dev(w) for w in wg], [dev(w) for w in wu], [dev(w) for w in wd], H, I, 2, T)
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    with pytest.raises(qmm.QmmError) as ei:
        qmm.moe_prefill(fmt, m, dev(idx), dev(np.full((T, 2), 0.5, np.float32)), x_tensor(x), y)
    assert ei.value.code == qmm.EINVAL
    torch.cuda.synchronize()
    with pytest.raises(qmm.QmmError):
        qmm.sync_check()  # the device flag of the bad index, cleared by the read
    qmm.sync_check()
    # the context stays usable
    idx[3, 1] = 3
    yv = run(fmt, wg, wu, wd, H, I, idx, np.full((T, 2), 0.5, np.float32), x)
    assert np.isfinite(yv).all()
