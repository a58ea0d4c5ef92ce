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

Two flows: experts whose gate, up and down matrices each lie at one fixed
stride (one tensor per projection) go through one grouped GEMM launch per
projection over row tiles padded per expert; any other table takes one GEMM
launch per expert and projection. Both are checked against the oracle.
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


def table(ws, layout):
    """the matrices on the device: "strided" in one tensor at a fixed stride
    (a multiple of 16 bytes past the matrix), "ragged" in one tensor at
    unequal gaps, "separate" one allocation each"""
    if layout == "separate":
        return [dev(w) for w in ws]
    nb = ws[0].nbytes
    gaps = [48] * len(ws) if layout == "strided" else [16 * (e % 3) + 16 for e in range(len(ws))]
    offs = np.cumsum([0] + [nb + g for g in gaps[:-1]])
    big = torch.zeros(int(offs[-1]) + nb, dtype=torch.uint8, device="cuda")
    for o, w in zip(offs, ws):
        big[int(o):int(o) + nb] = dev(w.view(np.uint8).reshape(-1))
    return [big[int(o):int(o) + nb] for o in offs]


def run(fmt, wg, wu, wd, H, I, idx, gate, x, layout="separate", live=None):
    T, k = idx.shape
    Wg, Wu, Wd = table(wg, layout), table(wu, layout), table(wd, layout)
    m = qmm.moe_experts(Wg, Wu, Wd, H, I, k, T)
    if live is not None:
        qmm.liveness_reset()
    y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    qmm.moe_prefill(fmt, m, dev(idx.astype(np.int32)), dev(gate.astype(np.float32)), x_tensor(x), y)
    torch.cuda.synchronize()
    qmm.sync_check()
    if live is not None:
        live.update(qmm.liveness())
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
@pytest.mark.parametrize("layout", ["strided", "ragged"])
def test_moe_prefill_vs_oracle(fmt, E, H, I, T, k, xdt, layout):
    wg, wu, wd = experts(fmt, E, H, I, 3000 + fmt * 10)
    x = scaled_x(3100 + T, T, H, xdt == "bf16")
    idx, gate = oracle.route_topk_softmax(synth.normal_f32(3200 + T, (T, E)), k)
    gate32 = gate.astype(np.float32)
    live = {}
    y = run(fmt, wg, wu, wd, H, I, idx, gate32, x, layout, live)
    used = len(np.unique(idx))
    gemm_slot = "gemm_q4_0" if fmt == synth.Q4_0 else "gemm_in_kernel"
    # grouped: the plan and the padded row map; one GEMM launch per projection
    grouped = layout == "strided"
    assert live["moe_prefill_plan"] == (2 if grouped else 1)
    assert live["moe_prefill_rows"] == 2 and live["moe_prefill_silu"] == 1
    assert live[gemm_slot] == (3 if grouped else 3 * used)
    ref, tight, loose = oracle.moe_q8(fmt, H, I, wg, wu, wd, idx, gate32.astype(np.float64), x)
    check(y, ref, tight, loose, f"fmt {fmt} T={T} k={k} {xdt} {layout}")
    # the order of every sum is fixed: a second call is bitwise identical
    y2 = run(fmt, wg, wu, wd, H, I, idx, gate32, x, layout)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("fmt", [synth.Q4_0, synth.Q6_K])
def test_moe_prefill_grouped_tiles_and_empty_experts(fmt):
    """grouped flow: 8 experts, three unused, one with 300 rows (three padded
    tiles), one with exactly 128, the rest ragged; and the per-expert flow on
    the same input agrees with it within the oracle's tight bound"""
    E, H, I = 8, 512, 512
    wg, wu, wd = experts(fmt, E, H, I, 3900 + fmt)
    n = {1: 300, 2: 128, 4: 1, 5: 77, 7: 130}
    ids = np.concatenate([np.full(c, e) for e, c in n.items()])
    rng = np.random.default_rng(fmt)
    ids = rng.permutation(ids).astype(np.int32)
    T = len(ids)
    idx = ids.reshape(T, 1)
    gate = rng.uniform(0.5, 1.5, (T, 1)).astype(np.float32)
    x = scaled_x(3910 + fmt, T, H)
    live = {}
    yg = run(fmt, wg, wu, wd, H, I, idx, gate, x, "strided", live)
    assert live["moe_prefill_plan"] == 2
    yr = run(fmt, wg, wu, wd, H, I, idx, gate, x, "ragged", live)
    assert live["moe_prefill_plan"] == 1
    ref, tight, loose = oracle.moe_q8(fmt, H, I, wg, wu, wd, idx, gate.astype(np.float64), x)
    check(yg, ref, tight, loose, f"grouped fmt {fmt}")
    check(yr, ref, tight, loose, f"per expert fmt {fmt}")
    assert (np.abs(yg.astype(np.float64) - yr) <= 2 * tight).mean() >= 0.95


@pytest.mark.parametrize("layout", ["strided", "ragged"])
def test_moe_prefill_q6k_full_int8_scales(layout):
    """q6_K experts whose sub-block scales span the whole int8 range: the
    prefill GEMM's second K pass (scales beyond 56) in the grouped launch
    and in the per-expert one, against the oracle"""
    fmt, E, H, I, T, k = synth.Q6_K, 4, 512, 256, 64, 2
    wg, wu, wd = experts(fmt, E, H, I, 3950)
    rng = np.random.default_rng(3951)

    def widen(w):
        w = w.copy()
        b = w.reshape(-1, 210)
        b[:, 192:208] = rng.integers(0, 256, (b.shape[0], 16)).astype(np.uint8)
        return w

    wg, wu, wd = [widen(w) for w in wg], [widen(w) for w in wu], [widen(w) for w in wd]
    x = synth.normal_bf16(3952, (T, H))
    idx, gate = oracle.route_topk_softmax(synth.normal_f32(3953, (T, E)), k)
    gate32 = gate.astype(np.float32)
    live = {}
    y = run(fmt, wg, wu, wd, H, I, idx, gate32, x, layout, live)
    assert live["moe_prefill_plan"] == (2 if layout == "strided" else 1)
    ref, tight, loose = oracle.moe_q8(fmt, H, I, wg, wu, wd, idx, gate32.astype(np.float64), x)
    check(y, ref, tight, loose, f"q6_K int8 scales {layout}")


def test_moe_prefill_one_expert_takes_every_token():
    """all tokens on one expert (its GEMMs span several 128-row tiles), the
    other experts unused"""
    fmt, E, H, I, T = synth.Q4_0, 4, 1024, 512, 384
    wg, wu, wd = experts(fmt, E, H, I, 3300)
    x = scaled_x(3310, T, H)
    idx = np.full((T, 1), 2, np.int32)
    gate = np.ones((T, 1), np.float32)
    y = run(fmt, wg, wu, wd, H, I, idx, gate, x, "strided")
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
    y = run(fmt, wg, wu, wd, H, I, idx, gate32, x, "strided")
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
