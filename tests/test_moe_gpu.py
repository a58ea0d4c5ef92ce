"""Routed-expert FFN and top-k softmax router on the GPU against the oracle.

y tolerance: the per-matvec bound 1e-4 * sum|w x| + 1e-6 carried through
silu (|silu'| <= 1.1) and the down projection (computed by the oracle).
Router: the selected indices are compared exactly; the gates within 2e-6
relative (fp32 exp vs the oracle's fp64)."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_quantized_weight_q6_gb300 as qmm  # noqa: E402


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def x_tensor(x):
    return dev(x.view(np.int16)).view(torch.bfloat16) if x.dtype == np.uint16 else dev(x)


def route(logits_np, k):
    T, E = logits_np.shape
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    qmm.route_topk_softmax(dev(logits_np), k, idx, gate)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), gate.cpu().numpy()


@pytest.mark.parametrize("T,E,k", [(16, 256, 8), (1, 256, 8), (5, 64, 6), (3, 1, 1), (2, 40, 32),
                                   (4, 1024, 32)])
def test_route_matches_oracle(T, E, k):
    logits = synth.normal_f32(700 + E, (T, E))
    if E >= 16:
        logits[0, 3] = logits[0, 11] = 50.0   # a tie at the top: lower index first
        logits[T - 1, 7] = logits[T - 1, 2]    # a tie somewhere
    idx, gate = route(logits, k)
    ridx, rgate = oracle.route_topk_softmax(logits, k)
    assert np.array_equal(idx, ridx)
    assert np.allclose(gate, rgate, rtol=2e-6, atol=1e-7)
    if E >= 16:
        assert list(idx[0, :2]) == [3, 11]


def run_moe(fmt, wg, wu, wd, H, I, idx, gate, x):
    T, k = idx.shape
    m = qmm.moe_experts(wg, wu, wd, H, I, k, T)
    y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    qmm.moe(fmt, m, dev(idx.astype(np.int32)), dev(gate.astype(np.float32)), x_tensor(x), y)
    torch.cuda.synchronize()
    qmm.sync_check()
    return y.cpu().numpy()


SMALL = [(synth.Q4_0, 8, 256, 128), (synth.Q6_K, 6, 512, 256), (synth.Q8_0, 5, 128, 64)]


@pytest.mark.parametrize("fmt,E,H,I", SMALL)
@pytest.mark.parametrize("T,k", [(1, 1), (1, 4), (5, 2), (16, 4)])
def test_moe_small_vs_oracle(fmt, E, H, I, T, k):
    wg = [synth.matrix(fmt, 800 + e, I, H) for e in range(E)]
    wu = [synth.matrix(fmt, 820 + e, I, H) for e in range(E)]
    wd = [synth.matrix(fmt, 840 + e, H, I) for e in range(E)]
    x = synth.normal_bf16(850 + T, (T, H))
    logits = synth.normal_f32(851 + T, (T, E))
    idx, gate = oracle.route_topk_softmax(logits, k)
    y = run_moe(fmt, [dev(w) for w in wg], [dev(w) for w in wu], [dev(w) for w in wd], H, I, idx,
                gate.astype(np.float32), x)
    ref, bound = oracle.moe_float(fmt, H, I, wg, wu, wd, idx, gate.astype(np.float32).astype(np.float64), x)
    err = np.abs(y.astype(np.float64) - ref)
    assert (err <= bound).all(), (err / bound).max()


@pytest.mark.parametrize("fmt,E,H,I", SMALL)
@pytest.mark.parametrize("T,k", [(1, 4), (16, 4)])
def test_moe_small_vs_oracle_outputs_of_order_one(fmt, E, H, I, T, k):
    """activations N(0,1) * 1000: with the synthetic scales the outputs are
    then of order 1, so the relative part of the propagated bound (not its
    1e-6 floor) is what the comparison tests"""
    wg = [synth.matrix(fmt, 800 + e, I, H) for e in range(E)]
    wu = [synth.matrix(fmt, 820 + e, I, H) for e in range(E)]
    wd = [synth.matrix(fmt, 840 + e, H, I) for e in range(E)]
    x = synth.to_bf16_bits(synth.normal_f32(860 + T, (T, H)) * 1000.0)
    logits = synth.normal_f32(861 + T, (T, E))
    idx, gate = oracle.route_topk_softmax(logits, k)
    y = run_moe(fmt, [dev(w) for w in wg], [dev(w) for w in wu], [dev(w) for w in wd], H, I, idx,
                gate.astype(np.float32), x)
    ref, bound = oracle.moe_float(fmt, H, I, wg, wu, wd, idx, gate.astype(np.float32).astype(np.float64), x)
    assert np.abs(ref).max() > 1.0 and bound.min() > 1e-4  # the 1e-6 floor is under 1% of every bound
    err = np.abs(y.astype(np.float64) - ref)
    assert (err <= bound).all(), (err / bound).max()


def test_moe_all_tokens_on_one_expert():
    """one expert chosen by every token (tasks of 2 tokens, odd tail)"""
    fmt, E, H, I, T = synth.Q4_0, 4, 256, 128, 7
    wg = [synth.matrix(fmt, 860 + e, I, H) for e in range(E)]
    wu = [synth.matrix(fmt, 870 + e, I, H) for e in range(E)]
    wd = [synth.matrix(fmt, 880 + e, H, I) for e in range(E)]
    x = synth.normal_f32(890, (T, H))
    idx = np.full((T, 2), 2, np.int32)
    idx[:, 1] = 0
    gate = np.tile(np.array([[0.75, 0.25]], np.float32), (T, 1))
    y = run_moe(fmt, [dev(w) for w in wg], [dev(w) for w in wu], [dev(w) for w in wd], H, I, idx, gate, x)
    ref, bound = oracle.moe_float(fmt, H, I, wg, wu, wd, idx, gate.astype(np.float64), x)
    assert (np.abs(y - ref) <= bound).all()


@pytest.fixture(scope="module")
def full_experts():
    """256 Q4_0 experts, hidden 7168, intermediate 2048, resident on the GPU"""
    E, H, I = 256, 7168, 2048
    g = synth.matrix_torch(synth.Q4_0, synth.workload_seed(3, 0), I, H, "cuda", E)
    u = synth.matrix_torch(synth.Q4_0, synth.workload_seed(3, 1), I, H, "cuda", E)
    d = synth.matrix_torch(synth.Q4_0, synth.workload_seed(3, 2), H, I, "cuda", E)
    yield E, H, I, g, u, d
    del g, u, d
    torch.cuda.empty_cache()


def test_moe_full_size_one_token_vs_oracle(full_experts):
    E, H, I, g, u, d = full_experts
    x = synth.normal_bf16(synth.workload_seed(3, 3), (1, H))
    logits = synth.normal_f32(synth.workload_seed(3, 4), (1, E))
    idx, gate = route(logits, 8)
    y = run_moe(synth.Q4_0, list(g), list(u), list(d), H, I, idx, gate, x)
    sel = set(idx.ravel().tolist())
    dummy = np.zeros(18, np.uint8)
    wg = [g[e].cpu().numpy() if e in sel else dummy for e in range(E)]
    wu = [u[e].cpu().numpy() if e in sel else dummy for e in range(E)]
    wd = [d[e].cpu().numpy() if e in sel else dummy for e in range(E)]
    ref, bound = oracle.moe_float(synth.Q4_0, H, I, wg, wu, wd, idx, gate.astype(np.float64), x)
    assert (np.abs(y - ref) <= bound).all()


def test_moe_full_size_tokens_are_independent(full_experts):
    """16 tokens routed together give, token for token, bitwise the result of
    routing each token alone (grouping by expert changes no arithmetic)"""
    E, H, I, g, u, d = full_experts
    T = 16
    x = synth.normal_bf16(synth.workload_seed(3, 5), (T, H))
    logits = synth.normal_f32(synth.workload_seed(3, 6), (T, E))
    idx, gate = route(logits, 8)
    y = run_moe(synth.Q4_0, list(g), list(u), list(d), H, I, idx, gate, x)
    for t in (0, 9, 15):
        yt = run_moe(synth.Q4_0, list(g), list(u), list(d), H, I, idx[t:t + 1], gate[t:t + 1],
                     x[t:t + 1])
        assert np.array_equal(yt[0].view(np.uint32), y[t].view(np.uint32))
    assert np.isfinite(y).all()


def test_moe_liveness_and_bad_index_flag():
    fmt, E, H, I = synth.Q4_0, 4, 128, 64
    ws = [dev(synth.matrix(fmt, 900 + e, I, H)) for e in range(E)]
    wd = [dev(synth.matrix(fmt, 910 + e, H, I)) for e in range(E)]
    x = synth.normal_f32(920, (2, H))
    qmm.liveness_reset()
    idx, gate = route(synth.normal_f32(921, (2, E)), 2)
    run_moe(fmt, ws, ws, wd, H, I, idx, gate, x)
    live = qmm.liveness()
    assert live["route"] == 1 and live["moe_gate_up"] == 1 and live["moe_down"] == 1
    assert live["moe_combine"] == 1 and live["moe_plan"] == 1 and live["moe_gather"] == 1
    # an expert index out of range is flagged on the device and contributes 0
    bad = idx.copy()
    bad[0, 0] = E + 3
    m = qmm.moe_experts(ws, ws, wd, H, I, 2, 2)
    y = torch.empty((2, H), dtype=torch.float32, device="cuda")
    qmm.moe(fmt, m, dev(bad), dev(gate), x_tensor(x), y)
    torch.cuda.synchronize()
    with pytest.raises(qmm.QmmError):
        qmm.sync_check()


# Expert tables at one fixed stride (experts drawn as one tensor, as an
# engine allocates them): the expert matvecs run on the warp-level MMA
# (fp16 operands; h as two fp16 terms). All three formats; tokens that share
# experts (tasks of up to 4 tokens, an expert with more than 4 tokens), T=1.
def _table(fmt, seed, N, K, E):
    return synth.matrix_torch(fmt, seed, N, K, "cuda", E)


@pytest.mark.parametrize("fmt,E,H,I", [(synth.Q4_0, 8, 512, 256), (synth.Q6_K, 6, 512, 768),
                                       (synth.Q8_0, 5, 256, 512)])
@pytest.mark.parametrize("T,k", [(1, 1), (1, 4), (5, 2), (16, 4), (9, 3)])
def test_moe_strided_tables_vs_oracle(fmt, E, H, I, T, k):
    g, u, d = _table(fmt, 1500, I, H, E), _table(fmt, 1501, I, H, E), _table(fmt, 1502, H, I, E)
    x = synth.normal_bf16(1503 + T, (T, H))
    logits = synth.normal_f32(1504 + T, (T, E))
    idx, gate = oracle.route_topk_softmax(logits, k)
    qmm.liveness_reset()
    y = run_moe(fmt, list(g), list(u), list(d), H, I, idx, gate.astype(np.float32), x)
    live = qmm.liveness()
    assert live["moe_silu"] == 1 and live["moe_gate_up"] == 1 and live["moe_down"] == 1
    ref, bound = oracle.moe_float(fmt, H, I, [w.cpu().numpy() for w in g], [w.cpu().numpy() for w in u],
                                  [w.cpu().numpy() for w in d], idx, gate.astype(np.float32).astype(np.float64), x)
    err = np.abs(y.astype(np.float64) - ref)
    assert (err <= bound).all(), (err / bound).max()


def test_moe_strided_one_expert_many_tokens():
    """every token picks expert 2 and then expert 0: tasks of 4, 4, 3 tokens
    per expert (11 tokens)"""
    fmt, E, H, I, T = synth.Q4_0, 4, 256, 512, 11
    g, u, d = _table(fmt, 1510, I, H, E), _table(fmt, 1511, I, H, E), _table(fmt, 1512, H, I, E)
    x = synth.normal_bf16(1513, (T, H))
    idx = np.full((T, 2), 2, np.int32)
    idx[:, 1] = 0
    gate = np.tile(np.array([[0.75, 0.25]], np.float32), (T, 1))
    y = run_moe(fmt, list(g), list(u), list(d), H, I, idx, gate, x)
    ref, bound = oracle.moe_float(fmt, H, I, [w.cpu().numpy() for w in g], [w.cpu().numpy() for w in u],
                                  [w.cpu().numpy() for w in d], idx, gate.astype(np.float64), x)
    assert (np.abs(y - ref) <= bound).all()


def test_moe_strided_matches_cuda_core_path():
    """the same call with QMM_MOE_MMA=0 (CUDA-core expert matvec) agrees
    within twice the bound, in a fresh process"""
    import os
    import subprocess
    import sys
    code = r"""
import numpy as np, torch, sys
sys.path.insert(0, {root!r})
import block_quantized_weight_q6_gb300 as qmm, synth, oracle
E, H, I, T, k = 6, 512, 256, 3, 2
g = synth.matrix_torch(synth.Q4_0, 1, I, H, "cuda", E)
u = synth.matrix_torch(synth.Q4_0, 2, I, H, "cuda", E)
d = synth.matrix_torch(synth.Q4_0, 3, H, I, "cuda", E)
x = torch.from_numpy(synth.normal_bf16(4, (T, H)).view(np.int16)).cuda().view(torch.bfloat16)
idx, gate = oracle.route_topk_softmax(synth.normal_f32(5, (T, E)), k)
m = qmm.moe_experts(list(g), list(u), list(d), H, I, k, T)
y = torch.empty((T, H), device="cuda")
qmm.liveness_reset()
qmm.moe(qmm.Q4_0, m, torch.from_numpy(idx).cuda(), torch.from_numpy(gate.astype(np.float32)).cuda(), x, y)
torch.cuda.synchronize()
print(qmm.liveness()["moe_silu"])
np.save(sys.argv[1], y.cpu().numpy())
"""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    import tempfile
    outs = []
    for flag in ("1", "0"):
        f = tempfile.mktemp(suffix=".npy")
        r = subprocess.run([sys.executable, "-c", code.format(root=root), f],
                           env=dict(os.environ, QMM_MOE_MMA=flag), capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr
        assert r.stdout.split()[-1] == ("1" if flag == "1" else "0")
        outs.append(np.load(f))
        os.unlink(f)
    scale = np.abs(outs[1]).max()
    assert np.allclose(outs[0], outs[1], rtol=1e-4, atol=1e-4 * scale)
