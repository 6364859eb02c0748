"""The Muon step around NS (muon_step_ws and its per-kernel chain) on the GPU.

  * against the fp64 oracle step (oracle.muon_step): M' to fp32 rounding,
    W' to the NS tolerance on its update term, and the orthogonalised update
    itself (W = 0, so W' = -lr scale O) per matrix within the NS tolerance;
  * the fused step (momentum kernel with the norm, NS without a norm pass,
    the last update product writing W) equals muon_momentum -> muon_ns_ws on
    U -> muon_apply bit for bit, wide and tall, with both pair modes of the
    products and with the per-matrix completion counters (batch > 1);
  * step counts 0, 1 and 2, plain momentum, weight decay, argument errors;
  * the full-size expert stack on sampled matrices.
"""
import ctypes

import numpy as np
import pytest
import torch

import newton_schulz_07_gb300 as ns
import ns_inputs
import oracle
from nsutil import NS_TOL, ns_tols, per_matrix_rel

pytestmark = pytest.mark.gpu


def f32_stack(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape, dtype=np.float32) * np.float32(scale))


def run_step(W, M, G, **kw):
    Wd, Md, Gd = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (W, M, G))
    b, r, c = W.shape
    ws = torch.empty(ns.step_workspace_size(b, r, c), dtype=torch.uint8, device="cuda")
    ns.muon_step(Wd, Md, Gd, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert ns.read_error(ws) == 0
    return Wd.cpu().numpy(), Md.cpu().numpy()


def run_chain(W, M, G, lr, momentum=0.95, nesterov=True, weight_decay=0.0, scale=None, steps=5):
    Wd, Md, Gd = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (W, M, G))
    b, r, c = W.shape
    ws = ns.alloc_workspace(b, r, c)
    U = ns.muon_momentum(Md, Gd, ws, momentum=momentum, nesterov=nesterov)
    O = ns.muon_ns(U, steps=steps, workspace=ns.alloc_workspace(b, r, c))
    ns.muon_apply(Wd, O, lr, weight_decay=weight_decay, scale=scale)
    torch.cuda.synchronize()
    return Wd.cpu().numpy(), Md.cpu().numpy(), U


def u_bits(M, G, mu, nesterov):
    """bf16 bits of the oracle's NS input, for the per-shape tolerance."""
    U = oracle.round_bf16(oracle.ns_input(G, oracle.momentum_update(M, G, mu), mu, nesterov))
    return ns_inputs.fp32_to_bf16_bits(U.astype(np.float32))


@pytest.mark.parametrize("shape", [(3, 256, 512), (2, 520, 264), (1, 136, 264), (2, 1040, 1280), (1, 8, 64)])
def test_orthogonalised_update_vs_oracle(shape):
    # W = 0: W' = -lr scale O exactly up to one rounding, so O is read back.
    mu, lr = 0.9, 0.5
    M, G = f32_stack(shape, 1, 0.02), f32_stack(shape, 2, 0.02)
    W = np.zeros(shape, np.float32)
    Wn, Mn = run_step(W, M, G, lr=lr, momentum=mu)
    s = ns.default_scale(shape[1], shape[2])
    O_gpu = -Wn.astype(np.float64) / (lr * s)
    _, _, O_ref = oracle.muon_step(W, M, G, lr, mu)
    errs = per_matrix_rel(O_gpu, O_ref)
    tols = ns_tols(u_bits(M, G, mu, True))
    assert all(e <= t for e, t in zip(errs, tols)), (errs, tols)


@pytest.mark.parametrize("shape,nesterov,wd", [((2, 256, 512), True, 0.0), ((2, 512, 256), False, 0.1),
                                               ((1, 264, 392), True, 0.3)])
def test_step_vs_oracle(shape, nesterov, wd):
    mu, lr = 0.95, 0.02
    W, M, G = f32_stack(shape, 3), f32_stack(shape, 4, 0.05), f32_stack(shape, 5, 0.05)
    Wn, Mn = run_step(W, M, G, lr=lr, momentum=mu, nesterov=nesterov, weight_decay=wd)
    W_ref, M_ref, O_ref = oracle.muon_step(W, M, G, lr, mu, nesterov=nesterov, weight_decay=wd)
    # M' = fma(mu, M, G): one fp32 rounding.
    bound = 2.0 ** -23 * (np.abs(mu * M.astype(np.float64)) + np.abs(G)) + 1e-38
    assert np.all(np.abs(Mn - M_ref) <= bound)
    s = ns.default_scale(shape[1], shape[2])
    for k in range(shape[0]):
        upd = lr * s * np.linalg.norm(O_ref[k])
        err = np.linalg.norm(Wn[k] - W_ref[k])
        assert err <= NS_TOL * upd + 4 * 2.0 ** -24 * np.linalg.norm(W[k]), (k, err, upd)


@pytest.mark.parametrize("shape", [(3, 256, 512), (2, 520, 264), (1, 1040, 1280), (2, 1040, 1280),
                                   (2, 1280, 1040), (4, 136, 264)])
def test_fused_step_equals_kernel_chain_bitwise(shape):
    W, M, G = f32_stack(shape, 6), f32_stack(shape, 7, 0.05), f32_stack(shape, 8, 0.05)
    kw = dict(lr=0.01, momentum=0.9, weight_decay=0.05)
    Wf, Mf = run_step(W, M, G, **kw)
    Wc, Mc, _ = run_chain(W, M, G, **kw)
    np.testing.assert_array_equal(Mf, Mc)
    np.testing.assert_array_equal(Wf.view(np.uint32), Wc.view(np.uint32))


@pytest.mark.parametrize("steps", [0, 1, 2])
def test_step_counts_bitwise_and_vs_oracle(steps):
    shape = (2, 256, 384)
    W, M, G = f32_stack(shape, 9), f32_stack(shape, 10, 0.05), f32_stack(shape, 11, 0.05)
    kw = dict(lr=0.05, momentum=0.8, nesterov=False)
    Wf, Mf = run_step(W, M, G, steps=steps, **kw)
    Wc, Mc, _ = run_chain(W, M, G, steps=steps, **kw)
    np.testing.assert_array_equal(Wf.view(np.uint32), Wc.view(np.uint32))
    W_ref, _, O_ref = oracle.muon_step(W, M, G, 0.05, 0.8, nesterov=False, steps=steps)
    for k in range(2):
        upd = 0.05 * np.linalg.norm(O_ref[k])
        assert np.linalg.norm(Wf[k] - W_ref[k]) <= NS_TOL * upd + 4 * 2.0 ** -24 * np.linalg.norm(W[k])


def test_momentum_norm_equals_ns_norm_bitwise():
    # The momentum kernel's ||U||_F is the NS norm kernel's value on the same U.
    shape = (3, 264, 520)
    M, G = f32_stack(shape, 12, 0.05), f32_stack(shape, 13, 0.05)
    Md, Gd = torch.from_numpy(M).cuda(), torch.from_numpy(G).cuda()
    ws1, ws2 = ns.alloc_workspace(*shape), ns.alloc_workspace(*shape)
    U = ns.muon_momentum(Md, Gd, ws1, momentum=0.9)
    ns.muon_ns_normalize(U, ws2, norms_only=True)
    torch.cuda.synchronize()
    off, nb = ns.workspace_region(*shape, ns._lib.WS_NORMS)
    np.testing.assert_array_equal(ws1[off:off + nb].cpu().numpy(), ws2[off:off + nb].cpu().numpy())
    # and U is bf16(G + mu M') of the oracle, up to fp32 double rounding at ties
    ref = oracle.round_bf16(oracle.ns_input(G, oracle.momentum_update(M, G, 0.9), 0.9, True))
    got = U.float().cpu().numpy().astype(np.float64)
    assert np.mean(got != ref) < 1e-4
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref))


def test_argument_errors():
    shape = (2, 64, 128)
    W, M, G = (torch.zeros(shape, dtype=torch.float32, device="cuda") for _ in range(3))
    ws = torch.empty(ns.step_workspace_size(*shape), dtype=torch.uint8, device="cuda")
    L = ns._lib.lib()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(Wp, Mp, Gp, hp, wsb=ws.numel()):
        return L.muon_step_ws(ctypes.c_void_p(Wp), ctypes.c_void_p(Mp), ctypes.c_void_p(Gp), *shape, ctypes.byref(hp),
                              5, None, ctypes.c_float(1e-7), ctypes.c_void_p(ws.data_ptr()), wsb, st)

    good = ns._lib.MuonStepHparams(0.02, 0.95, 0.0, 1.0, 1)
    assert call(W.data_ptr(), M.data_ptr(), G.data_ptr(), good) == ns._lib.OK
    assert call(W.data_ptr(), W.data_ptr(), G.data_ptr(), good) == ns._lib.ERR_INVALID_ARG  # W and M overlap
    assert call(W.data_ptr(), M.data_ptr(), M.data_ptr(), good) == ns._lib.ERR_INVALID_ARG  # M and G overlap
    bad = ns._lib.MuonStepHparams(float("nan"), 0.95, 0.0, 1.0, 1)
    assert call(W.data_ptr(), M.data_ptr(), G.data_ptr(), bad) == ns._lib.ERR_INVALID_ARG
    assert call(W.data_ptr(), M.data_ptr(), G.data_ptr(), good, ws.numel() - 1) == ns._lib.ERR_WORKSPACE
    big = torch.zeros(3 * 64 * 128 + 4, dtype=torch.float32, device="cuda")
    assert call(big.data_ptr() + 4, M.data_ptr(), G.data_ptr(), good) == ns._lib.ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert ns.read_error(ws) == 0


def test_step_captured_in_a_graph_equals_eager_steps():
    # muon_step_ws allocates nothing and does not synchronise: two replays of a
    # captured step give the bits of two eager steps on the same state.
    shape = (3, 256, 512)
    W, M, G = f32_stack(shape, 16), f32_stack(shape, 17, 0.05), f32_stack(shape, 18, 0.05)
    kw = dict(lr=0.02, momentum=0.9, weight_decay=0.01)
    Wd, Md, Gd = (torch.from_numpy(x).cuda() for x in (W, M, G))
    ws = torch.empty(ns.step_workspace_size(*shape), dtype=torch.uint8, device="cuda")
    We, Me = Wd.clone(), Md.clone()
    for _ in range(2):
        ns.muon_step(We, Me, Gd, workspace=ws, **kw)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    Wx, Mx = Wd.clone(), Md.clone()
    with torch.cuda.stream(side):  # first launches (per-device set-up) outside the capture
        ns.muon_step(Wx, Mx, Gd, workspace=ws, **kw)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ns.muon_step(Wd, Md, Gd, workspace=ws, **kw)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert ns.read_error(ws) == 0
    np.testing.assert_array_equal(Md.cpu().numpy(), Me.cpu().numpy())
    np.testing.assert_array_equal(Wd.cpu().numpy().view(np.uint32), We.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("steps,shared", [(5, False), (0, False), (5, True)])
def test_grouped_step_equals_separate_steps_bitwise(steps, shared):
    # An optimizer step's parameter groups: wide, tall (larger shape factor) and
    # a long-contraction stack, each with its own hyperparameters, plus an empty
    # group; one call equals one muon_step_ws call per group, bit for bit.
    # With `shared` the groups have the same factors (the last update's
    # launch-wide form), otherwise each its own (the per-group form).
    specs = [((3, 256, 512), dict(lr=0.02, momentum=0.95, weight_decay=0.01)),
             ((2, 520, 264), dict(lr=0.05, momentum=0.9, nesterov=False)),
             ((1, 1040, 1280), dict(lr=0.01, momentum=0.8, weight_decay=0.1, scale=0.7)),
             ((0, 64, 128), dict(lr=0.02))]
    if shared:
        specs = [(shape, dict(lr=0.02, momentum=0.95, weight_decay=0.01, scale=1.0)) for shape, _ in specs]
    base = []
    for i, (shape, hp) in enumerate(specs):
        base.append((f32_stack(shape, 30 + i), f32_stack(shape, 40 + i, 0.05), f32_stack(shape, 50 + i, 0.05), hp))
    groups = []
    for W, M, G, hp in base:
        groups.append(dict(W=torch.from_numpy(W).cuda(), M=torch.from_numpy(M).cuda(), G=torch.from_numpy(G).cuda(), **hp))
    ws = torch.empty(ns.step_grouped_workspace_size(groups), dtype=torch.uint8, device="cuda")
    ns.muon_step_grouped(groups, steps=steps, workspace=ws)
    torch.cuda.synchronize()
    assert ns.read_error(ws) == 0
    for (W, M, G, hp), g in zip(base, groups):
        if W.shape[0] == 0:
            continue
        Ws, Ms = run_step(W, M, G, steps=steps, **hp)
        np.testing.assert_array_equal(g["M"].cpu().numpy(), Ms)
        np.testing.assert_array_equal(g["W"].cpu().numpy().view(np.uint32), Ws.view(np.uint32))


@pytest.mark.slow
def test_full_size_expert_stack_sampled():
    w = ns_inputs.WORKLOADS["experts_128x1536x2048"]
    G = np.stack([ns_inputs.matrix_f32(w, k) for k in range(w.batch)])
    M = f32_stack(G.shape, 14, 0.02)
    W = f32_stack(G.shape, 15, 0.02)
    Wn, Mn = run_step(W, M, G, lr=0.02, momentum=0.95, weight_decay=0.01)
    for k in (0, 77, 127):
        W_ref, M_ref, O_ref = oracle.muon_step(W[k], M[k], G[k], 0.02, 0.95, weight_decay=0.01)
        assert np.all(np.abs(Mn[k] - M_ref) <= 2.0 ** -23 * (0.95 * np.abs(M[k]) + np.abs(G[k])) + 1e-38)
        upd = 0.02 * np.linalg.norm(O_ref)
        assert np.linalg.norm(Wn[k] - W_ref) <= NS_TOL * upd + 4 * 2.0 ** -24 * np.linalg.norm(W[k])


def _step_sweep(n=10):
    # Seeded draws: ragged shapes (multiples of 8, wide and tall, every third
    # with both sides past 1024 for 2-SM products), and hyperparameters.
    rng = np.random.default_rng(20261204)
    out = []
    for i in range(n):
        lo, hi = (1032, 1200) if i % 3 == 0 else (8, 880)
        r, c = (8 * int(rng.integers(lo // 8, hi // 8 + 1)) for _ in range(2))
        hp = dict(lr=float(rng.choice([0.002, 0.02, 0.2])), momentum=float(rng.choice([0.0, 0.8, 0.95])),
                  nesterov=bool(rng.integers(0, 2)), weight_decay=float(rng.choice([0.0, 0.01, 0.1])))
        out.append(((1 + int(rng.integers(0, 3)), r, c), hp))
    return out


STEP_SWEEP = _step_sweep()


@pytest.mark.parametrize("i,case", list(enumerate(STEP_SWEEP)),
                         ids=[f"{b}x{r}x{c}" for (b, r, c), _ in STEP_SWEEP])
def test_random_steps_vs_oracle_and_chain(i, case):
    # The fused step against the oracle step (M' to one fp32 rounding, W' to
    # the NS tolerance on its update term) and bit for bit against its chain
    # of separate kernels.
    shape, hp = case
    W, M, G = f32_stack(shape, 300 + i), f32_stack(shape, 400 + i, 0.05), f32_stack(shape, 500 + i, 0.05)
    Wn, Mn = run_step(W, M, G, **hp)
    Wc, Mc, _ = run_chain(W, M, G, **hp)
    np.testing.assert_array_equal(Mn, Mc)
    np.testing.assert_array_equal(Wn.view(np.uint32), Wc.view(np.uint32))
    mu = hp["momentum"]
    W_ref, M_ref, O_ref = oracle.muon_step(W, M, G, hp["lr"], mu, nesterov=hp["nesterov"],
                                           weight_decay=hp["weight_decay"])
    bound = 2.0 ** -23 * (np.abs(mu * M.astype(np.float64)) + np.abs(G)) + 1e-38
    assert np.all(np.abs(Mn - M_ref) <= bound)
    s = ns.default_scale(shape[1], shape[2])
    tols = ns_tols(u_bits(M, G, mu, hp["nesterov"]))
    for k in range(shape[0]):
        upd = hp["lr"] * s * np.linalg.norm(O_ref[k])
        err = np.linalg.norm(Wn[k] - W_ref[k])
        assert err <= tols[k] * upd + 4 * 2.0 ** -24 * np.linalg.norm(W[k]), (k, err, upd, tols[k])
