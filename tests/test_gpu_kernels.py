"""Per-kernel GPU parity through the C ABI: each kernel of the path against the
oracle's definition of its step, evaluated in fp64 on the same bf16 inputs.

Tolerance, from the arithmetic: each kernel rounds its fp32 result to bf16
once (relative error <= 2^-9 per element, so <= 2^-9 ~ 1.95e-3 in relative
Frobenius norm) after an fp32 accumulation whose error is far smaller at these
sizes; the bound used is 3e-3.  Shapes span several 128 x 256 tiles, ragged
edges in M, N and K, and batches.  Contractions above 1024 run on CTA pairs
with 2-SM MMAs, shorter ones on pairs sharing a multicast B panel; the
1096 x 1304 cases also give the pair walk an odd row-tile count (the second
CTA of the last pair has no rows to store).
"""
import numpy as np
import pytest
import torch

import newton_schulz_07_gb300 as ns
import oracle
from nsutil import per_matrix_rel, random_bits, symmetric_bits, to_bits, to_dev, to_f64
import ns_inputs

pytestmark = pytest.mark.gpu
KERNEL_TOL = 3e-3

SHAPES = [(1, 8, 8), (3, 136, 264), (2, 256, 512), (2, 264, 136), (1, 392, 200), (1, 200, 392),
          (2, 128, 128), (1, 520, 1040), (1, 1040, 520), (1, 1096, 1304), (1, 1304, 1096),
          (1, 1024, 1032), (1, 1032, 1024)]  # contraction 1024 (multicast pairs) next to 1032 (2-SM MMAs)


def f64(bits):
    return ns_inputs.bf16_bits_to_f64(bits)


@pytest.mark.parametrize("shape", SHAPES)
def test_normalize(shape):
    bits = random_bits(shape, seed=sum(shape))
    G = to_dev(bits)
    ws = ns.alloc_workspace(*shape)
    X = ns.muon_ns_normalize(G, ws, eps=1e-7)
    off, nb = ns.workspace_region(*shape, ns._lib.WS_NORMS)
    norms = ws[off:off + nb].view(torch.float32).cpu().numpy()
    g = f64(bits)
    for k in range(shape[0]):
        nu = oracle.frobenius_norm(g[k])
        assert abs(norms[k] - nu) <= 1e-5 * nu
    ref = np.stack([oracle.normalize(g[k], 1e-7) for k in range(shape[0])])
    assert max(per_matrix_rel(to_f64(X), ref)) <= KERNEL_TOL
    # Elementwise: one bf16 rounding of the scaled value.
    assert np.all(np.abs(to_f64(X) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)


def gram_ref(x):
    return oracle.gram(x) if x.shape[0] <= x.shape[1] else oracle.gram(x.T)


@pytest.mark.parametrize("shape", SHAPES)
def test_gram(shape):
    bits = random_bits(shape, seed=7 + sum(shape), scale=0.05)
    A = ns.muon_ns_gram(to_dev(bits))
    torch.cuda.synchronize()
    a = to_bits(A)
    np.testing.assert_array_equal(a, np.swapaxes(a, 1, 2))  # bit-symmetric
    x = f64(bits)
    ref = np.stack([gram_ref(x[k]) for k in range(shape[0])])
    assert max(per_matrix_rel(f64(a), ref)) <= KERNEL_TOL


@pytest.mark.parametrize("batch,m", [(1, 8), (2, 136), (3, 256), (1, 392), (2, 520), (1, 1024), (1, 1032), (1, 1040),
                                     (2, 1096)])
@pytest.mark.parametrize("split_diag", [False, True])
def test_poly(batch, m, split_diag):
    bits = symmetric_bits(batch, m, seed=m)
    b, c = -4.7750, 2.0315
    D = torch.full((batch, m), float("nan"), dtype=torch.float32, device="cuda") if split_diag else None
    B = ns.muon_ns_poly(to_dev(bits), b, c, diag=D)
    torch.cuda.synchronize()
    bb = to_bits(B)
    np.testing.assert_array_equal(bb, np.swapaxes(bb, 1, 2))
    a = f64(bits)
    ref = np.stack([oracle.poly(a[k], b, c) for k in range(batch)])
    got = f64(bb)
    if split_diag:
        idx = np.arange(m)
        assert np.all(bb[:, idx, idx] == 0)
        d = D.cpu().numpy().astype(np.float64)
        ref_d = ref[:, idx, idx]
        # fp32 epilogue, no bf16 rounding: fp32 accumulation error only.
        assert np.all(np.abs(d - ref_d) <= 1e-5 * np.abs(ref).max(axis=(1, 2))[:, None])
        got[:, idx, idx] = d
    assert max(per_matrix_rel(got, ref)) <= KERNEL_TOL


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("split_diag", [False, True])
def test_update(shape, split_diag):
    batch, r, c = shape
    m = min(r, c)
    xbits = random_bits(shape, seed=11 + r, scale=0.05)
    bbits = symmetric_bits(batch, m, seed=13 + c, scale=0.05)
    a = 3.4445
    D = None
    x, B = f64(xbits), f64(bbits)
    if split_diag:
        idx = np.arange(m)
        dvals = np.random.default_rng(r + c).uniform(-3.0, 1.0, size=(batch, m)).astype(np.float32)
        bbits[:, idx, idx] = 0
        B = f64(bbits)
        B[:, idx, idx] = dvals
        D = torch.from_numpy(dvals).cuda()
    Xn = ns.muon_ns_update(to_dev(xbits), to_dev(bbits), a, diag=D)
    torch.cuda.synchronize()
    ref = []
    for k in range(batch):
        if r <= c:
            ref.append(oracle.update(x[k], B[k], a))
        else:  # tall input kept in its own orientation: (a X^T + B X^T)^T
            ref.append(oracle.update(x[k].T, B[k], a).T)
    assert max(per_matrix_rel(to_f64(Xn), np.stack(ref))) <= KERNEL_TOL


def test_device_error_word_stays_clear():
    shape = (2, 256, 512)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    X = to_dev(random_bits(shape, seed=3))
    A = ns.muon_ns_gram(X, device_error=err)
    D = torch.empty((2, 256), dtype=torch.float32, device="cuda")
    B = ns.muon_ns_poly(A, -4.775, 2.0315, diag=D, device_error=err)
    ns.muon_ns_update(X, B, 3.4445, diag=D, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


@pytest.mark.parametrize("shape", [(3, 136, 264), (2, 264, 136), (1, 392, 200)])
def test_normalize_norms_only(shape):
    bits = random_bits(shape, seed=5 + sum(shape), scale=0.3)
    ws = ns.alloc_workspace(*shape)
    assert ns.muon_ns_normalize(to_dev(bits), ws, norms_only=True) is None
    off, nb = ns.workspace_region(*shape, ns._lib.WS_NORMS)
    norms = ws[off:off + nb].view(torch.float32).cpu().numpy()
    g = f64(bits)
    for k in range(shape[0]):
        assert abs(norms[k] - oracle.frobenius_norm(g[k])) <= 1e-5 * oracle.frobenius_norm(g[k])


@pytest.mark.parametrize("shape", SHAPES)
def test_gram_of_unscaled_input(shape):
    # The first NS step: X is the raw G and the Gram of G / (norm + eps) is formed.
    bits = random_bits(shape, seed=17 + sum(shape), scale=3.0)
    norms = torch.from_numpy(np.array([oracle.frobenius_norm(m) for m in f64(bits)], dtype=np.float32)).cuda()
    A = ns.muon_ns_gram(to_dev(bits), norms=norms, eps=1e-7)
    torch.cuda.synchronize()
    a = to_bits(A)
    np.testing.assert_array_equal(a, np.swapaxes(a, 1, 2))
    x = f64(bits)
    nu = norms.cpu().numpy().astype(np.float64)
    ref = np.stack([gram_ref(x[k] / (nu[k] + 1e-7)) for k in range(shape[0])])
    assert max(per_matrix_rel(f64(a), ref)) <= KERNEL_TOL


@pytest.mark.parametrize("shape", SHAPES)
def test_update_of_unscaled_input(shape):
    batch, r, c = shape
    m = min(r, c)
    xbits = random_bits(shape, seed=19 + r, scale=2.0)
    bbits = symmetric_bits(batch, m, seed=23 + c, scale=0.05)
    idx = np.arange(m)
    dvals = np.random.default_rng(r * c).uniform(-3.0, 1.0, size=(batch, m)).astype(np.float32)
    bbits[:, idx, idx] = 0
    B = f64(bbits)
    B[:, idx, idx] = dvals
    x = f64(xbits)
    nu = np.array([oracle.frobenius_norm(x[k]) for k in range(batch)], dtype=np.float32)
    a = 3.4445
    Xn = ns.muon_ns_update(to_dev(xbits), to_dev(bbits), a, diag=torch.from_numpy(dvals).cuda(),
                           norms=torch.from_numpy(nu).cuda(), eps=1e-7)
    torch.cuda.synchronize()
    ref = []
    for k in range(batch):
        xs = x[k] / (float(nu[k]) + 1e-7)
        ref.append(oracle.update(xs, B[k], a) if r <= c else oracle.update(xs.T, B[k], a).T)
    assert max(per_matrix_rel(to_f64(Xn), np.stack(ref))) <= KERNEL_TOL
