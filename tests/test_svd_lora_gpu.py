"""LoRA from the quantisation error on the GPU ("W4A4 CUDA Kernel for Voice
Clone", 2.1-2.2) against the CPU oracle (exact LAPACK SVD): the GPU's SVD is a
randomized subspace iteration, so it is held to the oracle through singular
values, residual norms and reconstructed products, not bits; the codes and
scales of each round are the packer's and are compared bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import w4a4_quantized_gemm_gb300 as w4
from synthetic import make_linear_case
from tests.helpers import check_tol
from tests.test_oracle_pins import planted_rank_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from w4a4_quantized_gemm_gb300 import build
    build.build()
    w4.lib()
    torch.cuda.init()


def _packed(N, K, r):
    return torch.empty(w4.packed_weights_bytes(N, K, r), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("N,K,r", [(512, 1024, 16), (1024, 384, 32), (256, 256, 64)])
def test_truncated_svd_decaying_spectrum(N, K, r):
    """A = U0 diag(0.9^i) V0^T: singular values, subspaces and the residual of the
    rank-r approximation match LAPACK's."""
    rng = np.random.default_rng(N + K + r)
    m = min(N, K)
    U0, _ = np.linalg.qr(rng.normal(size=(N, m)))
    V0, _ = np.linalg.qr(rng.normal(size=(K, m)))
    sig = 0.9 ** np.arange(m)
    A = ((U0 * sig) @ V0.T).astype(np.float32)
    U, S, V = w4.w4a4_truncated_svd(torch.from_numpy(A).cuda(), r, power_iters=8)
    U, S, V = U.cpu().numpy().astype(np.float64), S.cpu().numpy().astype(np.float64), V.cpu().numpy().astype(np.float64)
    Ue, Se, Ve = oracle.truncated_svd(A, r)
    np.testing.assert_allclose(S, Se, rtol=1e-4)
    # principal angles: the cosines between the spaces are all ~1
    assert np.linalg.svd(U.T @ Ue, compute_uv=False).min() > 1 - 1e-4
    assert np.linalg.svd(V.T @ Ve, compute_uv=False).min() > 1 - 1e-4
    A64 = A.astype(np.float64)
    opt = np.linalg.norm(A64 - (Ue * Se) @ Ve.T)
    assert np.linalg.norm(A64 - (U * S) @ V.T) <= opt * (1 + 1e-4) + 1e-6 * np.linalg.norm(A64)
    assert w4.w4a4_device_status() == 0


def test_svd_lora_recovers_a_planted_low_rank_error():
    """W = Q0 + D (D rank 2): the codes are Q0's, the LoRA product is D^T, and the
    W4A16 layer on the result reproduces the unquantised layer."""
    W, q0, s0, D = planted_rank_case(N=256, K=512, rank=2, seed=51)
    N, K, r = 256, 512, 16
    packed = _packed(N, K, r)
    Ld, Lu, errs = w4.w4a4_pack_weights_svd(torch.from_numpy(W).cuda(), r, packed, rounds=2, power_iters=8)
    codes, scales, _, _ = w4.w4a4_debug_unpack_weights(packed, N, K, r)
    assert np.array_equal(codes.cpu().numpy(), q0)
    assert np.array_equal(oracle.f16_to_f32_array(scales.cpu().numpy().view(np.uint16)).astype(np.float64), s0)
    L = Ld.cpu().numpy().astype(np.float64) @ Lu.cpu().numpy().astype(np.float64)   # [K, N]
    assert np.linalg.norm(L - D.T) <= 2e-3 * np.linalg.norm(D)                       # fp16 factors
    assert errs[0] <= 1e-3 * np.linalg.norm(D)
    # end to end through the W4A16 path (no activation quantisation): the layer of W itself
    c = make_linear_case(7, K, N, r, seed=52)
    X = torch.from_numpy(c.X.view(np.float16).copy()).cuda()
    cs = torch.from_numpy(c.colscale.view(np.float16).copy()).cuda()
    b = torch.from_numpy(c.bias.view(np.float16).copy()).cuda()
    Y = torch.empty((7, N), dtype=torch.float16, device="cuda")
    w4.w4a16_linear(X, packed, cs, b, Y, r)
    torch.cuda.synchronize()
    Xf = c.X.view(np.float16).astype(np.float64)
    y = c.colscale.view(np.float16).astype(np.float64) * (Xf @ W.astype(np.float64).T) + \
        c.bias.view(np.float16).astype(np.float64)
    check_tol(Y, y, "W4A16 layer with the SVD LoRA vs the unquantised layer")
    assert w4.w4a4_device_status() == 0


@pytest.mark.parametrize("N,K,r", [(1024, 1024, 32), (512, 2048, 16)])
def test_svd_lora_on_quantisation_error_matches_lapack(N, K, r):
    """Noise-like quantisation error (flat spectrum): one round gives the packer's
    codes and a rank-r correction whose residual is within 1e-3 of the exact
    truncated SVD's; three rounds never end above the first."""
    c = make_linear_case(1, K, N, 0, seed=N + K)
    Wd = torch.from_numpy(c.W).cuda()
    packed = _packed(N, K, r)
    Ld, Lu, errs = w4.w4a4_pack_weights_svd(Wd, r, packed, rounds=1, power_iters=16)
    best, oerrs = oracle.svd_lora(c.W, r, rounds=1)
    codes, scales, _, _ = w4.w4a4_debug_unpack_weights(packed, N, K, r)
    assert np.array_equal(codes.cpu().numpy(), best["codes"])
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), best["scales"])
    assert abs(errs[0] / oerrs[0] - 1) <= 1e-3, (errs, oerrs)
    # the fp16 factors as stored reconstruct the error about as well
    E = c.W.astype(np.float64) - oracle.dequantize_weights(best["codes"], best["scales"])
    L = (Ld.cpu().numpy().astype(np.float64) @ Lu.cpu().numpy().astype(np.float64)).T
    assert np.linalg.norm(E - L) <= oerrs[0] * (1 + 2e-3)
    packed3 = _packed(N, K, r)
    _, _, errs3 = w4.w4a4_pack_weights_svd(Wd, r, packed3, rounds=3, power_iters=16)
    kept = [e for e in errs3 if e >= 0]
    assert min(kept) <= errs3[0] and abs(errs3[0] / errs[0] - 1) <= 1e-3
    best3, oerrs3 = oracle.svd_lora(c.W, r, rounds=3)
    assert abs(min(kept) / best3["err"] - 1) <= 1e-2, (errs3, oerrs3)
    assert w4.w4a4_device_status() == 0
