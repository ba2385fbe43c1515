"""GPU check of the batched path's 3xTF32 tensor-core GEMM against float64.

C = A W^T is computed by the tcgen05 kernel through the library's
l2_gemm_tf32x3 hook and compared with a float64 product. The error of each
element is normalised by sum_k |A_ik| |W_jk|, the scale every fp32 summation
error is measured against. A single-pass TF32 product (10-bit mantissa) errs by
~1e-4 of that scale; an fp32-accurate product stays near 1e-7. Shapes cover a
full 128-row tile pair, a ragged M/N/K, K below one 32-float block, the
vocabulary-sized classifier, both N tiles (64 and 128), and K split over
clusters of 3, 6 and 8 CTAs (deterministic reduction through distributed
shared memory).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

SHAPES = [(256, 1536, 512), (200, 328, 1376), (1, 64, 4), (130, 4099, 36), (256, 32000, 512),
          (129, 8192, 64), (256, 512, 1376), (256, 2752, 512), (256, 512, 512)]


@pytest.fixture(scope="module")
def l2():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_fp32_token_decode_b300 as m
    return m


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_3xtf32_matches_float64(l2, M, N, K):
    import torch
    rng = np.random.default_rng(M * 7919 + N * 31 + K)
    A = rng.standard_normal((M, K)).astype(np.float32)
    W = (0.02 * rng.standard_normal((N, K))).astype(np.float32)
    ref = A.astype(np.float64) @ W.astype(np.float64).T
    scale = np.abs(A).astype(np.float64) @ np.abs(W).astype(np.float64).T
    dA = torch.from_numpy(A).cuda()
    dW = torch.from_numpy(W).cuda()
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    l2.l2_gemm_tf32x3(dA, dW, dC, M, N, K)
    C = dC.cpu().numpy()
    assert np.all(np.isfinite(C))
    err = np.abs(C.astype(np.float64) - ref) / scale
    assert err.max() < 1e-5, err.max()
    assert err.mean() < 1e-6, err.mean()


def test_gemm_rejects_bad_sizes(l2):
    import torch
    d = torch.zeros(64, dtype=torch.float32, device="cuda")
    for M, N, K in [(0, 8, 8), (8, 0, 8), (8, 8, 6), (8, 8, 0)]:
        with pytest.raises(l2.L2Error):
            l2.l2_gemm_tf32x3(d, d, d, M, N, K)


@pytest.mark.parametrize("M,N,K", [(64, 1024, 11008), (32, 512, 32768), (256, 512, 4096)])
def test_gemm_long_k_accuracy_is_fp32_class(l2, M, N, K):
    # relative L2 error of the whole product against float64: an fp32 GEMM with
    # round-to-nearest accumulation stays near 1e-6 at these lengths, while
    # letting the tensor core's accumulator absorb all of K grows linearly
    # (about 2e-5 at K = 11008, 6e-5 at 32768)
    import torch
    rng = np.random.default_rng(K + N)
    A = rng.standard_normal((M, K)).astype(np.float32)
    W = (0.02 * rng.standard_normal((N, K))).astype(np.float32)
    ref = A.astype(np.float64) @ W.astype(np.float64).T
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    l2.l2_gemm_tf32x3(torch.from_numpy(A).cuda(), torch.from_numpy(W).cuda(), dC, M, N, K)
    C = dC.cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(C - ref) / np.linalg.norm(ref)
    assert rel < 3e-6, rel
