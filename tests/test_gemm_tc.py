"""The tcgen05 tensor-core GEMMs of the prefill (qw_op_gemm_f16, qw_op_gemm_swiglu_f16)
against float64 numpy on the same fp16 operands: tile-aligned and ragged M, N, K, the
bias, residual-accumulate and fused SwiGLU epilogues, and more output tiles than SMs (each
persistent CTA then runs several tiles through its two TMEM accumulators)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _f16(a):
    return a.astype(np.float16)


@pytest.mark.parametrize("M,N,K,bias,acc", [
    (128, 256, 64, False, False),
    (1, 256, 64, True, False),
    (100, 1536, 1536, True, False),
    (300, 896, 896, False, True),     # N not a multiple of the 256-column tile
    (257, 128, 1000, True, False),    # K not a multiple of the 64-element stage
    (129, 2048, 1536, False, True),
    (512, 1536, 8960, False, True),   # the down projection's K
    (2048, 4096, 256, True, False),   # more tiles than SMs: each persistent CTA takes several
    (1000, 2056, 320, False, True),   # several tiles per CTA with ragged M and N
    (4096, 1536, 256, True, False),   # 192-column tiles, several per CTA
    (2000, 1536, 512, False, True),   # 192-column tiles, residual add, ragged M
    (128, 1536, 8960, False, True),   # short prompt: 64-column tiles, the down projection's K
    (77, 2048, 1536, True, False),    # short ragged prompt, fused q/k/v width
])
def test_gemm_f16(M, N, K, bias, acc):
    from qwen2_decoder_forward_decode_gb300 import binding
    rng = np.random.default_rng(M * 7 + N + K)
    A = _f16(rng.standard_normal((M, K)))
    B = _f16(rng.standard_normal((N, K)) * 0.02)
    bb = torch.from_numpy((rng.standard_normal(N) * 0.02).astype(np.float32)).to(torch.bfloat16)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    tA, tB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    tbias = bb.cuda() if bias else None
    tC = torch.from_numpy(C0.copy()).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.gemm_f16(M, N, K, tA.data_ptr(), tB.data_ptr(), tbias.data_ptr() if bias else None,
                     tC.data_ptr(), acc, err.data_ptr())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    if bias:
        ref += bb.float().numpy().astype(np.float64)[None, :]
    if acc:
        ref += C0
    got = tC.cpu().numpy()
    # fp32 accumulation bound: a small multiple of 2^-24 per term of sum_k |a_k b_k|
    bound = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)).T
    tol = 1e-5 * bound + 1e-6 * np.abs(C0 if acc else 0) + 1e-7
    assert np.all(np.abs(got - ref) <= tol), float(np.max(np.abs(got - ref) / tol))


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (33, 1000, 384), (200, 8960, 1536), (1100, 8960, 256)])
def test_gemm_swiglu_f16(M, N, K):
    from qwen2_decoder_forward_decode_gb300 import binding
    rng = np.random.default_rng(M + N + K)
    A = _f16(rng.standard_normal((M, K)))
    Wg = _f16(rng.standard_normal((N, K)) * 0.05)
    Wu = _f16(rng.standard_normal((N, K)) * 0.05)
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tA, tG, tU = (torch.from_numpy(x).cuda() for x in (A, Wg, Wu))
    binding.gemm_swiglu_f16(M, N, K, tA.data_ptr(), tG.data_ptr(), tU.data_ptr(), out.data_ptr(),
                            err.data_ptr())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    g = A.astype(np.float64) @ Wg.astype(np.float64).T
    u = A.astype(np.float64) @ Wu.astype(np.float64).T
    ref = g / (1 + np.exp(-g)) * u
    got = out.float().cpu().numpy()
    np.testing.assert_allclose(got, ref, rtol=2e-3, atol=1e-4 * np.abs(ref).max())


def test_gemm_rejects_bad_shapes():
    from qwen2_decoder_forward_decode_gb300 import binding
    with pytest.raises(binding.QwError):
        binding.gemm_f16(16, 12, 64, 16, 16, None, 16, 0, 16)   # N not a multiple of 8
    with pytest.raises(binding.QwError):
        binding.gemm_f16(16, 16, 64, 8, 16, None, 16, 0, 16)    # misaligned A
