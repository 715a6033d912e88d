"""qw_op_decode_attention_noalloc: decode attention for callers that cannot allocate device
memory (code inside another runtime that owns the device memory, or loops that must not
pay cudaMalloc's synchronisation). Its scratch is a fixed array inside the library; the
result must equal the workspace entry point's and the oracle's on the same inputs, call
after call, whatever shape the previous call left in the shared array.

This file is collected last so that a failure here leaves every other test already run."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _inputs(kv_dtype, nq, nkv, hd, stride, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal(nq * hd).astype(np.float32)
    k = rng.standard_normal((nkv, stride, hd)).astype(np.float32)
    v = rng.standard_normal((nkv, stride, hd)).astype(np.float32)
    dt = torch.float16 if kv_dtype == 2 else torch.float32
    if kv_dtype == 2:  # the values the device holds
        k, v = k.astype(np.float16).astype(np.float32), v.astype(np.float16).astype(np.float32)
    dev = [torch.from_numpy(q).cuda(), torch.from_numpy(k).to(dt).cuda(), torch.from_numpy(v).to(dt).cuda()]
    return q, k, v, dev


def _oracle(q, k, v, nq, nkv, hd, ctx):
    g = nq // nkv
    qh = q.reshape(nq, hd).astype(np.float64)
    return np.stack([oracle.attend_one_head(qh[h][:, None], k[h // g, :ctx].T.astype(np.float64),
                                            v[h // g, :ctx].T.astype(np.float64), [ctx - 1], hd)[:, 0]
                     for h in range(nq)]).reshape(-1)


def _noalloc(kv_dtype, nq, nkv, hd, ctx, stride, dev):
    from qwen2_decoder_forward_decode_gb300 import binding
    got = torch.full((nq * hd,), float("nan"), dtype=torch.float32, device="cuda")
    binding.decode_attention_noalloc(kv_dtype, nq, nkv, hd, ctx, stride, dev[0].data_ptr(),
                                     dev[1].data_ptr(), dev[2].data_ptr(), got.data_ptr())
    torch.cuda.synchronize()
    return got.cpu().numpy()


def _tol(ref):
    return 2e-5 * max(1.0, float(np.abs(ref).max()))


@pytest.mark.parametrize("kv_dtype,nq,nkv,hd,ctx,stride", [
    (2, 12, 2, 128, 178, 2048),    # the 1.5B decode shape
    (2, 12, 2, 128, 8192, 8192),   # the longest context that fits the fixed array
    (0, 4, 2, 16, 9, 16),
])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(kv_dtype, nq, nkv, hd, ctx, stride):
    from qwen2_decoder_forward_decode_gb300 import binding
    assert binding.decode_attention_workspace(nq, nkv, hd, stride) <= \
        int(binding.lib().qw_op_decode_attention_noalloc_limit())
    q, k, v, dev = _inputs(kv_dtype, nq, nkv, hd, stride, ctx + nq)
    nbytes = binding.decode_attention_workspace(nq, nkv, hd, stride)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    want = torch.empty(nq * hd, dtype=torch.float32, device="cuda")
    binding.decode_attention(kv_dtype, nq, nkv, hd, ctx, stride, dev[0].data_ptr(), dev[1].data_ptr(),
                             dev[2].data_ptr(), want.data_ptr(), ws.data_ptr(), nbytes)
    torch.cuda.synchronize()
    ref = want.cpu().numpy()
    exact = _oracle(q, k, v, nq, nkv, hd, ctx)
    for _ in range(2):
        got = _noalloc(kv_dtype, nq, nkv, hd, ctx, stride, dev)
        np.testing.assert_allclose(got, ref, rtol=0, atol=_tol(ref))
        np.testing.assert_allclose(got, exact, rtol=0, atol=_tol(exact))


def test_noalloc_after_a_call_of_another_kv_type():
    """An fp32 call at stride 8192 splits the context into more chunks than an fp16 call
    of the same heads, so its partials cover the place where the fp16 call keeps its
    counters. The fp16 call that follows must still clear its own counters and write
    every output."""
    nq, nkv, hd, stride = 12, 2, 128, 8192
    q32, k32, v32, dev32 = _inputs(0, nq, nkv, hd, stride, 5)
    got32 = _noalloc(0, nq, nkv, hd, stride, stride, dev32)
    exact32 = _oracle(q32, k32, v32, nq, nkv, hd, stride)
    np.testing.assert_allclose(got32, exact32, rtol=0, atol=_tol(exact32))
    q16, k16, v16, dev16 = _inputs(2, nq, nkv, hd, stride, 6)
    for ctx in (stride, 1000):
        got16 = _noalloc(2, nq, nkv, hd, ctx, stride, dev16)
        assert np.all(np.isfinite(got16))
        exact16 = _oracle(q16, k16, v16, nq, nkv, hd, ctx)
        np.testing.assert_allclose(got16, exact16, rtol=0, atol=_tol(exact16))


def test_noalloc_rejects_shapes_beyond_the_fixed_array():
    from qwen2_decoder_forward_decode_gb300 import binding
    with pytest.raises(binding.QwError) as e:
        binding.decode_attention_noalloc(2, 64, 8, 128, 100, 65536, 16, 16, 16, 16)
    assert e.value.status == 2  # QW_ERR_UNSUPPORTED
