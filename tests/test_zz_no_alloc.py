"""qw_op_decode_attention_noalloc: decode attention for callers that cannot allocate device
memory (code inside another runtime that owns the device memory, or loops that must not
pay cudaMalloc's synchronisation). Its scratch is a fixed array inside the library; the
result must equal the workspace entry point's on the same inputs, call after call.

This file is collected last so that a failure here leaves every other test already run."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("kv_dtype,nq,nkv,hd,ctx,stride", [
    (2, 12, 2, 128, 178, 2048),    # the 1.5B decode shape
    (2, 12, 2, 128, 8192, 8192),   # the longest context that fits the fixed array
    (0, 4, 2, 16, 9, 16),
])
def test_noalloc_matches_workspace_entry_point_twice(kv_dtype, nq, nkv, hd, ctx, stride):
    from qwen2_decoder_forward_decode_gb300 import binding
    assert binding.decode_attention_workspace(nq, nkv, hd, stride) <= \
        int(binding.lib().qw_op_decode_attention_noalloc_limit())
    rng = np.random.default_rng(ctx + nq)
    dt = torch.float16 if kv_dtype == 2 else torch.float32
    q = torch.from_numpy(rng.standard_normal(nq * hd).astype(np.float32)).cuda()
    k = torch.from_numpy(rng.standard_normal((nkv, stride, hd)).astype(np.float32)).to(dt).cuda()
    v = torch.from_numpy(rng.standard_normal((nkv, stride, hd)).astype(np.float32)).to(dt).cuda()
    nbytes = binding.decode_attention_workspace(nq, nkv, hd, stride)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    want = torch.empty(nq * hd, dtype=torch.float32, device="cuda")
    binding.decode_attention(kv_dtype, nq, nkv, hd, ctx, stride, q.data_ptr(), k.data_ptr(),
                             v.data_ptr(), want.data_ptr(), ws.data_ptr(), nbytes)
    torch.cuda.synchronize()
    ref = want.cpu().numpy()
    for _ in range(2):
        got = torch.full((nq * hd,), float("nan"), dtype=torch.float32, device="cuda")
        binding.decode_attention_noalloc(kv_dtype, nq, nkv, hd, ctx, stride, q.data_ptr(),
                                         k.data_ptr(), v.data_ptr(), got.data_ptr())
        torch.cuda.synchronize()
        np.testing.assert_allclose(got.cpu().numpy(), ref, rtol=0,
                                   atol=2e-5 * max(1.0, float(np.abs(ref).max())))


def test_noalloc_rejects_shapes_beyond_the_fixed_array():
    from qwen2_decoder_forward_decode_gb300 import binding
    with pytest.raises(binding.QwError) as e:
        binding.decode_attention_noalloc(2, 64, 8, 128, 100, 65536, 16, 16, 16, 16)
    assert e.value.status == 2  # QW_ERR_UNSUPPORTED
