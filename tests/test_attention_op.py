"""Decode attention as a single operation (qw_op_decode_attention) against the oracle's
causal softmax attention, over context lengths that cover one key, chunk boundaries,
ragged tails and the full capacity."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("dtype", [0, 2])  # KV cache element: fp32, fp16
@pytest.mark.parametrize("nq,nkv,hd,ctx,stride", [
    (12, 2, 128, 1, 2048),
    (12, 2, 128, 31, 2048),
    (12, 2, 128, 32, 2048),
    (12, 2, 128, 33, 2048),
    (12, 2, 128, 178, 2048),
    (12, 2, 128, 2048, 2048),
    (14, 2, 64, 63, 64),
    (4, 2, 16, 16, 16),
    (4, 4, 16, 9, 16),
    (12, 2, 128, 4224, 8192),
    (12, 2, 128, 8192, 8192),
])
def test_decode_attention_matches_oracle(dtype, nq, nkv, hd, ctx, stride):
    from qwen2_decoder_forward_decode_gb300 import binding
    rng = np.random.default_rng(ctx * 7 + nq)
    q = rng.standard_normal(nq * hd).astype(np.float32)
    k = rng.standard_normal((nkv, stride, hd)).astype(np.float32)
    v = rng.standard_normal((nkv, stride, hd)).astype(np.float32)
    if dtype == 2:
        k, v = k.astype(np.float16).astype(np.float32), v.astype(np.float16).astype(np.float32)
        tk = torch.from_numpy(k).to(torch.float16).cuda()
        tv = torch.from_numpy(v).to(torch.float16).cuda()
    else:
        tk, tv = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    tq = torch.from_numpy(q).cuda()
    out = torch.empty(nq * hd, dtype=torch.float32, device="cuda")
    nbytes = binding.decode_attention_workspace(nq, nkv, hd, stride)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call checks that the counters were left at zero
        out.fill_(float("nan"))
        binding.decode_attention(dtype, nq, nkv, hd, ctx, stride, tq.data_ptr(), tk.data_ptr(),
                                 tv.data_ptr(), out.data_ptr(), ws.data_ptr(), nbytes)
        torch.cuda.synchronize()
        got = out.cpu().numpy().reshape(nq, hd)
        g = nq // nkv
        for h in range(nq):
            ref = oracle.attend_one_head(q.reshape(nq, hd)[h][:, None].astype(np.float64),
                                         k[h // g, :ctx].T.astype(np.float64),
                                         v[h // g, :ctx].T.astype(np.float64), [ctx - 1], hd)[:, 0]
            np.testing.assert_allclose(got[h], ref, rtol=0, atol=2e-5 * max(1.0, np.abs(ref).max()))


def test_decode_attention_rejects_bad_arguments():
    from qwen2_decoder_forward_decode_gb300 import binding
    with pytest.raises(binding.QwError):
        binding.decode_attention(2, 12, 2, 128, 100, 50, 1, 1, 1, 1, 1, 1 << 20)  # ctx > stride
    with pytest.raises(binding.QwError):
        binding.decode_attention(2, 12, 2, 128, 10, 64, 16, 16, 16, 16, 16, 8)   # workspace small
    with pytest.raises(binding.QwError):
        binding.decode_attention(1, 12, 2, 128, 10, 64, 16, 16, 16, 16, 16, 1 << 20)  # bf16 KV
