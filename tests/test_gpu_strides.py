"""Strided layouts through the C ABI: the attention entry points read Q, K, V
and write O through {batch, head, row} element strides, so a packed QKV
tensor [B][S][3][H][D] is attended without a copy (the FastVideo compare
view's minimax_h3_prefix.cu accepts any layout whose last dimension is
contiguous).  Each case is checked against the oracle on contiguous copies,
and the memory around a strided output is checked to be untouched."""

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import attention as OA

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


def assert_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    bad = np.abs(got - ref) > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance"


def test_dense_packed_qkv_into_token_major_output(gb):
    B, H, S, D = 2, 3, 300, 128                      # ragged tail: 300 = 2 tiles + 44 rows
    rng = np.random.default_rng(61)
    qkv = rng.standard_normal((B, S, 3, H, D)).astype(np.float16)
    dq = torch.from_numpy(qkv).cuda()
    q, k, v = (dq[:, :, i].permute(0, 2, 1, 3) for i in range(3))   # [B, H, S, D] views
    assert q.stride() == (S * 3 * H * D, D, 3 * H * D, 1)
    # output token-major [B, S, H, D] inside a larger buffer with guard bands
    guard = 4096
    buf = torch.full((guard + B * S * H * D + guard,), 7.0, dtype=torch.float16, device="cuda")
    o = buf[guard:guard + B * S * H * D].view(B, S, H, D).permute(0, 2, 1, 3)
    gb.attn_dense_fwd(q, k, v, o=o)
    torch.cuda.synchronize()
    hq, hk, hv = (np.ascontiguousarray(qkv[:, :, i].transpose(0, 2, 1, 3)) for i in range(3))
    ro, _ = OA.dense_attention(hq, hk, hv, inputs.softmax_scale(D))
    assert_close(o.float().cpu().numpy(), ro, "packed qkv")
    g = buf.cpu()
    assert torch.all(g[:guard] == 7.0) and torch.all(g[-guard:] == 7.0)
    assert gb.device_status() == 0


def test_dense_strided_equals_contiguous_bit_for_bit(gb):
    q, k, v = (torch.from_numpy(x).cuda() for x in inputs.dense_inputs(1, 4, 512, 128, seed=62))
    ref = gb.attn_dense_fwd(q, k, v)
    # the same tensors stored with padded rows (row stride 192 elements)
    def padded(x):
        big = torch.zeros((x.shape[0], x.shape[1], x.shape[2], 192), dtype=x.dtype, device="cuda")
        big[..., :128] = x
        return big[..., :128]
    got = gb.attn_dense_fwd(padded(q), padded(k), padded(v))
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


@pytest.mark.parametrize("split", [False, True])
def test_causal_token_major_layouts(gb, split):
    B, Hq, Hkv, Qp, q_real, KV, D = 2, 6, 2, 192, 170, 1056, 256
    q, k, v = inputs.causal_inputs(B, Hq, Hkv, Qp, KV, D, seed=63)
    # token-major storage [B, S, H, D], passed as [B, H, S, D] views
    tq = torch.from_numpy(np.ascontiguousarray(q.transpose(0, 2, 1, 3))).cuda().permute(0, 2, 1, 3)
    tk = torch.from_numpy(np.ascontiguousarray(k.transpose(0, 2, 1, 3))).cuda().permute(0, 2, 1, 3)
    tv = torch.from_numpy(np.ascontiguousarray(v.transpose(0, 2, 1, 3))).cuda().permute(0, 2, 1, 3)
    o = torch.full((B, Qp, Hq, D), 3.0, dtype=torch.float16, device="cuda").permute(0, 2, 1, 3)
    gb.attn_causal_prefill_fwd(tq, tk, tv, q_real=q_real, o=o, prob_split=split)
    torch.cuda.synchronize()
    ro, _ = OA.causal_prefill_attention(q, k, v, inputs.softmax_scale(D), q_real)
    got = o.float().cpu().numpy()
    assert_close(got, ro, "causal token-major")
    assert np.all(got[:, :, q_real:] == 0)
    assert gb.device_status() == 0
