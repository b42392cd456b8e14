"""GPU parity of the paged E4M3 decode against the CPU oracle.

The decode kernel reads the E4M3 pages itself and must see exactly the
bridge's FP16 values; its outputs satisfy |o - ref| <= 2e-3 + 1e-2 |ref| (and
the same for lse) element by element against the float64 oracle.  Cases cover
ragged lengths (one token, one stage, a ragged last stage, several chunks),
several new tokens per sequence (causal among them, several query-row groups),
shared-KV head ratios, both head widths, page sizes 16..256, the three scale
paths (power of two, FP16-valued, general FP32), NaN codes past the cache end,
full and reduced workspaces (fewer warps, longer ranges), bad page-table
entries and lengths, and the full 4-sequence workload the benchmark times.
"""

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import decode as OD

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2
DEV = "cuda"


def t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    excess = np.where(both_inf, -1.0, np.abs(got - ref) - (ATOL + RTOL * np.abs(ref)))
    bad = int((excess > 0).sum())
    assert bad == 0, f"{what}: {bad} of {excess.size} outside tolerance, max excess {excess.max():.3e}"


def run(gb, q, kp, vp, table, lens, ks, vs, scale=None, workspace="auto", max_kv=None):
    B, Hq, nq, D = q.shape
    lse = torch.empty((B, Hq, nq), dtype=torch.float32, device=DEV)
    ws = None if workspace == "auto" else torch.empty(max(int(workspace), 16), dtype=torch.uint8,
                                                      device=DEV)
    o = gb.attn_paged_decode_fwd(t(q), t(kp), t(vp), t(table), t(lens), ks, vs,
                                 max_kv_len=max_kv, lse=lse, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(gb, B, Hq, Hkv, nq, lens, D=256, ps=32, ks=0.0625, vs=0.125, codes="moderate", seed=7,
          workspace="auto", spare=0, poison_tail=False, max_kv=None):
    q, kp, vp, table, lens = inputs.paged_decode_inputs(B, Hq, Hkv, nq, lens, D, seed,
                                                        page_size=ps, spare_pages=spare,
                                                        codes=codes)
    if poison_tail:   # NaN codes in every slot past each cache end
        for b, n in enumerate(lens):
            if n % ps:
                kp[table[b, (n - 1) // ps], n % ps:] = 0x7F
                vp[table[b, (n - 1) // ps], n % ps:] = 0xFF
    scale = inputs.softmax_scale(D)
    o, lse = run(gb, q, kp, vp, table, lens, ks, vs, scale, workspace, max_kv)
    ro, rl = OD.paged_decode_attention(q, kp, vp, table, lens, ks, vs, scale)
    assert gb.device_status() == 0
    assert_close(o, ro, "o")
    assert_close(lse, rl, "lse")
    return o


@pytest.mark.parametrize("lens", [(1, 64, 1000, 4097), (63, 65, 129, 3000), (2048,)])
def test_decode_ragged_lengths(gb, lens):
    check(gb, len(lens), 6, 1, 1, lens)


@pytest.mark.parametrize("codes", ["finite", "moderate"])
def test_decode_code_distributions(gb, codes):
    check(gb, 2, 6, 1, 1, (5000, 777), codes=codes, seed=8)


@pytest.mark.parametrize("nq", [2, 3, 4])
def test_decode_several_new_tokens(gb, nq):
    check(gb, 2, 6, 1, nq, (900, 1537), seed=9)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (16, 4), (4, 4), (32, 1)])
def test_decode_shared_kv_heads(gb, Hq, Hkv):
    check(gb, 2, Hq, Hkv, 1, (700, 1301), seed=10)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("ps", [16, 64, 128, 256])
def test_decode_page_sizes_and_widths(gb, D, ps):
    check(gb, 2, 6, 2 if D == 128 else 1, 2, (1000, 333), D=D, ps=ps, seed=11, spare=3)


@pytest.mark.parametrize("ks,vs", [
    (0.0625, 0.125),                                         # powers of two (folded)
    (float(np.float16(0.3)), float(np.float16(0.7))),        # FP16 values
    (1 / 3, 0.3),                                            # general FP32
    (2.0 ** -15, 2.0 ** 7),                                  # folding range ends
    (2.0 ** -16, 2.0 ** 8)])                                 # just outside it
def test_decode_scale_paths(gb, ks, vs):
    check(gb, 2, 6, 1, 1, (1500, 430), ks=ks, vs=vs, seed=12)


def test_decode_nan_codes_past_the_cache_end(gb):
    check(gb, 3, 6, 1, 2, (37, 1000, 65), poison_tail=True, seed=13)


def test_decode_smaller_workspace_fewer_warps(gb):
    """A workspace below the full plan runs fewer warps (longer ranges); too small is an error."""
    full = gb.attn_paged_decode_workspace_size(2, 6, 1, 1, 6016, 256)
    many = check(gb, 2, 6, 1, 1, (6000, 2500), seed=14)
    few = check(gb, 2, 6, 1, 1, (6000, 2500), seed=14, workspace=full // 5)
    one = check(gb, 2, 6, 1, 1, (6000, 2500), seed=14, workspace=full // 100)
    assert np.abs(many - few).max() < 2e-3 and np.abs(many - one).max() < 2e-3
    with pytest.raises(gb.GbattnError):
        check(gb, 2, 6, 1, 1, (6000, 2500), seed=14, workspace=16)


def test_decode_loose_length_bound(gb):
    """max_kv_len well above the real lengths (the default: the table's span)."""
    check(gb, 2, 6, 1, 1, (300, 2000), seed=15, max_kv=None)
    check(gb, 2, 6, 1, 1, (300, 2000), seed=15, max_kv=2000)


def test_decode_bad_page_and_length_flags(gb):
    q, kp, vp, table, lens = inputs.paged_decode_inputs(2, 6, 1, 1, (500, 300), 256, 16,
                                                        codes="moderate")
    bad = table.copy()
    bad[0, 3] = kp.shape[0] + 5
    run(gb, q, kp, vp, bad, lens, 0.0625, 0.125)
    assert gb.device_status() & gb.DEV_BAD_PAGE
    lens2 = np.array([500, 0], dtype=np.int32)            # shorter than nq: rejected
    full = gb.attn_paged_decode_workspace_size(2, 6, 1, 1, 512, 256)
    for ws in ("auto", full // 50):
        o, lse = run(gb, q, kp, vp, table, lens2, 0.0625, 0.125, workspace=ws, max_kv=512)
        assert gb.device_status() & gb.DEV_BAD_LENGTH
        assert np.all(o[1] == 0) and np.all(np.isneginf(lse[1]))
        ro, _ = OD.paged_decode_attention(q[:1], kp, vp, table[:1], lens2[:1], 0.0625, 0.125,
                                          inputs.softmax_scale(256))
        assert_close(o[:1], ro, "valid sequence next to a rejected one")
    lens3 = np.array([500, 513], dtype=np.int32)          # above max_kv_len
    run(gb, q, kp, vp, table, lens3, 0.0625, 0.125, max_kv=512)
    assert gb.device_status() & gb.DEV_BAD_LENGTH


def test_decode_deterministic(gb):
    q, kp, vp, table, lens = inputs.paged_decode_inputs(3, 6, 1, 1, (4000, 100, 2345), 256, 17)
    a, la = run(gb, q, kp, vp, table, lens, 0.0625, 0.125)
    b, lb = run(gb, q, kp, vp, table, lens, 0.0625, 0.125)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_decode_full_workload(gb):
    """The benchmark's launch: 4 sequences, 65571..131072 cached tokens, every row."""
    w = inputs.WORKLOADS["paged_decode"]
    q, kp, vp, table, lens = inputs.paged_decode_inputs(w["B"], w["Hq"], w["Hkv"], w["nq"],
                                                        w["kv_lens"], w["D"], w["seed"],
                                                        w["page_size"])
    scale = inputs.softmax_scale(w["D"])
    o, lse = run(gb, q, kp, vp, table, lens, w["k_scale"], w["v_scale"], scale,
                 max_kv=max(w["kv_lens"]))
    assert gb.device_status() == 0
    ro, rl = OD.paged_decode_attention(q, kp, vp, table, lens, w["k_scale"], w["v_scale"], scale)
    assert_close(o, ro, "o")
    assert_close(lse, rl, "lse")
