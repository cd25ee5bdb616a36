"""GPU parity of masked decode against the fp64 oracle, through the C ABI: the 2-D bool mask
on single-token decode (decode_attn_paged_masked) and the packed 3-D mask together with the
causal rule of multi-token decode (decode_attn_paged_multi with a mask).

Element by element: |gpu - oracle| <= 1e-2 + 1e-2 * |oracle| (AstrAI csrc log, numerics
commit: atol = rtol = 0.01).  The caches are poisoned (NaN) past every sequence's end and in
unused pages, so a key read outside a sequence shows up as NaN.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_298_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_close(out: torch.Tensor, ref: np.ndarray, what=""):
    got = out.detach().float().cpu().double().numpy()
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, f"{what}: worst at {i}: gpu {got[i]} oracle {ref[i]}"


def make_mask(rows, width, seed, p_keep=0.5, stride=None):
    """uint8 [rows, width] view of a [rows, stride] buffer (stride a multiple of 16)."""
    stride = stride or (width + 15) // 16 * 16
    g = torch.Generator().manual_seed(seed)
    full = (torch.rand((rows, stride), generator=g) < p_keep).to(torch.uint8)
    return full, full[:, :width]


def oracle_masked(case, mask):
    return oracle.decode_paged_masked(bits(case.q), bits(case.k_cache), bits(case.v_cache),
                                      case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(),
                                      mask.cpu().numpy(), case.scale)


def gpu_masked(case, mask, S=0, **kw):
    return binding.decode_attn_paged_masked(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                            mask, max_kv_len=case.max_kv_len, scale=case.scale, num_splits=S, **kw)


@pytest.fixture(autouse=True)
def _clean_errors():
    binding.get_device_errors(clear=True)
    yield


SHAPES = [
    # B, Hq, Hkv, D, ps, lens
    (3, 8, 8, 128, 16, [1, 33, 64]),           # G=1
    (4, 16, 8, 64, 32, [65, 130, 9, 500]),     # G=2
    (3, 32, 8, 128, 16, [257, 1000, 17]),      # G=4
    (2, 64, 8, 128, 64, [128, 777]),           # G=8
    (3, 16, 4, 256, 16, [300, 17, 64]),        # D=256: 32-key tiles, two key slices
    (2, 64, 8, 256, 8, [100, 513]),            # D=256, G=8, page 8
    (3, 16, 16, 32, 16, [1, 200, 65]),         # D=32: 64-byte swizzle, G=1
    (2, 32, 4, 32, 32, [700, 5]),              # D=32, G=8
    # page sizes that are not multiples of 8 (rows copied one by one into the tiles)
    (3, 32, 8, 128, 12, [257, 1000, 17]),      # G=4, page 12
    (2, 16, 4, 256, 5, [300, 64]),             # D=256, page 5
    (2, 32, 4, 32, 3, [700, 5]),               # D=32, page 3
    (3, 8, 8, 64, 1, [1, 33, 64]),             # D=64, page 1
]


@pytest.mark.parametrize("B,Hq,Hkv,D,ps,lens", SHAPES)
def test_masked_parity(B, Hq, Hkv, D, ps, lens):
    case = inputs.make_paged_case(B, Hq, Hkv, D, ps, lens, 6100 + Hq + D).to("cuda")
    full, mask = make_mask(B, max(lens), 6101 + D)
    ref = oracle_masked(case, full)
    dm = full.cuda()
    for S in [0, 1, 3]:
        assert_close(gpu_masked(case, dm, S), ref, f"G={Hq // Hkv} D={D} S={S}")
    assert binding.get_device_errors() == 0


def test_all_ones_mask_is_plain_decode_and_empty_mask_gives_zeros():
    case = inputs.make_paged_case(3, 32, 8, 128, 16, [300, 45, 1200], 6200).to("cuda")
    ones = torch.ones((3, 1216), dtype=torch.uint8, device="cuda")
    plain = binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                      max_kv_len=case.max_kv_len, num_splits=3)
    got = gpu_masked(case, ones, 3)
    assert torch.allclose(got.float(), plain.float(), atol=ATOL, rtol=RTOL)
    zero_row = ones.clone()
    zero_row[1] = 0
    out = gpu_masked(case, zero_row, 2)
    assert (out[1].float() == 0).all()
    assert_close(out, oracle_masked(case, zero_row.cpu()), "one sequence fully masked")


def test_bool_mask_with_wide_rows():
    case = inputs.make_paged_case(2, 16, 4, 128, 16, [90, 400], 6300).to("cuda")
    g = torch.Generator().manual_seed(6301)
    full = torch.rand((2, 512), generator=g) < 0.3    # a bool mask, rows of 512 bytes
    ref = oracle_masked(case, full.to(torch.uint8))
    assert_close(gpu_masked(case, full.cuda(), 2), ref, "bool mask")


def test_full_size_ragged_with_mask():
    """The benchmark's masked workload (the ragged batch, 90% of keys kept) at its launch
    configuration; every output element against the oracle."""
    case = inputs.ragged_paged(device="cuda")
    full, _ = make_mask(case.B, case.max_kv_len, 6400, p_keep=0.9)
    out = gpu_masked(case, full.cuda(), 0, total_kv=case.total_kv)
    assert_close(out, oracle_masked(case, full), "full size")
    assert binding.get_device_errors() == 0


# ---- multi-token decode with a mask ---------------------------------------------------

@pytest.mark.parametrize("Hq,Hkv,D,qlens,ps", [(8, 2, 64, [5, 1, 9], 16), (32, 8, 128, [4, 4, 2], 16),
                                               (16, 2, 128, [3, 2, 1], 16), (16, 4, 256, [5, 1, 7], 16),
                                               (64, 8, 32, [2, 1, 2], 16), (32, 8, 128, [4, 4, 2], 12),
                                               (16, 4, 256, [5, 1, 7], 3), (64, 8, 128, [16, 9, 3], 16),
                                               (64, 8, 128, [16, 9, 3], 5), (8, 8, 64, [30, 1, 17], 8)])
def test_multi_token_mask_with_causal_rule(Hq, Hkv, D, qlens, ps):
    lens = [100, 37, 300]
    case = inputs.make_multi_case(3, Hq, Hkv, D, ps, lens, qlens, 6500 + Hq).to("cuda")
    kv = case.kv
    full, _ = make_mask(case.total_q, max(lens), 6501 + D, p_keep=0.6)
    qi = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    ref = oracle.decode_paged_multi(bits(case.q), bits(kv.k_cache), bits(kv.v_cache), kv.block_table.cpu().numpy(),
                                    kv.seq_lens.cpu().numpy(), qi, kv.scale, mask=full.numpy())
    # a mask rides with 16-column tiles and, at D 64, 128 and 256, with 128-row tiles
    G = Hq // Hkv
    for tpt in [16 // G] + ([128 // G] if D in (64, 128, 256) else []):
        plan = binding.MultiPlan(case.q_lens, kv.Hq, kv.Hkv, "cuda", tokens_per_tile=tpt)
        for S in [1, 3]:
            got = binding.decode_attn_paged_multi(case.q, kv.k_cache, kv.v_cache, kv.block_table, kv.seq_lens, plan,
                                                  max_kv_len=kv.max_kv_len, scale=kv.scale, num_splits=S,
                                                  mask=full.cuda())
            assert_close(got, ref, f"G={G} tpt={tpt} S={S}")
    assert binding.get_device_errors() == 0


def test_full_size_multi_token_mask_in_128_row_tiles():
    """The G = 8 speculative-verification batch (B=128, q_len 8, ragged lengths) with a
    random 3-D mask (70% kept), in 128-row tiles at the planner's split count: every output
    element against the oracle."""
    case = inputs.spec_verify_paged(device="cuda", q_len=8, Hq=64)
    kv = case.kv
    full, _ = make_mask(case.total_q, kv.max_kv_len, 6600, p_keep=0.7)
    qi = np.concatenate([[0], np.cumsum(case.q_lens)]).astype(np.int32)
    ref = oracle.decode_paged_multi(bits(case.q), bits(kv.k_cache), bits(kv.v_cache), kv.block_table.cpu().numpy(),
                                    kv.seq_lens.cpu().numpy(), qi, kv.scale, mask=full.numpy())
    plan = binding.MultiPlan(case.q_lens, 64, 8, "cuda", D=128)
    assert plan.tokens_per_tile == 16
    got = binding.decode_attn_paged_multi(case.q, kv.k_cache, kv.v_cache, kv.block_table, kv.seq_lens, plan,
                                          max_kv_len=kv.max_kv_len, scale=kv.scale, num_splits=0,
                                          total_kv=kv.total_kv, mask=full.cuda())
    assert_close(got, ref, "full size, G=8 q_len=8, mask")
    assert binding.get_device_errors() == 0
