"""GPU parity of the paged GQA decode over an e4m3 K/V cache, and of its fp8 append,
against the fp64 oracle, through the C ABI.

Decode: element by element, |gpu - oracle| <= 1e-2 + 1e-2 * |oracle| (AstrAI csrc log,
numerics commit: atol = rtol = 0.01).  Unused pages and rows past every sequence's end hold
the e4m3 NaN code and NaN factors, so any read outside the attended rows shows up as NaN.
Append: codes and factors bit for bit.
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


def oracle_fp8kv(case):
    return oracle.decode_paged_fp8kv(bits(case.q), case.k_codes.cpu().numpy(), case.v_codes.cpu().numpy(),
                                     bits(case.k_scale), bits(case.v_scale), case.block_table.cpu().numpy(),
                                     case.seq_lens.cpu().numpy(), case.scale)


def gpu_fp8kv(case, S=0, **kw):
    return binding.decode_attn_paged_fp8kv(case.q, case.k_codes, case.v_codes, case.k_scale, case.v_scale,
                                           case.block_table, case.seq_lens, max_kv_len=case.max_kv_len,
                                           scale=case.scale, num_splits=S, **kw)


@pytest.fixture(autouse=True)
def _clean_errors():
    binding.get_device_errors(clear=True)
    yield


SHAPES = [
    # B, Hq, Hkv, ps, lens
    (3, 8, 8, 16, [1, 33, 64]),             # G=1
    (4, 16, 8, 8, [65, 130, 0, 500]),       # G=2, page 8, an empty sequence
    (3, 32, 8, 16, [257, 1000, 17]),        # G=4
    (2, 64, 8, 64, [128, 777]),             # G=8, page 64
    (5, 16, 2, 32, [1, 2, 63, 64, 65]),     # G=8, lengths around one tile
    (3, 12, 3, 16, [40, 300, 129]),         # G=4, odd kv head count: one kv head per CTA
    (2, 8, 1, 256, [1000, 257]),            # one kv head, 256-token pages
    (3, 16, 4, 48, [100, 47, 400]),         # page 48: boxes of 16 rows
]


@pytest.mark.parametrize("B,Hq,Hkv,ps,lens", SHAPES)
def test_parity_across_groups_pages_and_splits(B, Hq, Hkv, ps, lens):
    case = inputs.make_fp8kv_case(B, Hq, Hkv, 128, ps, lens, 5100 + Hq + ps).to("cuda")
    ref = oracle_fp8kv(case)
    for S in [0, 1, 3, 7, 20]:
        assert_close(gpu_fp8kv(case, S), ref, f"G={Hq // Hkv} ps={ps} S={S}")
    assert binding.get_device_errors() == 0


# head dims 64 and 256 (64-byte lines with the 64-byte swizzle; two 128-byte line blocks,
# one kv head per CTA), and page sizes that are not multiples of 8 (rows copied one by one,
# factors stored by the producer), at every head dim
OTHER = [
    # B, Hq, Hkv, D, ps, lens
    (3, 32, 8, 64, 16, [257, 1000, 17]),      # D=64, kv-head pairs
    (3, 12, 3, 64, 8, [40, 300, 129]),        # D=64, odd kv head count
    (2, 64, 8, 256, 16, [128, 777]),          # D=256, G=8
    (4, 16, 8, 256, 32, [65, 130, 0, 500]),   # D=256, G=2, an empty sequence
    (3, 32, 8, 128, 12, [257, 1000, 17]),     # page 12
    (2, 8, 1, 128, 1, [100, 3]),              # page 1, one kv head
    (3, 16, 4, 64, 5, [100, 47, 400]),        # D=64, page 5
    (3, 12, 3, 256, 3, [40, 300, 129]),       # D=256, page 3
    (5, 16, 2, 128, 100, [1, 2, 63, 64, 650]),  # page 100, lengths around one tile
]


@pytest.mark.parametrize("B,Hq,Hkv,D,ps,lens", OTHER, ids=[f"D{o[3]}_ps{o[4]}_G{o[1] // o[2]}" for o in OTHER])
def test_head_dims_64_256_and_any_page_size(B, Hq, Hkv, D, ps, lens):
    case = inputs.make_fp8kv_case(B, Hq, Hkv, D, ps, lens, 5300 + D + ps).to("cuda")
    ref = oracle_fp8kv(case)
    for S in [0, 1, 3, 7]:
        assert_close(gpu_fp8kv(case, S), ref, f"D={D} ps={ps} S={S}")
    assert binding.get_device_errors() == 0


def test_row_gather_page_permutation_and_bad_page_id():
    """Page size 12: the same bits under a permutation of the physical pages; a page id
    outside the pool is read as page 0 and flagged."""
    case = inputs.make_fp8kv_case(4, 32, 8, 128, 12, [700, 33, 1024, 260], 5400).to("cuda")
    P = case.k_codes.shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(7)).cuda()
    inv = torch.argsort(perm)
    table = inv[case.block_table.long()].to(torch.int32).contiguous()
    for S in [0, 1, 5]:
        a = gpu_fp8kv(case, S)
        b = binding.decode_attn_paged_fp8kv(case.q, case.k_codes[perm].contiguous(), case.v_codes[perm].contiguous(),
                                            case.k_scale[perm].contiguous(), case.v_scale[perm].contiguous(), table,
                                            case.seq_lens, max_kv_len=case.max_kv_len, scale=case.scale,
                                            num_splits=S)
        assert torch.equal(a, b), f"S={S}"
    assert binding.get_device_errors() == 0
    bad = case.block_table.clone()
    bad[1, 0] = P + 3
    fixed = bad.clone()
    fixed[1, 0] = 0
    kw = dict(max_kv_len=case.max_kv_len, scale=case.scale, num_splits=1)
    out = binding.decode_attn_paged_fp8kv(case.q, case.k_codes, case.v_codes, case.k_scale, case.v_scale, bad,
                                          case.seq_lens, **kw)
    torch.cuda.synchronize()
    assert binding.get_device_errors(clear=True) & binding.DEVERR_PAGE
    want = binding.decode_attn_paged_fp8kv(case.q, case.k_codes, case.v_codes, case.k_scale, case.v_scale, fixed,
                                           case.seq_lens, **kw)
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))
    assert binding.get_device_errors(clear=True) == 0


def test_wide_factor_range_and_q_beyond_f16():
    # factors spread over 2^-6 .. 2^7 within every page; q times 2^16 (most elements beyond
    # f16's range before the kernel's power-of-two shift) with the softmax scale divided by
    # 2^16, so the attention itself is unchanged
    case = inputs.make_fp8kv_case(3, 32, 8, 128, 16, [300, 45, 1200], 5200)
    g = torch.Generator().manual_seed(5201)
    for f in (case.k_scale, case.v_scale):
        e = torch.randint(-6, 7, f.shape, generator=g).float()
        f.copy_((torch.pow(2.0, e) * (1 + torch.rand(f.shape, generator=g))).to(torch.bfloat16))
    case.q.mul_(2.0 ** 16)
    case.scale = case.scale / 2.0 ** 16
    assert case.q.float().abs().max() > 65504
    case = case.to("cuda")
    ref = oracle_fp8kv(case)
    for S in [1, 4]:
        assert_close(gpu_fp8kv(case, S), ref, f"S={S}")


def test_every_sequence_empty_gives_zero_rows():
    case = inputs.make_fp8kv_case(3, 16, 4, 128, 16, [0, 0, 0], 5250).to("cuda")
    for S in [1, 3]:
        out = torch.full_like(case.q, 5.0)
        binding.decode_attn_paged_fp8kv(case.q, case.k_codes, case.v_codes, case.k_scale, case.v_scale,
                                        case.block_table, case.seq_lens, max_kv_len=16, num_splits=S, out=out)
        assert (out.float() == 0).all(), f"S={S}"
    assert binding.get_device_errors() == 0


def test_strided_q_and_out():
    case = inputs.make_fp8kv_case(2, 16, 4, 128, 16, [90, 400], 5300).to("cuda")
    big_q = torch.zeros(2, 24, 136, dtype=torch.bfloat16, device="cuda")
    big_q[:, :16, :128] = case.q
    out_big = torch.full((2, 20, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    out = out_big[:, 2:18, 64:192]
    binding.decode_attn_paged_fp8kv(big_q[:, :16, :128], case.k_codes, case.v_codes, case.k_scale, case.v_scale,
                                    case.block_table, case.seq_lens, max_kv_len=case.max_kv_len, num_splits=2,
                                    out=out)
    assert_close(out, oracle_fp8kv(case), "strided")
    assert (out_big[:, :2] == 7).all() and (out_big[:, :, :64] == 7).all()


def test_page_permutation_is_bit_identical():
    case = inputs.make_fp8kv_case(3, 32, 8, 128, 16, [100, 513, 64], 5400, poison=False)
    P = case.k_codes.shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(5401))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    moved = inputs.Fp8KvCase(case.q, case.k_codes[perm], case.v_codes[perm], case.k_scale[perm],
                             case.v_scale[perm], inv[case.block_table.long()].to(torch.int32), case.seq_lens,
                             case.page_size, case.scale)
    a = gpu_fp8kv(case.to("cuda"), 3)
    b = gpu_fp8kv(moved.to("cuda"), 3)
    assert torch.equal(a, b)


def test_full_size_ragged_batch():
    """The ragged B=128 batch over an e4m3 cache, the planner's split count made with the
    summed lengths (the benchmark's launch) and without them; every output element against
    the oracle."""
    case = inputs.ragged_fp8kv(device="cuda")
    ref = oracle_fp8kv(case)
    assert_close(gpu_fp8kv(case, 0, total_kv=case.total_kv), ref, "full size, benchmark launch")
    assert_close(gpu_fp8kv(case, 0), ref, "full size, S resolved by the library")
    assert binding.get_device_errors() == 0


def test_out_of_range_page_is_flagged():
    case = inputs.make_fp8kv_case(2, 16, 4, 128, 16, [40, 40], 5500).to("cuda")
    case.block_table[1, 1] = 10 ** 6
    gpu_fp8kv(case, 1)
    torch.cuda.synchronize()
    assert binding.get_device_errors() & binding.DEVERR_PAGE


# ---- fp8 append for the GQA cache ------------------------------------------------------

@pytest.mark.parametrize("D", [64, 128, 256])
def test_append_paged_fp8_is_bit_exact(D):
    case = inputs.make_fp8kv_case(4, 8, 2, D, 16, [16, 5, 31, 0], 5600 + D, poison=False)
    g = torch.Generator().manual_seed(5601)
    k_new = (inputs.randn_bf16((4, 2, D), g, "cpu").float() *
             torch.tensor([1.0, 30.0, 1e-3, 0.0])[:, None, None]).to(torch.bfloat16)
    v_new = inputs.randn_bf16((4, 2, D), g, "cpu")
    pos = case.seq_lens.clone()
    kc, vc = case.k_codes.numpy().copy(), case.v_codes.numpy().copy()
    ks, vs = bits(case.k_scale).copy(), bits(case.v_scale).copy()
    assert oracle.kv_append_paged_fp8(bits(k_new), bits(v_new), kc, vc, ks, vs, case.block_table.numpy(),
                                      pos.numpy()) == 0
    d = case.to("cuda")
    binding.kv_append_paged_fp8(k_new.cuda(), v_new.cuda(), d.k_codes, d.v_codes, d.k_scale, d.v_scale,
                                d.block_table, pos.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(d.k_codes.cpu().numpy(), kc) and np.array_equal(d.v_codes.cpu().numpy(), vc)
    assert np.array_equal(bits(d.k_scale), ks) and np.array_equal(bits(d.v_scale), vs)
    assert binding.get_device_errors() == 0


def test_append_then_decode_round_trip():
    # decode after appending one token per sequence equals the oracle on the grown cache
    case = inputs.make_fp8kv_case(3, 32, 8, 128, 16, [40, 127, 300], 5700, poison=False)
    g = torch.Generator().manual_seed(5701)
    k_new = inputs.randn_bf16((3, 8, 128), g, "cpu").cuda()
    v_new = inputs.randn_bf16((3, 8, 128), g, "cpu").cuda()
    d = case.to("cuda")
    binding.kv_append_paged_fp8(k_new, v_new, d.k_codes, d.v_codes, d.k_scale, d.v_scale, d.block_table,
                                d.seq_lens.clone())
    grown = inputs.Fp8KvCase(d.q, d.k_codes, d.v_codes, d.k_scale, d.v_scale, d.block_table, d.seq_lens + 1,
                             d.page_size, d.scale)
    assert_close(gpu_fp8kv(grown, 2), oracle_fp8kv(grown), "grown")
