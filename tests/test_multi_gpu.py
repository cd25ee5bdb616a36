"""GPU parity of the multi-token causal decode (packed new tokens per sequence, work map of
q tiles) against the fp64 oracle, through the C ABI.

Element by element: |gpu - oracle| <= 1e-2 + 1e-2 * |oracle| on the bf16 output (AstrAI
csrc log, numerics commit: atol = rtol = 0.01).  The caches are poisoned (NaN) past every
sequence's end and in every unused page, so a key read past a token's causal limit or
outside its sequence turns into a non-finite output.
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


def oracle_multi(case: inputs.MultiCase):
    kv = case.kv
    qi = np.concatenate([[0], np.cumsum(case.q_lens)]).astype(np.int32)
    return oracle.decode_paged_multi(bits(case.q), bits(kv.k_cache), bits(kv.v_cache), kv.block_table.cpu().numpy(),
                                     kv.seq_lens.cpu().numpy(), qi, kv.scale)


def gpu_multi(case: inputs.MultiCase, S=0, plan=None, **kw):
    kv = case.kv
    if plan is None:
        plan = binding.MultiPlan(case.q_lens, kv.Hq, kv.Hkv, case.q.device, D=kv.D)
    return binding.decode_attn_paged_multi(case.q, kv.k_cache, kv.v_cache, kv.block_table, kv.seq_lens, plan,
                                           max_kv_len=kv.max_kv_len, scale=kv.scale, num_splits=S, **kw)


@pytest.fixture(autouse=True)
def _clean_errors():
    binding.get_device_errors(clear=True)
    yield


def tile_sizes(Hq, Hkv, D=None):
    """Every tile size of the work map: 16 and 32 query columns, and 128 query rows of the
    tensor-memory tiles where the head dim has them (64, 128 and 256)."""
    G = Hq // Hkv
    return [16 // G, 32 // G] + ([128 // G] if D in (64, 128, 256) else [])


def test_small_case_several_tiles_and_split_counts():
    # G = 4: 4 (or 8) tokens per q tile; 9 new tokens -> three (two) tiles, the last ragged
    case = inputs.make_multi_case(3, 8, 2, 64, 16, [100, 37, 300], [5, 1, 9], 4001).to("cuda")
    ref = oracle_multi(case)
    for tpt in tile_sizes(8, 2, 64):
        plan = binding.MultiPlan(case.q_lens, 8, 2, "cuda", tokens_per_tile=tpt)
        for S in [0, 1, 2, 3, 5]:
            assert_close(gpu_multi(case, S, plan=plan), ref, f"tpt={tpt} S={S}")
    assert binding.get_device_errors() == 0


SHAPES = [
    # B, Hq, Hkv, D, ps, kv lens, q lens
    (3, 8, 8, 128, 16, [20, 200, 64], [16, 17, 3]),            # G=1: 16 tokens per tile
    (4, 16, 8, 64, 32, [65, 130, 9, 500], [8, 0, 9, 2]),       # G=2, a sequence with no new token
    (2, 32, 8, 128, 16, [257, 1000], [4, 13]),                 # G=4, tile edges at 4
    (3, 64, 8, 128, 64, [128, 1, 777], [2, 1, 7]),              # G=8: 2 tokens per tile, L = q_len
    (2, 16, 2, 64, 8, [300, 64], [30, 64]),                     # G=8, D=64, every key new
    (3, 16, 4, 256, 16, [300, 17, 64], [9, 3, 5]),              # D=256 (32-key tiles), G=4
    (2, 64, 8, 256, 8, [100, 513], [3, 6]),                      # D=256, G=8, page 8
    (3, 16, 16, 32, 16, [1, 200, 65], [1, 20, 33]),              # D=32 (64-byte swizzle), G=1
    (2, 32, 4, 32, 32, [700, 5], [11, 5]),                       # D=32, G=8
    # page sizes that are not multiples of 8 (rows copied one by one into the tiles)
    (3, 32, 8, 128, 12, [257, 1000, 5], [4, 13, 5]),            # G=4, page 12
    (2, 64, 8, 128, 5, [128, 333], [2, 7]),                      # G=8, page 5
    (2, 16, 4, 256, 3, [300, 64], [9, 5]),                       # D=256, page 3
    (2, 32, 4, 32, 1, [200, 65], [11, 5]),                       # D=32, page 1
    (3, 16, 8, 64, 100, [650, 9, 301], [8, 9, 2]),               # D=64, page 100
    # the tensor-memory tiles' other K/V layouts: 8-row boxes, 32-row boxes, more than one
    # 128-row tile per sequence
    (2, 32, 8, 128, 8, [300, 77], [6, 40]),                      # G=4, page 8
    (3, 64, 8, 128, 32, [500, 90, 2100], [16, 9, 17]),           # G=8, page 32
    (2, 8, 8, 64, 16, [400, 150], [130, 3]),                     # G=1, D=64
]


@pytest.mark.parametrize("B,Hq,Hkv,D,ps,lens,qlens", SHAPES)
def test_parity_across_groups_and_dims(B, Hq, Hkv, D, ps, lens, qlens):
    case = inputs.make_multi_case(B, Hq, Hkv, D, ps, lens, qlens, 4100 + Hq + D).to("cuda")
    ref = oracle_multi(case)
    for tpt in tile_sizes(Hq, Hkv, D):
        plan = binding.MultiPlan(case.q_lens, Hq, Hkv, "cuda", tokens_per_tile=tpt)
        for S in [0, 1, 4]:
            assert_close(gpu_multi(case, S, plan=plan), ref, f"G={Hq // Hkv} D={D} tpt={tpt} S={S}")
    assert binding.get_device_errors() == 0


@pytest.mark.parametrize("B", [70, 1100])
def test_many_sequences_with_empty_ones(B):
    """More sequences than one 32-wide step of the combine's qo_indptr search covers (70:
    two steps; 1100: three), with runs of sequences that have no new token (repeated
    offsets), checked against the oracle on every token."""
    rng = np.random.default_rng(4700 + B)
    qlens = rng.integers(0, 4, size=B)
    qlens[rng.integers(0, B, size=B // 4)] = 0
    qlens[0] = qlens[-1] = 2
    lens = rng.integers(4, 90, size=B)
    case = inputs.make_multi_case(B, 8, 2, 64, 16, lens.tolist(), qlens.tolist(), 4700 + B).to("cuda")
    ref = oracle_multi(case)
    for S in [2, 3]:
        assert_close(gpu_multi(case, S), ref, f"B={B} S={S}")
    assert binding.get_device_errors() == 0


def test_one_new_token_each_matches_single_token_decode():
    case = inputs.make_multi_case(5, 32, 8, 128, 16, [1, 70, 129, 640, 2000], [1] * 5, 4200).to("cuda")
    kv = case.kv
    single = binding.decode_attn_paged(case.q, kv.k_cache, kv.v_cache, kv.block_table, kv.seq_lens,
                                       max_kv_len=kv.max_kv_len, num_splits=3)
    multi = gpu_multi(case, 3)
    assert_close(multi, oracle_multi(case), "q_len=1")
    assert torch.allclose(multi.float(), single.float(), atol=ATOL, rtol=RTOL)


@pytest.mark.parametrize("D", [None, 128])
def test_strided_q_and_out(D):
    # D=None: 32-column tiles; D=128: the 128-row tcgen05 tiles
    case = inputs.make_multi_case(2, 16, 4, 128, 16, [90, 400], [6, 3], 4300).to("cuda")
    big_q = torch.zeros(case.total_q, 24, 136, dtype=torch.bfloat16, device="cuda")
    big_q[:, :16, :128] = case.q
    q = big_q[:, :16, :128]
    out_big = torch.full((case.total_q, 20, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    out = out_big[:, 2:18, 64:192]
    kv = case.kv
    plan = binding.MultiPlan(case.q_lens, kv.Hq, kv.Hkv, "cuda", D=D)
    binding.decode_attn_paged_multi(q, kv.k_cache, kv.v_cache, kv.block_table, kv.seq_lens, plan,
                                    max_kv_len=kv.max_kv_len, num_splits=2, out=out)
    assert_close(out, oracle_multi(case), "strided")
    assert (out_big[:, :2] == 7).all() and (out_big[:, :, :64] == 7).all()


def test_full_size_speculative_verification():
    """The q_len=4 speculative-verification batch (B=128, ragged lengths), run with the
    launch configuration the benchmark times and with the library's own plan; the oracle
    checks every new token of every sequence, every head and dim."""
    case = inputs.spec_verify_paged(device="cuda")
    ref = oracle_multi(case)
    out = gpu_multi(case, 0, total_kv=case.kv.total_kv)
    assert_close(out, ref, "full size, benchmark launch")
    assert_close(gpu_multi(case, 0), ref, "full size, S resolved by the library")
    assert binding.get_device_errors() == 0


@pytest.mark.parametrize("q_len", [4, 8])
def test_full_size_eight_heads_per_kv_head(q_len):
    """The ragged B=128 batch at Hq=64, Hkv=8 (G = 8) with 4 or 8 new tokens per sequence in
    32-column tiles (the head-dim-agnostic rule's choice): all of a sequence's tokens (or
    half of them, at 8) against one K/V stream; every output element against the oracle,
    at the planner's split count."""
    case = inputs.spec_verify_paged(device="cuda", q_len=q_len, Hq=64)
    plan = binding.MultiPlan(case.q_lens, 64, 8, "cuda")
    assert plan.tokens_per_tile == 4 and plan.num_tiles == 128 * (q_len // 4)
    ref = oracle_multi(case)
    assert_close(gpu_multi(case, 0, plan=plan, total_kv=case.kv.total_kv), ref, f"G=8 q_len={q_len}")
    assert binding.get_device_errors() == 0


@pytest.mark.parametrize("q_len", [4, 8, 16])
def test_full_size_eight_heads_tensor_memory_tiles(q_len):
    """The same G = 8 batch in 128-row tiles (16 tokens x 8 heads): one tile, and so one
    K/V stream, per sequence and kv head at every q_len up to 16; every output element
    against the oracle at the planner's split count and at one split."""
    case = inputs.spec_verify_paged(device="cuda", q_len=q_len, Hq=64)
    plan = binding.MultiPlan(case.q_lens, 64, 8, "cuda", D=128)
    assert plan.tokens_per_tile == 16 and plan.num_tiles == 128
    ref = oracle_multi(case)
    assert_close(gpu_multi(case, 0, plan=plan, total_kv=case.kv.total_kv), ref, f"G=8 q_len={q_len} 128 rows")
    assert_close(gpu_multi(case, 1, plan=plan), ref, f"G=8 q_len={q_len} 128 rows, one split")
    assert binding.get_device_errors() == 0


@pytest.mark.parametrize("ps", [16, 7])
def test_tensor_memory_tiles_head_dim_256(ps):
    """D = 256 in 128-row tiles (one CTA per SM, 64 KB stages, O in tensor-memory columns
    256..511), 16 tokens per sequence at G = 8, TMA boxes and the row gather, against the
    oracle at three split counts."""
    lens = [2900, 700, 65, 1800, 16, 3000]
    case = inputs.make_multi_case(6, 64, 8, 256, ps, lens, [16, 9, 16, 1, 16, 12], 4690 + ps).to("cuda")
    plan = binding.MultiPlan(case.q_lens, 64, 8, "cuda", D=256)
    assert plan.tokens_per_tile == 16
    ref = oracle_multi(case)
    for S in [0, 1, 3]:
        assert_close(gpu_multi(case, S, plan=plan), ref, f"D=256 ps={ps} S={S}")
    assert binding.get_device_errors() == 0


@pytest.mark.parametrize("S", [1, 2])
def test_tensor_memory_tiles_long_sequence(S):
    """A 20,000-key sequence in one or two splits (over 150 K/V tiles per CTA: every stage
    and buffer barrier turns many times) next to a short one, 16 tokens at G = 8."""
    case = inputs.make_multi_case(2, 64, 8, 128, 16, [20000, 70], [16, 3], 4680).to("cuda")
    plan = binding.MultiPlan(case.q_lens, 64, 8, "cuda", D=128)
    assert plan.tokens_per_tile == 16
    assert_close(gpu_multi(case, S, plan=plan), oracle_multi(case), f"long sequence, S={S}")
    assert binding.get_device_errors() == 0


def test_tensor_memory_tiles_repeat_bit_identically():
    case = inputs.make_multi_case(4, 64, 8, 128, 16, [500, 800, 90, 1500], [5, 16, 1, 9], 4650).to("cuda")
    plan = binding.MultiPlan(case.q_lens, 64, 8, "cuda", tokens_per_tile=16)
    a = gpu_multi(case, 3, plan=plan)
    b = gpu_multi(case, 3, plan=plan)
    assert torch.equal(a, b)
    assert_close(a, oracle_multi(case), "repeat")


def test_more_new_tokens_than_keys_gives_zero_rows_and_a_flag():
    # sequence 1 claims 6 new tokens but holds only 4 keys: its first two tokens would sit
    # before the cache start, attend nothing and come out zero (as in the oracle)
    case = inputs.make_multi_case(2, 8, 2, 64, 16, [50, 4], [3, 6], 4400).to("cuda")
    ref = oracle_multi(case)
    for tpt in tile_sizes(8, 2, 64):
        binding.get_device_errors(clear=True)
        plan = binding.MultiPlan(case.q_lens, 8, 2, "cuda", tokens_per_tile=tpt)
        out = gpu_multi(case, 1, plan=plan)
        torch.cuda.synchronize()
        assert binding.get_device_errors() & binding.DEVERR_SEQLEN
        assert_close(out, ref, f"q_len > L, tpt={tpt}")
        assert (out[3:5].float() == 0).all()


@pytest.mark.parametrize("tpt", [4, 32])
def test_bad_work_map_entry_is_skipped_and_flagged(tpt):
    # 4 tokens per tile: the mma.sync consumer; 32 (128 rows at G = 4): the tcgen05 one
    case = inputs.make_multi_case(2, 8, 2, 64, 16, [50, 40], [3, 2], 4500).to("cuda")
    kv = case.kv
    plan = binding.MultiPlan(case.q_lens, kv.Hq, kv.Hkv, "cuda", tokens_per_tile=tpt)
    good = gpu_multi(case, 1, plan=plan).clone()
    binding.get_device_errors(clear=True)
    plan.tile_batch[1] = 7          # names no sequence
    out = torch.zeros_like(good)
    gpu_multi(case, 1, plan=plan, out=out)
    torch.cuda.synchronize()
    assert binding.get_device_errors() & binding.DEVERR_QMAP
    assert torch.equal(out[:3], good[:3])   # the first tile is unaffected
    assert (out[3:] == 0).all()              # the skipped tile's rows are left as they were


@pytest.mark.parametrize("ps", [16, 5])
def test_tensor_memory_tiles_flag_a_bad_page_id(ps):
    """A block-table entry outside the pool is read as page 0 and flagged (TMA and row-gather
    producers of the 128-row tiles); the other sequence's rows are unaffected."""
    case = inputs.make_multi_case(2, 64, 8, 128, ps, [300, 200], [9, 4], 4750).to("cuda")
    kv = case.kv
    plan = binding.MultiPlan(case.q_lens, 64, 8, "cuda", D=128)
    assert plan.tokens_per_tile == 16
    good = gpu_multi(case, 2, plan=plan).clone()
    binding.get_device_errors(clear=True)
    kv.block_table[1, 3] = kv.num_pages + 5
    out = gpu_multi(case, 2, plan=plan)
    torch.cuda.synchronize()
    assert binding.get_device_errors() & binding.DEVERR_PAGE
    assert torch.equal(out[:9], good[:9])


def test_repeat_is_deterministic():
    case = inputs.make_multi_case(4, 32, 8, 128, 16, [500, 800, 90, 1500], [4, 4, 4, 4], 4600).to("cuda")
    a = gpu_multi(case, 3)
    b = gpu_multi(case, 3)
    assert torch.equal(a, b)
