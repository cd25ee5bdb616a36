"""GPU parity of the bf16 paged / contiguous decode kernels against the fp64 oracle.

Every comparison is element by element: |gpu - oracle| <= 1e-2 + 1e-2 * |oracle| on the bf16
output (AstrAI csrc log, numerics commit: atol = rtol = 0.01).  Integer-exact properties
(page-permutation invariance, paged == contiguous, run-to-run) are checked bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_298_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2
BAL = binding.SPLITS_BALANCED


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_close(out: torch.Tensor, ref: np.ndarray, what=""):
    got = out.detach().float().cpu().double().numpy()
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, f"{what}: worst at {i}: gpu {got[i]} oracle {ref[i]}"


def oracle_paged(case):
    return oracle.decode_paged(bits(case.q), bits(case.k_cache), bits(case.v_cache),
                               case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(), case.scale)


def gpu_paged(case, S=0, **kw):
    return binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                     max_kv_len=case.max_kv_len, scale=case.scale, num_splits=S, **kw)


@pytest.fixture(autouse=True)
def _clean_errors():
    binding.get_device_errors(clear=True)
    yield


def test_tiny_workload_all_split_counts():
    case = inputs.tiny_paged().to("cuda")
    ref = oracle_paged(case)
    for S in [BAL, 0, 1, 2, 3, 4]:
        assert_close(gpu_paged(case, S), ref, f"S={S}")
    assert binding.get_device_errors() == 0


SHAPES = [
    # B, Hq, Hkv, D, ps, lens
    (3, 8, 8, 128, 16, [1, 33, 64]),            # G=1
    (3, 16, 8, 128, 16, [5, 100, 257]),          # G=2
    (4, 32, 8, 128, 16, [256, 17, 1000, 31]),    # G=4
    (2, 64, 8, 128, 64, [300, 129]),             # G=8, page 64
    (2, 8, 1, 128, 8, [77, 200]),                # G=8, one kv head
    (3, 4, 2, 64, 16, [37, 100, 0]),             # D=64, empty sequence
    (2, 8, 2, 64, 1, [40, 9]),                   # page size 1
    (2, 16, 4, 64, 3, [50, 3]),                  # page size 3 (one-token boxes)
    (2, 32, 4, 128, 100, [250, 99]),             # page size not a power of two
    (2, 16, 2, 64, 32, [513, 64]),               # G=8, D=64
    (3, 8, 2, 256, 16, [300, 17, 64]),           # D=256 (32-token tiles, two consumer warps)
    (2, 64, 8, 256, 8, [100, 513]),              # D=256, G=8, page 8
    (3, 16, 16, 32, 16, [1, 200, 65]),           # D=32 (64-byte swizzle), G=1
    (2, 32, 4, 32, 32, [700, 5]),                # D=32, G=8
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}_Hq{s[1]}_Hkv{s[2]}_D{s[3]}_ps{s[4]}" for s in SHAPES])
def test_paged_parity(shape):
    B, Hq, Hkv, D, ps, lens = shape
    case = inputs.make_paged_case(B, Hq, Hkv, D, ps, lens, 1000 + sum(lens)).to("cuda")
    ref = oracle_paged(case)
    for S in [BAL, 0, 1, 2, 5, 20]:    # 20: more than 16 splits, the CTA-per-row combine
        assert_close(gpu_paged(case, S), ref, f"S={S}")
    assert binding.get_device_errors() == 0


def test_contiguous_matches_oracle_and_paged_bit_for_bit():
    case = inputs.make_paged_case(4, 32, 8, 128, 16, [300, 1, 64, 129], 77).to("cuda")
    k, v = inputs.logical_kv(case, max_len=320)
    ref = oracle.decode_contig(bits(case.q), bits(k), bits(v), case.seq_lens.cpu().numpy(), case.scale)
    for S in [BAL, 0, 1, 3]:
        c = binding.decode_attn_contig(case.q, k, v, case.seq_lens, max_kv_len=case.max_kv_len,
                                       num_splits=S)
        assert_close(c, ref, f"contig S={S}")
        assert torch.equal(c, gpu_paged(case, S))


def test_page_permutation_is_bit_identical():
    case = inputs.make_paged_case(5, 32, 8, 128, 16, [700, 33, 1024, 5, 260], 78).to("cuda")
    perm = torch.randperm(case.num_pages, generator=torch.Generator().manual_seed(5)).cuda()
    inv = torch.argsort(perm)
    moved = inputs.PagedCase(case.q, case.k_cache[perm].contiguous(), case.v_cache[perm].contiguous(),
                             inv[case.block_table.long()].to(torch.int32).contiguous(), case.seq_lens,
                             case.page_size, case.scale)
    for S in [BAL, 0, 1, 4, 9]:
        assert torch.equal(gpu_paged(case, S), gpu_paged(moved, S)), f"S={S}"


def test_cluster_merge_equals_the_combine_kernel_bit_for_bit():
    """2..8 splits of a one-wave grid merge inside a thread-block cluster; the same sequences
    in a batch too large for one wave merge in the combine kernel.  Same arithmetic, same
    order: the outputs agree bit for bit (and with the oracle)."""
    lens = [700, 33, 1024, 5, 260, 1]
    small = inputs.make_paged_case(6, 32, 8, 128, 16, lens, 92).to("cuda")
    reps = 120   # 720 sequences x 8 kv heads x S CTAs: several waves
    big = inputs.PagedCase(small.q.repeat(reps, 1, 1), small.k_cache, small.v_cache, small.block_table.repeat(reps, 1),
                           small.seq_lens.repeat(reps), small.page_size, small.scale)
    ref = oracle_paged(small)
    for S in [2, 3, 5, 8]:
        a = gpu_paged(small, S)
        bb = binding.decode_attn_paged(big.q, big.k_cache, big.v_cache, big.block_table, big.seq_lens,
                                       max_kv_len=small.max_kv_len, scale=small.scale, num_splits=S)
        assert torch.equal(a, bb[:6]), f"S={S}"
        assert_close(a, ref, f"S={S}")
    assert binding.get_device_errors() == 0


def test_split_count_sweep_stays_within_tolerance():
    case = inputs.make_paged_case(2, 64, 8, 128, 64, [4096, 2500], 79).to("cuda")
    ref = oracle_paged(case)
    outs = []
    for S in [1, 8, 32, 128]:
        o = gpu_paged(case, S)
        assert_close(o, ref, f"S={S}")
        outs.append(o.float())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() < 2e-2


def test_balanced_schedule_many_short_and_empty_sequences():
    # 300 sequences: the persistent CTAs' scan of seq_lens crosses many 32-wide chunks, some
    # units are empty, many CTAs cover several whole units, and ranges start mid-unit.
    lens = inputs.uniform_lengths(300, 0, 200, 84)
    lens[7] = 0
    lens[299] = 0
    case = inputs.make_paged_case(300, 8, 2, 64, 16, lens, 84).to("cuda")
    ref = oracle_paged(case)
    assert_close(gpu_paged(case, BAL), ref, "balanced B=300")
    assert binding.get_device_errors() == 0


def test_balanced_schedule_fewer_tiles_than_ctas():
    # 4 tiles in all, but a loose max_kv_len bound sizes the grid for 64: most persistent
    # CTAs get an empty range, and the combine must skip them
    case = inputs.make_paged_case(2, 16, 2, 128, 16, [40, 20], 85, max_pages=64).to("cuda")
    out = binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                    max_kv_len=1000, num_splits=BAL)
    assert_close(out, oracle_paged(case), "tiny balanced")
    assert binding.get_device_errors() == 0


@pytest.mark.parametrize("max_kv_len", [0, 64])
def test_every_sequence_empty_gives_zero_rows(max_kv_len):
    case = inputs.make_paged_case(4, 16, 4, 128, 16, [0, 0, 0, 0], 86, max_pages=4).to("cuda")
    for S in [BAL, 0, 1, 3]:
        out = torch.full_like(case.q, 5.0)
        binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                  max_kv_len=max_kv_len, num_splits=S, out=out)
        assert (out.float() == 0).all(), f"S={S}"
    assert binding.get_device_errors() == 0


def test_thousands_of_short_sequences_per_sequence_schedule():
    # 2048 sequences of 1..40 keys at S = 2: a grid of 8192 CTAs, most sequences in one chunk
    lens = inputs.uniform_lengths(2048, 1, 40, 87)
    case = inputs.make_paged_case(2048, 8, 2, 64, 16, lens, 87).to("cuda")
    ref = oracle_paged(case)
    assert_close(gpu_paged(case, 2), ref, "B=2048")
    assert binding.get_device_errors() == 0


def test_strided_q_and_out_and_garbage_workspace():
    case = inputs.make_paged_case(3, 16, 4, 128, 16, [90, 200, 7], 80).to("cuda")
    ref = oracle_paged(case)
    qbig = torch.zeros((3, 16, 3 * 128), dtype=torch.bfloat16, device="cuda")
    qbig[:, :, 128:256] = case.q
    q = qbig[:, :, 128:256]                      # stride_h = 384
    obig = torch.full((3, 16, 2 * 128), 7.0, dtype=torch.bfloat16, device="cuda")
    out = obig[:, :, :128]
    for S in [BAL, 4]:
        ws = torch.full((binding.workspace_bytes(3, 16, 4, 128, S),), 0xFF, dtype=torch.uint8, device="cuda")
        binding.decode_attn_paged(q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                  max_kv_len=case.max_kv_len, num_splits=S, workspace=ws, out=out)
        assert_close(out, ref, f"strided S={S}")
        assert torch.all(obig[:, :, 128:] == 7.0), "wrote outside the output rows"


def test_repeat_runs_are_identical():
    case = inputs.make_paged_case(4, 32, 8, 128, 16, [1000, 2000, 10, 555], 81).to("cuda")
    for S in [BAL, 0]:
        assert torch.equal(gpu_paged(case, S), gpu_paged(case, S))


def test_seq_len_above_bound_is_flagged_and_clamped():
    case = inputs.make_paged_case(2, 8, 2, 64, 16, [64, 40], 82).to("cuda")
    lens = torch.tensor([64, 40], dtype=torch.int32, device="cuda")
    bad = torch.tensor([64, 41], dtype=torch.int32, device="cuda")   # 41 > max_kv_len = 40 below
    out = binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, case.block_table, bad,
                                    max_kv_len=40, num_splits=1)
    assert binding.get_device_errors() & binding.DEVERR_SEQLEN
    ref = oracle.decode_paged(bits(case.q), bits(case.k_cache), bits(case.v_cache),
                              case.block_table.cpu().numpy(), np.array([40, 40], np.int32), case.scale)
    assert_close(out, ref, "clamped")
    del lens


def test_wait_that_runs_out_is_flagged_and_the_context_stays_usable():
    """The failure path of the pipeline waits, run on purpose: a bounded wait on a barrier
    nothing arrives on gives up after its limit (about a second), flags DEVERR_TIMEOUT and
    returns; a decode on the same context afterwards runs clean and matches the oracle."""
    binding.selftest_wait_timeout()
    torch.cuda.synchronize()
    assert binding.get_device_errors(clear=True) & binding.DEVERR_TIMEOUT
    case = inputs.make_paged_case(2, 8, 2, 64, 16, [40, 90], 88).to("cuda")
    assert_close(gpu_paged(case, 2), oracle_paged(case), "after the timeout")
    assert binding.get_device_errors() == 0


def test_page_index_outside_pool_is_flagged():
    case = inputs.make_paged_case(1, 8, 2, 64, 16, [40], 83).to("cuda")
    table = case.block_table.clone()
    table[0, 1] = case.num_pages + 5
    out = binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, table, case.seq_lens,
                                    max_kv_len=40, num_splits=1)
    torch.cuda.synchronize()
    assert binding.get_device_errors() & binding.DEVERR_PAGE
    del out


# ---- the named workloads at full size: every output element against the oracle -----------

def test_llama_workload_paged_and_contiguous():
    case = inputs.llama_paged(device="cuda")
    ref = oracle_paged(case)
    out = gpu_paged(case, 0)
    assert_close(out, ref, case.name)
    assert_close(gpu_paged(case, BAL), ref, case.name + ", balanced")
    k, v = inputs.logical_kv(case)
    c = binding.decode_attn_contig(case.q, k, v, case.seq_lens, max_kv_len=case.max_kv_len)
    assert torch.equal(c, out)
    assert binding.get_device_errors() == 0


def test_ragged_workload():
    """The benchmark's launch (the planner's S with the summed lengths known) and the
    planner's S without them, on all 128 x 32 x 128 outputs."""
    case = inputs.ragged_paged(device="cuda")
    ref = oracle_paged(case)
    assert_close(gpu_paged(case, 0, total_kv=case.total_kv), ref, case.name)
    assert_close(gpu_paged(case, 0), ref, case.name + ", S resolved by the library")
    assert_close(gpu_paged(case, BAL), ref, case.name + ", balanced")
    assert binding.get_device_errors() == 0


@pytest.mark.parametrize("B", [1, 4])
def test_long_context_workload_split_sweep(B):
    case = inputs.long_paged(B=B, device="cuda")
    ref = oracle_paged(case)
    for S in [BAL, 0, 1, 8, 32, 128]:
        assert_close(gpu_paged(case, S), ref, f"{case.name} S={S}")
    assert binding.get_device_errors() == 0


@pytest.mark.parametrize("shape", [(3, 8, 2, 64, 16, [100, 37, 300]), (130, 32, 8, 128, 16, None),
                                   (1, 64, 8, 128, 64, [20000])])
def test_zero_splits_is_the_resolved_planner_count(shape):
    """num_splits = 0 passed through the C ABI runs dap_resolve_splits(0, ...)'s S: the same
    bits as that explicit count, on the paged and the contiguous cache."""
    B, Hq, Hkv, D, ps, lens = shape
    lens = lens or inputs.uniform_lengths(B, 1, 3000, 90)
    case = inputs.make_paged_case(B, Hq, Hkv, D, ps, lens, 91 + B).to("cuda")
    S = binding.resolve_splits(0, binding.device_sm_count(), B, Hq, Hkv, D, ps, case.max_kv_len)
    a = gpu_paged(case, 0)
    assert torch.equal(a, gpu_paged(case, S)), f"planner S={S}"
    k, v = inputs.logical_kv(case)
    c0 = binding.decode_attn_contig(case.q, k, v, case.seq_lens, max_kv_len=case.max_kv_len, num_splits=0)
    cS = binding.decode_attn_contig(case.q, k, v, case.seq_lens, max_kv_len=case.max_kv_len, num_splits=S)
    assert torch.equal(c0, cS) and torch.equal(c0, a)
    assert_close(a, oracle_paged(case), f"planner S={S}")


@pytest.mark.parametrize("D", [32, 256])
def test_contiguous_head_dims_32_and_256(D):
    case = inputs.make_paged_case(3, 16, 4, D, 16, [150, 1, 64], 79 + D).to("cuda")
    k, v = inputs.logical_kv(case, max_len=160)
    ref = oracle.decode_contig(bits(case.q), bits(k), bits(v), case.seq_lens.cpu().numpy(), case.scale)
    for S in [BAL, 0, 1, 3]:
        c = binding.decode_attn_contig(case.q, k, v, case.seq_lens, max_kv_len=case.max_kv_len, num_splits=S)
        assert_close(c, ref, f"contig D={D} S={S}")
        assert torch.equal(c, gpu_paged(case, S))


# page sizes that are not multiples of 8: rows copied one by one into the swizzled tiles
ODD_PAGES = [
    # Hq, Hkv, D, ps
    (8, 2, 32, 12), (16, 16, 32, 3), (16, 2, 64, 1), (8, 8, 64, 7), (32, 8, 128, 12),
    (64, 8, 128, 100), (16, 8, 128, 5), (8, 2, 256, 12), (16, 2, 256, 5), (8, 8, 256, 1),
]


@pytest.mark.parametrize("Hq,Hkv,D,ps", ODD_PAGES, ids=[f"Hq{a}_Hkv{b}_D{c}_ps{d}" for a, b, c, d in ODD_PAGES])
def test_page_sizes_that_are_not_multiples_of_8(Hq, Hkv, D, ps):
    """Every head dim and schedule on page sizes off the TMA grid: the oracle within
    tolerance, and the contiguous cache (TMA tiles) bit for bit, since the tiles hold the
    same rows whichever way they were filled."""
    case = inputs.make_paged_case(4, Hq, Hkv, D, ps, [1, 150, 333, 64], 83 + D + ps).to("cuda")
    ref = oracle_paged(case)
    k, v = inputs.logical_kv(case)
    for S in [BAL, 0, 1, 3]:
        got = gpu_paged(case, S)
        assert_close(got, ref, f"D={D} ps={ps} S={S}")
        c = binding.decode_attn_contig(case.q, k, v, case.seq_lens, max_kv_len=case.max_kv_len, scale=case.scale,
                                       num_splits=S)
        assert torch.equal(got, c), f"D={D} ps={ps} S={S}: paged (row gather) != contiguous"
    assert binding.get_device_errors() == 0


def test_row_gather_page_permutation_and_bad_page_id():
    """Page size 12: a permutation of the physical pages gives the same bits; a page id
    outside the pool is read as page 0 and flagged, as on the TMA path."""
    case = inputs.make_paged_case(5, 32, 8, 128, 12, [700, 33, 1024, 5, 260], 84).to("cuda")
    perm = torch.randperm(case.num_pages, generator=torch.Generator().manual_seed(6)).cuda()
    inv = torch.argsort(perm)
    moved = inputs.PagedCase(case.q, case.k_cache[perm].contiguous(), case.v_cache[perm].contiguous(),
                             inv[case.block_table.long()].to(torch.int32).contiguous(), case.seq_lens,
                             case.page_size, case.scale)
    for S in [BAL, 0, 1, 4, 9]:
        assert torch.equal(gpu_paged(case, S), gpu_paged(moved, S)), f"S={S}"
    assert binding.get_device_errors() == 0
    bad = case.block_table.clone()
    bad[1, 0] = case.num_pages + 5
    out = binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, bad, case.seq_lens,
                                    max_kv_len=case.max_kv_len, scale=case.scale, num_splits=1)
    torch.cuda.synchronize()
    assert binding.get_device_errors(clear=True) & binding.DEVERR_PAGE
    fixed = bad.clone()
    fixed[1, 0] = 0
    want = binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, fixed, case.seq_lens,
                                     max_kv_len=case.max_kv_len, scale=case.scale, num_splits=1)
    # (page 0 may be an unused, NaN-filled page: compare bits)
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))
    assert binding.get_device_errors(clear=True) == 0
