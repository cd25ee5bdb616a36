"""The no-allocation paged decode entry point against the workspace one and the oracle.

decode_attn_paged_noalloc serves callers that cannot give the library scratch memory (a host
that reserves its whole device-memory budget at start-up, or a plugin interface that passes
only input and output buffers).  Its split partials live in a fixed device array inside the
library, so this file checks, through the C ABI, that two calls in a row (different
problems, the second reusing what the first left in the array) give what decode_attn_paged
gives with a caller workspace and what the fp64 oracle gives; that the planner's split count
is lowered until its partials fit the array; that a problem too big for the array is
refused; and that once a device has made its first call, later calls take no device memory.

Named to be collected last: it must pass alone in a fresh process and after the rest.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_298_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_close(got: torch.Tensor, want, what=""):
    g = got.float().cpu().double().numpy()
    w = want if isinstance(want, np.ndarray) else want.float().cpu().double().numpy()
    assert np.isfinite(g).all(), what
    excess = np.abs(g - w) - (ATOL + RTOL * np.abs(w))
    assert excess.max() <= 0, f"{what}: worst excess {excess.max():.3g}"


def oracle_paged(case):
    return oracle.decode_paged(bits(case.q), bits(case.k_cache), bits(case.v_cache),
                               case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(), case.scale)


def noalloc(case, S):
    return binding.decode_attn_paged_noalloc(case.q, case.k_cache, case.v_cache, case.block_table,
                                             case.seq_lens, max_kv_len=case.max_kv_len, num_splits=S)


def run_both(case, S):
    ref = binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                    max_kv_len=case.max_kv_len, num_splits=S)
    got = noalloc(case, S)
    torch.cuda.synchronize()
    return got, ref


def test_two_calls_in_a_row_match_the_workspace_entry_point_and_the_oracle():
    a = inputs.make_paged_case(6, 32, 8, 128, 16, [1000, 37, 2048, 500, 1, 3000], 9001).to("cuda")
    b = inputs.make_paged_case(3, 16, 2, 64, 16, [700, 0, 129], 9002).to("cuda")
    ra, rb = oracle_paged(a), oracle_paged(b)
    got, ref = run_both(a, 6)        # uses the scratch (6 splits)
    assert_close(got, ref, "S=6 vs workspace")
    assert_close(got, ra, "S=6 vs oracle")
    got, ref = run_both(b, 3)        # second call, the scratch holds the first call's partials
    assert_close(got, ref, "S=3 vs workspace")
    assert_close(got, rb, "S=3 vs oracle")
    got, ref = run_both(a, 0)        # the planner's split count, which fits here
    assert_close(got, ref, "planner vs workspace")
    assert_close(got, ra, "planner vs oracle")
    got, ref = run_both(b, binding.SPLITS_BALANCED)   # balanced partials fit at D = 64
    assert_close(got, ref, "balanced vs workspace")
    assert_close(got, rb, "balanced vs oracle")
    assert binding.get_device_errors() == 0


def test_page_size_that_is_not_a_multiple_of_8():
    """Page size 12 (rows copied one by one into the tiles): the same bits as the workspace
    entry point at the planner's split count, and the oracle."""
    case = inputs.make_paged_case(5, 32, 8, 128, 12, [700, 33, 1024, 5, 260], 9007, device="cuda")
    got, want = run_both(case, 0)
    assert torch.equal(got, want)
    assert_close(got, oracle_paged(case), "page 12 vs oracle")
    assert binding.get_device_errors() == 0


def test_head_dim_256_with_eight_heads_per_kv_head():
    """D = 256, G = 8: the planner's partials fit, the balanced schedule's (16 MiB of
    accumulators alone) do not and are refused."""
    case = inputs.make_paged_case(4, 64, 8, 256, 16, [5000, 77, 2600, 4096], 9004, device="cuda")
    ref = oracle_paged(case)
    got, want = run_both(case, 0)
    assert_close(got, want, "D=256 planner vs workspace")
    assert_close(got, ref, "D=256 planner vs oracle")
    assert binding.workspace_bytes(4, 64, 8, 256, binding.SPLITS_BALANCED) > binding.NOALLOC_SCRATCH_BYTES
    with pytest.raises(binding.DapError) as e:
        noalloc(case, binding.SPLITS_BALANCED)
    assert e.value.status == 7  # DAP_ERR_SCRATCH_LIMIT
    assert binding.get_device_errors() == 0


def test_planner_split_count_is_lowered_to_fit_the_scratch():
    """700 sequences of up to 600 keys, D = 256, 8 query heads on one kv head: on a GPU with
    141 to 210 SMs the planner picks 3 splits (17.5 MB of partials, more than the 16 MiB
    array), so the call runs 2; the result equals decode_attn_paged at 2 splits bit for bit
    and matches the oracle."""
    B, Hq, Hkv, D, ps = 700, 8, 1, 256, 16
    lens = inputs.uniform_lengths(B, 1, 600, 9005)
    lens[0] = 600
    case = inputs.make_paged_case(B, Hq, Hkv, D, ps, lens, 9005, device="cuda")
    sms = binding.device_sm_count()
    planned = binding.resolve_splits(0, sms, B, Hq, Hkv, D, ps, case.max_kv_len)
    cap = binding.NOALLOC_SCRATCH_BYTES
    fits = max(s for s in range(1, planned + 1) if binding.workspace_bytes(B, Hq, Hkv, D, s) <= cap)
    assert binding.workspace_bytes(B, Hq, Hkv, D, planned) > cap and 1 < fits < planned, (planned, fits)
    got = noalloc(case, 0)
    want = binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                     max_kv_len=case.max_kv_len, num_splits=fits)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    assert_close(got, oracle_paged(case), "lowered split count vs oracle")
    assert binding.get_device_errors() == 0


def test_partials_beyond_the_scratch_are_refused():
    case = inputs.make_paged_case(4, 64, 8, 128, 64, [8192] * 4, 9003).to("cuda")
    S = 128
    assert binding.workspace_bytes(4, 64, 8, 128, S) > binding.NOALLOC_SCRATCH_BYTES
    with pytest.raises(binding.DapError) as e:
        noalloc(case, S)
    assert e.value.status == 7  # DAP_ERR_SCRATCH_LIMIT


_FRESH = r"""
import json, sys, torch
sys.path.insert(0, sys.argv[1])
from paged_kv_cache_298_gb300 import binding, inputs
torch.cuda.set_device(0)
case = inputs.make_paged_case(5, 32, 8, 128, 16, [900, 3000, 17, 1, 2048], 9006, device="cuda")
outs = [torch.empty_like(case.q) for _ in range(3)]
torch.cuda.synchronize()
free = [torch.cuda.mem_get_info()[0]]
for o in outs:
    binding.decode_attn_paged_noalloc(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                      max_kv_len=case.max_kv_len, num_splits=4, out=o)
    torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info()[0])
same = bool(torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2]))
print(json.dumps({"free": free, "same": same, "errors": binding.get_device_errors()}))
"""


def test_calls_after_the_first_take_no_device_memory():
    """In a fresh process (so the first call is the device's first): the first call may
    reserve the array (lazy module loading); the calls after it change the device's free
    memory (cudaMemGetInfo) by 0 bytes and give the same bits."""
    r = subprocess.run([sys.executable, "-c", _FRESH, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    free = res["free"]
    assert free[0] >= free[1], free
    assert free[2] == free[1] and free[3] == free[1], free
    assert res["same"] and res["errors"] == 0
