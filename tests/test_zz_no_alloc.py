"""The no-allocation paged decode entry point against the workspace one.

decode_attn_paged_noalloc serves callers that cannot give the library scratch memory (a host
that reserves its whole device-memory budget at start-up, or a plugin interface that passes
only input and output buffers).  Its split partials live in a fixed device array inside the
library, so this file checks, through the C ABI, that two calls in a row (different
problems, the second reusing what the first left in the array) give what decode_attn_paged
gives with a caller workspace, and that a problem too big for the array is refused.

Named to be collected last: it must pass alone in a fresh process and after the rest.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_298_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2


def assert_close(got: torch.Tensor, want: torch.Tensor):
    g = got.float().cpu().double().numpy()
    w = want.float().cpu().double().numpy()
    assert np.isfinite(g).all()
    assert (np.abs(g - w) <= ATOL + RTOL * np.abs(w)).all()


def run_both(case, S):
    ref = binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                    max_kv_len=case.max_kv_len, num_splits=S)
    got = binding.decode_attn_paged_noalloc(case.q, case.k_cache, case.v_cache, case.block_table,
                                            case.seq_lens, max_kv_len=case.max_kv_len, num_splits=S)
    torch.cuda.synchronize()
    return got, ref


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    a = inputs.make_paged_case(6, 32, 8, 128, 16, [1000, 37, 2048, 500, 1, 3000], 9001).to("cuda")
    b = inputs.make_paged_case(3, 16, 2, 64, 16, [700, 0, 129], 9002).to("cuda")
    got, ref = run_both(a, 6)        # uses the scratch (6 splits)
    assert_close(got, ref)
    got, ref = run_both(b, 3)        # second call, scratch holds the first call's partials
    assert_close(got, ref)
    got, ref = run_both(a, 0)        # planner choice, fitted to the scratch
    assert_close(got, ref)
    assert binding.get_device_errors() == 0


def test_partials_beyond_the_scratch_are_refused():
    case = inputs.make_paged_case(4, 64, 8, 128, 64, [8192] * 4, 9003).to("cuda")
    S = 128
    assert binding.workspace_bytes(4, 64, 8, 128, S) > binding.NOALLOC_SCRATCH_BYTES
    with pytest.raises(binding.DapError) as e:
        binding.decode_attn_paged_noalloc(case.q, case.k_cache, case.v_cache, case.block_table,
                                          case.seq_lens, max_kv_len=case.max_kv_len, num_splits=S)
    assert e.value.status == 7  # DAP_ERR_SCRATCH_LIMIT
