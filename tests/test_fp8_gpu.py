"""GPU parity of the fp8 sliding-window latent decode (K = V) against the fp64 oracle,
element by element: |gpu - oracle| <= 1e-2 + 1e-2 * |oracle|."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_298_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run(case):
    d = case.to("cuda")
    return binding.decode_attn_paged_fp8(d.q, d.kv_cache, d.inv_scale, d.indices, d.lens, scale=d.scale)


def ref(case):
    return oracle.fp8_swa(bits(case.q), case.kv_cache.numpy(), bits(case.inv_scale), case.indices.numpy(),
                          case.lens.numpy(), case.block_size, case.scale)


def assert_close(out, want, what=""):
    got = out.float().cpu().double().numpy()
    assert np.isfinite(got).all(), what
    excess = np.abs(got - want) - (1e-2 + 1e-2 * np.abs(want))
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, f"{what}: worst at {i}: gpu {got[i]} oracle {want[i]}"


@pytest.fixture(autouse=True)
def _clean():
    binding.get_device_errors(clear=True)
    yield


def test_fp8_workload_full_size():
    case = inputs.fp8_swa()
    assert_close(run(case), ref(case), case.name)
    assert binding.get_device_errors() == 0


@pytest.mark.parametrize("T,NH,NB,bs,W,lens", [
    (4, 128, 4, 64, 32, [32, 1, 17, 5]),        # ragged windows, one single row
    (3, 128, 2, 256, 128, [128, 0, 100]),       # full window, an empty token
    (2, 256, 4, 32, 64, [64, 33]),              # two head groups
    (5, 128, 1, 16, 16, [16, 16, 3, 9, 12]),    # tiny cache, rows shared between tokens
])
def test_fp8_parity(T, NH, NB, bs, W, lens):
    case = inputs.make_fp8_case(T, NH, 512, NB, bs, W, 7000 + T * W, lens=lens)
    if W > 8:
        case.indices[0, 3] = -1          # padding inside the window
    assert_close(run(case), ref(case), f"T={T} NH={NH} W={W}")
    assert binding.get_device_errors() == 0


def test_fp8_large_scales_and_window_past_len():
    case = inputs.make_fp8_case(4, 128, 512, 2, 64, 48, 7100, lens=[10, 48, 20, 1])
    case.inv_scale[:] = 2.0
    case.indices[0, 10:] = 3           # slots past len must be ignored
    assert_close(run(case), ref(case), "scales")


def test_fp8_slot_outside_cache_is_skipped_and_flagged():
    case = inputs.make_fp8_case(2, 128, 512, 2, 64, 16, 7200, lens=[16, 16])
    case.indices[1, 4] = 2 * 64 + 7    # past num_blocks * block_size
    out = run(case)
    torch.cuda.synchronize()
    assert binding.get_device_errors() & binding.DEVERR_SLOT
    assert_close(out, ref(case), "slot outside")   # the oracle skips it too


def test_fp8_repeat_is_deterministic():
    case = inputs.make_fp8_case(8, 128, 512, 4, 64, 64, 7300).to("cuda")
    a = binding.decode_attn_paged_fp8(case.q, case.kv_cache, case.inv_scale, case.indices, case.lens)
    b = binding.decode_attn_paged_fp8(case.q, case.kv_cache, case.inv_scale, case.indices, case.lens)
    assert torch.equal(a, b)


def test_single_row_windows_return_the_dequantised_row_exactly():
    """With one participating row the softmax weight is exactly 1, so every head's output is
    that row's dequantised value bf16(e4m3(code) * inv_scale) bit for bit.  The row holds
    every non-NaN code twice (subnormals, zeros, both signs, the largest magnitudes), and
    the tokens use inverse scales from 2^-100 to 3e30 (scores near 1e34: the kernel rounds
    each score once, so the largest one minus the maximum is exactly 0)."""
    inv_values = [1.0, 0.5, 2.0, 1.75, 0.5390625, 255.0, 256.0, 1000.0, 2.0 ** -20, 3e30, 2.0 ** -100, 1.0 / 3.0,
                  2.0 ** 60]
    T = len(inv_values)
    case = inputs.make_fp8_case(T, 128, 512, 1, 16, 4, 7400, lens=[1] * T)
    finite = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
    row = torch.cat([finite, finite, torch.zeros(512 - 2 * finite.numel(), dtype=torch.uint8)])
    case.kv_cache[0, :T] = row[None, :]
    case.inv_scale[:T, 0] = torch.tensor(inv_values, dtype=torch.float32).to(torch.bfloat16)
    case.indices[:] = -1
    case.indices[:, 0] = torch.arange(T)
    got = run(case).float().cpu().double().numpy()
    want = ref(case)
    assert np.isfinite(want).all()
    assert np.array_equal(got, want)
    # the output of every head is the same dequantised row
    assert np.array_equal(want[:, :1, :].repeat(128, axis=1), want)


def test_a_nan_code_in_a_row_makes_the_token_nan_like_the_fallback():
    """A NaN code (0x7F) in a participating row turns its scores into NaN; the fallback's
    softmax then gives NaN for every head of the token, and so does the kernel."""
    case = inputs.make_fp8_case(2, 128, 512, 1, 16, 4, 7401, lens=[2, 2])
    case.indices[:] = -1
    case.indices[0, :2] = torch.tensor([0, 1])
    case.indices[1, :2] = torch.tensor([2, 3])
    case.kv_cache[0, 1, 100] = 0x7F
    got = run(case).float().cpu().numpy()
    want = ref(case)
    assert np.isnan(want[0]).all() and np.isnan(got[0]).all()
    assert_close(torch.from_numpy(got[1:]), want[1:], "token without NaN codes")
