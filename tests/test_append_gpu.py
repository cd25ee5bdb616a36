"""GPU parity of the cache-append kernels against the oracle: the paged bf16 append and the
fp8 quantised append are compared byte for byte (integer work: codes, scale bits, copied
rows); decoding right after an append is compared with the oracle within the decode
tolerance."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_298_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u16_to_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


@pytest.fixture(autouse=True)
def _clean():
    binding.get_device_errors(clear=True)
    yield


@pytest.mark.parametrize("B,Hkv,D,ps,lens", [(3, 8, 128, 16, [16, 5, 31]), (4, 2, 64, 1, [3, 0, 7, 9]),
                                              (2, 8, 128, 64, [64, 127])])
def test_paged_append_is_bit_exact(B, Hkv, D, ps, lens):
    case = inputs.make_paged_case(B, 4 * Hkv, Hkv, D, ps, [L + 1 for L in lens], 60 + D, poison=False)
    g = torch.Generator().manual_seed(61)
    k_new = inputs.randn_bf16((B, Hkv, D), g, "cpu")
    v_new = inputs.randn_bf16((B, Hkv, D), g, "cpu")
    pos = torch.tensor(lens, dtype=torch.int32)
    kc, vc, bad = oracle.kv_append_paged(bits(k_new), bits(v_new), bits(case.k_cache), bits(case.v_cache),
                                         case.block_table.numpy(), pos.numpy())
    assert bad == 0
    dk, dv = case.k_cache.cuda(), case.v_cache.cuda()
    binding.kv_append_paged(k_new.cuda(), v_new.cuda(), dk, dv, case.block_table.cuda(), pos.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bits(dk), kc) and np.array_equal(bits(dv), vc)
    assert binding.get_device_errors() == 0


def test_paged_append_then_decode_matches_oracle():
    lens = [100, 31, 2048, 0]
    case = inputs.make_paged_case(4, 32, 8, 128, 16, [L + 1 for L in lens], 62)
    g = torch.Generator().manual_seed(63)
    k_new = inputs.randn_bf16((4, 8, 128), g, "cpu")
    v_new = inputs.randn_bf16((4, 8, 128), g, "cpu")
    pos = torch.tensor(lens, dtype=torch.int32)
    kc, vc, _ = oracle.kv_append_paged(bits(k_new), bits(v_new), bits(case.k_cache), bits(case.v_cache),
                                       case.block_table.numpy(), pos.numpy())
    want = oracle.decode_paged(bits(case.q), kc, vc, case.block_table.numpy(), (pos + 1).numpy(), case.scale)
    dev = case.to("cuda")
    binding.kv_append_paged(k_new.cuda(), v_new.cuda(), dev.k_cache, dev.v_cache, dev.block_table, pos.cuda())
    for S in [0, 3]:
        out = binding.decode_attn_paged(dev.q, dev.k_cache, dev.v_cache, dev.block_table, (pos + 1).cuda(),
                                        max_kv_len=2049, num_splits=S)
        got = out.float().cpu().double().numpy()
        assert np.all(np.abs(got - want) <= 1e-2 + 1e-2 * np.abs(want)), f"S={S}"


def test_paged_append_out_of_range_position_is_skipped_and_flagged():
    case = inputs.make_paged_case(2, 4, 2, 64, 16, [20, 20], 64, poison=False)
    k_new = torch.ones((2, 2, 64), dtype=torch.bfloat16)
    dk, dv = case.k_cache.cuda(), case.v_cache.cuda()
    before = dk.clone()
    pos = torch.tensor([10 ** 6, -1], dtype=torch.int32).cuda()
    binding.kv_append_paged(k_new.cuda(), k_new.cuda(), dk, dv, case.block_table.cuda(), pos)
    torch.cuda.synchronize()
    assert binding.get_device_errors() & binding.DEVERR_SEQLEN
    assert torch.equal(dk, before)


@pytest.mark.parametrize("HD", [512, 256])
def test_fp8_append_is_bit_exact(HD):
    g = torch.Generator().manual_seed(65)
    T, NB, bs = 40, 4, 64
    mags = torch.tensor([1.0, 1e-3, 80.0, 0.0, 3.0] * 8)[:T, None]
    rows = (inputs.randn_bf16((T, HD), g, "cpu").float() * mags).to(torch.bfloat16)
    slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    cache = torch.randint(0, 255, (NB, bs, HD), generator=g, dtype=torch.uint8)
    inv = inputs.randn_bf16((NB * bs,), g, "cpu")
    c2, i2, bad = oracle.kv_append_fp8(bits(rows), cache.numpy(), bits(inv), slots.numpy())
    assert bad == 0
    dc, di = cache.cuda(), inv.cuda()
    binding.kv_append_fp8(rows.cuda(), dc, di, slots.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(dc.cpu().numpy(), c2)
    assert np.array_equal(bits(di), i2)
    assert binding.get_device_errors() == 0


def test_fp8_append_then_decode_matches_oracle():
    case = inputs.fp8_swa()
    g = torch.Generator().manual_seed(66)
    T = case.T
    rows = inputs.randn_bf16((T, case.HD), g, "cpu")
    # every token appends its own latent row to a fresh slot and puts it at the window's end
    slots = torch.randperm(case.num_blocks * case.block_size, generator=g)[:T].to(torch.int64)
    idx = case.indices.clone()
    lens = case.lens.clone()
    for t in range(T):
        n = int(min(lens[t], case.W - 1))
        idx[t, n] = slots[t]
        lens[t] = n + 1
    c2, i2, _ = oracle.kv_append_fp8(bits(rows), case.kv_cache.numpy(), bits(case.inv_scale), slots.numpy())
    want = oracle.fp8_swa(bits(case.q), c2, i2, idx.numpy(), lens.numpy(), case.block_size, case.scale)
    dev = case.to("cuda")
    binding.kv_append_fp8(rows.cuda(), dev.kv_cache, dev.inv_scale, slots.cuda())
    out = binding.decode_attn_paged_fp8(dev.q, dev.kv_cache, dev.inv_scale, idx.cuda(), lens.cuda())
    got = out.float().cpu().double().numpy()
    assert np.all(np.abs(got - want) <= 1e-2 + 1e-2 * np.abs(want))


def test_fp8_append_slot_outside_cache_is_skipped_and_flagged():
    rows = torch.ones((2, 512), dtype=torch.bfloat16).cuda()
    cache = torch.zeros((2, 16, 512), dtype=torch.uint8).cuda()
    inv = torch.zeros(32, dtype=torch.bfloat16).cuda()
    binding.kv_append_fp8(rows, cache, inv, torch.tensor([5, 32], dtype=torch.int64).cuda())
    torch.cuda.synchronize()
    assert binding.get_device_errors() & binding.DEVERR_SLOT
    assert cache.view(-1, 512)[5].ne(0).all() and float(inv[5]) > 0
