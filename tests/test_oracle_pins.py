"""Pins for the fp64 CPU oracle: each check ties it to something other than itself.

* scalar conversions against torch's own conversions (bf16 bits, e4m3 codes, fp32->bf16);
* closed forms of attention: constant V, a single key, a shift of every key, q = 0;
* brute force against torch's float64 scaled_dot_product_attention (with its own GQA
  head expansion) on logical K/V gathered here through the block table;
* page-permutation invariance and paged == contiguous;
* the fp8 sliding-window variant against the fallback's semantics written with torch ops
  (float8_e4m3fn view, bf16 multiply, boolean mask, float64 SDPA), plus its closed forms.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_298_gb300 import inputs


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


# ---- scalar conversions --------------------------------------------------------------

def test_bf16_value_all_codes():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    want = codes.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_value(c) for c in range(65536)])
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()


def test_e4m3_table_matches_torch_float8():
    want = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    want = want.to(torch.float64).numpy()
    got = oracle.e4m3_table()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(got[~np.isnan(got)], want[~np.isnan(want)])
    # two NaN codes (S.1111.111), largest finite 448, smallest subnormal 2^-9
    assert np.isnan(got).sum() == 2 and got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_round_to_bf16_matches_torch():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(4000, generator=g, dtype=torch.float32) * 3
    # exact ties: 9 significant bits with the last one set
    ties = torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(2.0 + 2 ** -7), 0.5 + 2 ** -9])
    x = torch.cat([x, ties])
    want = x.to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_to_bf16(float(v)) for v in x])
    assert np.array_equal(got, want)


# ---- paged decode: brute force against torch SDPA ------------------------------------

def gather_logical(case):
    """Logical [B][L_b, Hkv, D] float64 K and V, gathered here by a direct table walk."""
    k = as_f64(case.k_cache.float())
    v = as_f64(case.v_cache.float())
    table = case.block_table.numpy()
    ks, vs = [], []
    for b in range(case.B):
        L = int(case.seq_lens[b])
        t = np.arange(L)
        pages = table[b, t // case.page_size]
        slots = t % case.page_size
        ks.append(k[pages, slots])
        vs.append(v[pages, slots])
    return ks, vs


def sdpa_reference(case):
    q = as_f64(case.q.float())
    ks, vs = gather_logical(case)
    out = np.zeros((case.B, case.Hq, case.D))
    for b in range(case.B):
        if ks[b].shape[0] == 0:
            continue
        qb = torch.from_numpy(q[b])[:, None, :]                 # [Hq, 1, D]
        kb = torch.from_numpy(ks[b]).permute(1, 0, 2)           # [Hkv, L, D]
        vb = torch.from_numpy(vs[b]).permute(1, 0, 2)
        o = F.scaled_dot_product_attention(qb[None], kb[None], vb[None], scale=case.scale,
                                           enable_gqa=True)
        out[b] = o[0, :, 0, :].numpy()
    return out


def run_oracle(case):
    return oracle.decode_paged(bits(case.q), bits(case.k_cache), bits(case.v_cache),
                               case.block_table.numpy(), case.seq_lens.numpy(), case.scale)


SHAPES = [
    # B, Hq, Hkv, D, ps, lens
    (2, 4, 2, 64, 16, [37, 100]),
    (3, 8, 8, 64, 1, [5, 1, 9]),
    (2, 8, 2, 128, 3, [7, 20]),
    (4, 16, 2, 32, 8, [1, 8, 9, 33]),
    (1, 6, 3, 64, 64, [130]),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_paged_matches_torch_sdpa_float64(shape):
    B, Hq, Hkv, D, ps, lens = shape
    case = inputs.make_paged_case(B, Hq, Hkv, D, ps, lens, 11 + len(lens) + D)
    got = run_oracle(case)
    want = sdpa_reference(case)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_tiny_workload_matches_sdpa():
    case = inputs.tiny_paged()
    assert tuple(case.block_table.shape) == (2, 7) and case.num_pages == 16
    np.testing.assert_allclose(run_oracle(case), sdpa_reference(case), rtol=1e-11, atol=1e-12)


def test_head_mapping_is_consecutive_groups():
    # Hq=4, Hkv=2: heads 0,1 read kv head 0 and heads 2,3 read kv head 1.  Make the kv
    # heads' V constant and different; the outputs then name the kv head each q head used.
    case = inputs.make_paged_case(1, 4, 2, 64, 16, [20], 5)
    case.v_cache[:, :, 0, :] = 1.0
    case.v_cache[:, :, 1, :] = -2.0
    out = run_oracle(case)
    np.testing.assert_allclose(out[0, :2], 1.0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(out[0, 2:], -2.0, rtol=0, atol=1e-13)


# ---- paged decode: closed forms -------------------------------------------------------

def test_constant_v_gives_v():
    case = inputs.make_paged_case(2, 8, 2, 64, 16, [50, 3], 21, poison=False)
    row = inputs.randn_bf16((2, 64), torch.Generator().manual_seed(3), "cpu")
    case.v_cache[:] = row[None, None]
    out = run_oracle(case)
    for h in range(8):
        np.testing.assert_allclose(out[:, h], np.broadcast_to(as_f64(row.float())[h // 4], (2, 64)),
                                   rtol=0, atol=1e-13)


def test_single_key_returns_its_value_row():
    case = inputs.make_paged_case(3, 4, 1, 64, 16, [1, 1, 1], 22)
    out = run_oracle(case)
    ks, vs = gather_logical(case)
    for b in range(3):
        for h in range(4):
            assert np.array_equal(out[b, h], vs[b][0, 0])


def test_key_shift_leaves_output_unchanged():
    # Values on a quarter grid keep k + u exact in bf16, so the shift is exact.
    g = torch.Generator().manual_seed(23)
    case = inputs.make_paged_case(2, 4, 2, 64, 16, [40, 17], 23, poison=False)
    case.k_cache.copy_((torch.randint(-4, 5, case.k_cache.shape, generator=g) / 4).to(torch.bfloat16))
    base = run_oracle(case)
    u = (torch.randint(-2, 3, (2, 64), generator=g)).to(torch.bfloat16)
    shifted = case.k_cache + u[None, None]
    assert torch.equal(shifted.float(), case.k_cache.float() + u.float()[None, None])
    case.k_cache.copy_(shifted)
    np.testing.assert_allclose(run_oracle(case), base, rtol=1e-12, atol=1e-13)


def test_zero_query_gives_mean_of_values():
    case = inputs.make_paged_case(2, 4, 2, 64, 16, [37, 100], 24)
    case.q.zero_()
    out = run_oracle(case)
    _, vs = gather_logical(case)
    for b in range(2):
        for h in range(4):
            np.testing.assert_allclose(out[b, h], vs[b][:, h // 2].mean(axis=0), rtol=1e-12,
                                       atol=1e-13)


def test_empty_sequence_gives_zero_row():
    case = inputs.make_paged_case(2, 4, 2, 64, 16, [0, 19], 25)
    out = run_oracle(case)
    assert np.array_equal(out[0], np.zeros((4, 64)))
    np.testing.assert_allclose(out[1], sdpa_reference(case)[1], rtol=1e-11, atol=1e-12)


def test_scale_enters_once():
    # Doubling q with half the scale gives the same logits.
    case = inputs.make_paged_case(1, 4, 2, 64, 16, [30], 26)
    case.q.copy_((case.q.float() / 2).to(torch.bfloat16) * 2)   # keep q exactly halvable
    base = run_oracle(case)
    q2 = case.q.float() * 2
    out = oracle.decode_paged(bits(q2.to(torch.bfloat16)), bits(case.k_cache), bits(case.v_cache),
                              case.block_table.numpy(), case.seq_lens.numpy(), case.scale / 2)
    np.testing.assert_allclose(out, base, rtol=1e-12, atol=1e-13)


# ---- paged decode: invariants ---------------------------------------------------------

def test_physical_page_permutation_is_invisible():
    case = inputs.make_paged_case(3, 8, 2, 64, 16, [37, 100, 64], 27)
    base = run_oracle(case)
    perm = torch.randperm(case.num_pages, generator=torch.Generator().manual_seed(99))
    inv = torch.argsort(perm)
    k2 = case.k_cache[perm]
    v2 = case.v_cache[perm]
    t2 = inv[case.block_table.long()].to(torch.int32)
    out = oracle.decode_paged(bits(case.q), bits(k2), bits(v2), t2.numpy(), case.seq_lens.numpy(),
                              case.scale)
    assert np.array_equal(out, base)


def test_paged_equals_contiguous():
    case = inputs.make_paged_case(3, 8, 2, 64, 16, [37, 100, 1], 28)
    k, v = inputs.logical_kv(case)
    out = oracle.decode_contig(bits(case.q), bits(k), bits(v), case.seq_lens.numpy(), case.scale)
    assert np.array_equal(out, run_oracle(case))


def test_selected_rows_equal_full_rows():
    case = inputs.make_paged_case(3, 8, 2, 64, 16, [37, 100, 5], 29)
    full = run_oracle(case).reshape(-1, 64)
    rows = np.array([0, 5, 23, 9, 16])
    got = oracle.decode_paged_rows(bits(case.q), bits(case.k_cache), bits(case.v_cache),
                                   case.block_table.numpy(), case.seq_lens.numpy(), case.scale, rows)
    assert np.array_equal(got, full[rows])


def test_out_of_range_page_is_reported():
    case = inputs.make_paged_case(1, 4, 2, 64, 16, [20], 30)
    case.block_table[0, 1] = case.num_pages
    with pytest.raises(ValueError):
        run_oracle(case)


# ---- fp8 sliding-window latent decode ---------------------------------------------------

def fp8_torch_semantics(case):
    """The fallback's semantics written with torch ops: clamp the slot, split it into
    block and offset, view the bytes as float8_e4m3fn, multiply in bf16 by the inverse
    scale, mask j >= len and slot < 0, then float64 SDPA with K = V."""
    T, NH, HD, W, bs = case.T, case.NH, case.HD, case.W, case.block_size
    idx = case.indices
    safe = idx.clamp(min=0)
    rows = case.kv_cache[safe // bs, safe % bs]                       # [T, W, HD] u8
    deq = rows.view(torch.float8_e4m3fn).to(torch.bfloat16) * case.inv_scale[safe]
    deq = deq.to(torch.bfloat16)
    masked = (torch.arange(W)[None, :] >= case.lens[:, None]) | (idx < 0)
    kv = deq.to(torch.float64)
    q = case.q.to(torch.float64)
    out = torch.zeros(T, NH, HD, dtype=torch.float64)
    for t in range(T):
        keep = ~masked[t]
        if keep.sum() == 0:
            continue
        o = F.scaled_dot_product_attention(q[t][:, None, :], kv[t][keep][None],
                                           kv[t][keep][None], scale=case.scale)
        out[t] = o[:, 0, :]
    return out.numpy()


def run_fp8(case):
    return oracle.fp8_swa(bits(case.q), case.kv_cache.numpy(), bits(case.inv_scale),
                          case.indices.numpy(), case.lens.numpy(), case.block_size, case.scale)


@pytest.mark.parametrize("shape", [(6, 16, 64, 4, 32, 16), (3, 8, 128, 2, 64, 40),
                                   (4, 128, 512, 2, 256, 128)])
def test_fp8_matches_torch_semantics(shape):
    T, NH, HD, NB, bs, W = shape
    case = inputs.make_fp8_case(T, NH, HD, NB, bs, W, 31 + HD)
    # exercise the -1 padding inside the window too, not only after len
    case.indices[0, 0] = -1
    got = run_fp8(case)
    np.testing.assert_allclose(got, fp8_torch_semantics(case), rtol=1e-11, atol=1e-12)


def test_fp8_masked_rows_do_not_matter():
    case = inputs.make_fp8_case(4, 16, 64, 4, 32, 16, 41, lens=[3, 16, 1, 8])
    base = run_fp8(case)
    # rewrite every cache row that no token attends to
    used = set()
    for t in range(4):
        for j in range(int(case.lens[t])):
            if case.indices[t, j] >= 0:
                used.add(int(case.indices[t, j]))
    flat = case.kv_cache.view(-1, 64)
    for s in range(flat.shape[0]):
        if s not in used:
            flat[s] = 0x7E
    # and what sits in the window past len
    case.indices[0, 3:] = 5
    assert np.array_equal(run_fp8(case), base)


def test_fp8_single_row_and_constant_rows():
    case = inputs.make_fp8_case(2, 8, 64, 2, 16, 8, 42, lens=[1, 8])
    out = run_fp8(case)
    s0 = int(case.indices[0, 0])
    row = case.kv_cache.view(-1, 64)[s0].view(torch.float8_e4m3fn).to(torch.float64)
    inv = float(case.inv_scale[s0, 0].float())
    want = np.array([oracle.round_to_bf16(float(x) * inv) for x in row])
    for h in range(8):
        assert np.array_equal(out[0, h], want)
    # token 1: every slot holds the same bytes and scale -> output is that row
    flat = case.kv_cache.view(-1, 64)
    for j in range(8):
        s = int(case.indices[1, j])
        flat[s] = flat[s0]
        case.inv_scale[s] = case.inv_scale[s0]
    out = run_fp8(case)
    for h in range(8):
        np.testing.assert_allclose(out[1, h], want, rtol=0, atol=1e-13)


def test_fp8_empty_window_gives_zero():
    case = inputs.make_fp8_case(3, 8, 64, 2, 16, 8, 43, lens=[0, 4, 2])
    case.indices[1, :] = -1
    out = run_fp8(case)
    assert np.array_equal(out[0], np.zeros((8, 64))) and np.array_equal(out[1], np.zeros((8, 64)))
    assert np.abs(out[2]).sum() > 0


def test_fp8_with_unit_scales_is_mqa_decode():
    # inv_scale = 1 and full windows: the variant is single-kv-head decode with K = V over
    # the dequantised rows, which the (separately pinned) bf16 path also computes.
    case = inputs.make_fp8_case(2, 8, 64, 2, 16, 8, 44, lens=[8, 8])
    case.inv_scale[:] = 1.0
    out = run_fp8(case)
    flat = case.kv_cache.view(-1, 64)
    rows = flat[case.indices.clamp(min=0)].view(torch.float8_e4m3fn).to(torch.bfloat16)  # [T,W,HD]
    k = rows[:, :, None, :].contiguous()                                  # [T, W, 1, HD]
    got = oracle.decode_contig(bits(case.q), bits(k), bits(k),
                               np.full(2, 8, dtype=np.int32), case.scale)
    np.testing.assert_allclose(out, got, rtol=1e-12, atol=1e-13)


# ---- KV append (the step before decode) -----------------------------------------------

def test_e4m3_from_float_matches_torch_in_range():
    g = torch.Generator().manual_seed(51)
    x = torch.cat([torch.randn(3000, generator=g) * s for s in (0.01, 1.0, 30.0, 200.0)])
    x = x.clamp(-447.9, 447.9)
    # exact ties between neighbouring codes: 1 + 1/16 (between 1 and 1.125), 3 * 2^-10
    # (between the subnormals 2^-9 and 2 * 2^-9), 0.5 * (256 + 288)
    ties = torch.tensor([1.0625, -1.0625, 3 * 2.0 ** -10, 272.0, 0.0, -0.0, 2.0 ** -12])
    x = torch.cat([x, ties])
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_float(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_e4m3_from_float_roundtrips_every_code_and_saturates():
    table = oracle.e4m3_table()
    for code in range(256):
        if np.isnan(table[code]):
            continue
        assert oracle.e4m3_from_float(float(table[code])) == code or table[code] == 0.0
    assert oracle.e4m3_from_float(1e6) == 0x7E and oracle.e4m3_from_float(-1e6) == 0xFE
    assert oracle.e4m3_from_float(449.0) == 0x7E


def test_kv_append_paged_places_rows_where_decode_reads_them():
    case = inputs.make_paged_case(3, 8, 2, 64, 16, [16, 5, 31], 52, poison=False)
    g = torch.Generator().manual_seed(53)
    k_new = inputs.randn_bf16((3, 2, 64), g, "cpu")
    v_new = inputs.randn_bf16((3, 2, 64), g, "cpu")
    pos = case.seq_lens.numpy().copy()            # append at the current end
    kc, vc, bad = oracle.kv_append_paged(bits(k_new), bits(v_new), bits(case.k_cache), bits(case.v_cache),
                                         case.block_table.numpy(), pos)
    assert bad == 0
    grown = inputs.PagedCase(case.q, torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16),
                             torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16), case.block_table,
                             case.seq_lens + 1, case.page_size, case.scale)
    ks, vs = gather_logical(grown)
    for b in range(3):
        assert np.array_equal(ks[b][-1], as_f64(k_new[b].float()))
        assert np.array_equal(vs[b][-1], as_f64(v_new[b].float()))
        assert np.array_equal(ks[b][:-1], gather_logical(case)[0][b])   # nothing else moved
    # a position beyond the table is refused, not written
    _, _, bad = oracle.kv_append_paged(bits(k_new), bits(v_new), bits(case.k_cache), bits(case.v_cache),
                                       case.block_table.numpy(), np.array([0, 10 ** 6, 1], np.int32))
    assert bad == 2


def test_kv_append_fp8_matches_torch_quantisation_and_error_bound():
    g = torch.Generator().manual_seed(54)
    T, HD, NB, bs = 6, 512, 2, 16
    rows = inputs.randn_bf16((T, HD), g, "cpu") * torch.tensor([1.0, 0.001, 50.0, 1.0, 3.0, 0.0])[:, None]
    rows = rows.to(torch.bfloat16)
    cache = torch.zeros((NB, bs, HD), dtype=torch.uint8)
    inv = torch.zeros(NB * bs, dtype=torch.bfloat16)
    slots = np.array([3, 17, 0, 31, 8, 9], dtype=np.int64)
    c2, i2, bad = oracle.kv_append_fp8(bits(rows), cache.numpy(), bits(inv), slots)
    assert bad == 0
    flat = c2.reshape(-1, HD)
    for t in range(T):
        x = rows[t].float()
        amax = float(x.abs().max())
        s_bits = i2[slots[t]]
        s = float(torch.tensor(int(s_bits), dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float())
        want_s = torch.tensor([amax / 448.0 if amax > 0 else 1.0], dtype=torch.float32).to(torch.bfloat16)
        assert s == float(want_s.float())
        y = x / torch.tensor(s, dtype=torch.float32)
        codes = torch.from_numpy(flat[slots[t]].copy())
        inrange = y.abs() <= 448.0
        want = y[inrange].to(torch.float8_e4m3fn).view(torch.uint8)
        assert torch.equal(codes[inrange], want)
        assert torch.all(codes[~inrange] & 0x7F == 0x7E)           # saturated to +-448
        deq = codes.view(torch.float8_e4m3fn).float() * s
        err = (deq - x).abs()
        assert torch.all(err <= x.abs() * 2.0 ** -4 + s * 2.0 ** -10 + 1e-30)
    # untouched slots stay zero
    used = set(slots.tolist())
    for sl in range(NB * bs):
        if sl not in used:
            assert not flat[sl].any() and i2[sl] == 0


# ---- multi-token decode ----------------------------------------------------------------

def test_q_tile_map_matches_the_pages_worked_example():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "q_tile_map_astrai.json")))
    qi, tb, ti = oracle.q_tile_map(g["q_lens"], g["tokens_per_tile"])
    assert qi.tolist() == g["qo_indptr"]
    assert tb.tolist() == g["q_tile_to_batch"]
    assert ti.tolist() == g["q_tile_to_index"]


def multi_case(lens, qlens, seed, Hq=8, Hkv=2, D=64, ps=16):
    case = inputs.make_paged_case(len(lens), Hq, Hkv, D, ps, lens, seed)
    g = torch.Generator().manual_seed(seed + 1)
    q = inputs.randn_bf16((sum(qlens), Hq, D), g, "cpu")
    qi = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    return case, q, qi


def test_multi_token_with_one_token_each_is_single_token_decode():
    case, _, qi = multi_case([37, 100, 5], [1, 1, 1], 70)
    got = oracle.decode_paged_multi(bits(case.q), bits(case.k_cache), bits(case.v_cache), case.block_table.numpy(),
                                    case.seq_lens.numpy(), qi, case.scale)
    assert np.array_equal(got, run_oracle(case))


def test_multi_token_matches_causal_sdpa_float64():
    lens, qlens = [37, 100, 5, 64], [3, 4, 5, 1]
    case, q, qi = multi_case(lens, qlens, 71)
    got = oracle.decode_paged_multi(bits(q), bits(case.k_cache), bits(case.v_cache), case.block_table.numpy(),
                                    case.seq_lens.numpy(), qi, case.scale)
    ks, vs = gather_logical(case)
    qd = as_f64(q.float())
    for b, (L, n) in enumerate(zip(lens, qlens)):
        kb = torch.from_numpy(ks[b]).permute(1, 0, 2)[None]     # [1, Hkv, L, D]
        vb = torch.from_numpy(vs[b]).permute(1, 0, 2)[None]
        qb = torch.from_numpy(qd[qi[b]:qi[b + 1]]).permute(1, 0, 2)[None]   # [1, Hq, n, D]
        pos = torch.arange(L - n, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos                   # [n, L]: token i sees keys <= its position
        o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=case.scale, enable_gqa=True)
        np.testing.assert_allclose(got[qi[b]:qi[b + 1]], o[0].permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)


# ---- paged GQA decode over an e4m3 cache -----------------------------------------------

def fp8kv_decoded(case):
    """Logical float64 K and V per sequence, decoded by torch: float8_e4m3fn view of the
    codes times the bf16 factor of (page, kv head, slot)."""
    kval = case.k_codes.view(torch.float8_e4m3fn).to(torch.float64)
    vval = case.v_codes.view(torch.float8_e4m3fn).to(torch.float64)
    ksc = case.k_scale.to(torch.float64).permute(0, 2, 1)[..., None]   # [P, ps, Hkv, 1]
    vsc = case.v_scale.to(torch.float64).permute(0, 2, 1)[..., None]
    k = (kval * ksc).numpy()
    v = (vval * vsc).numpy()
    table = case.block_table.numpy()
    ks, vs = [], []
    for b in range(case.B):
        t = np.arange(int(case.seq_lens[b]))
        ks.append(k[table[b, t // case.page_size], t % case.page_size])
        vs.append(v[table[b, t // case.page_size], t % case.page_size])
    return ks, vs


def run_fp8kv(case, scale=None):
    return oracle.decode_paged_fp8kv(bits(case.q), case.k_codes.numpy(), case.v_codes.numpy(), bits(case.k_scale),
                                     bits(case.v_scale), case.block_table.numpy(), case.seq_lens.numpy(),
                                     case.scale if scale is None else scale)


FP8KV_SHAPES = [
    (2, 4, 2, 64, 16, [37, 100]),
    (3, 8, 8, 128, 8, [5, 1, 9]),
    (2, 32, 8, 128, 16, [70, 20]),
    (1, 16, 2, 128, 64, [130]),
]


@pytest.mark.parametrize("shape", FP8KV_SHAPES)
def test_fp8kv_matches_torch_float8_and_sdpa_float64(shape):
    B, Hq, Hkv, D, ps, lens = shape
    case = inputs.make_fp8kv_case(B, Hq, Hkv, D, ps, lens, 61 + D + len(lens))
    got = run_fp8kv(case)
    ks, vs = fp8kv_decoded(case)
    q = as_f64(case.q.float())
    for b in range(B):
        kb = torch.from_numpy(ks[b]).permute(1, 0, 2)[None]
        vb = torch.from_numpy(vs[b]).permute(1, 0, 2)[None]
        o = F.scaled_dot_product_attention(torch.from_numpy(q[b])[None, :, None, :], kb, vb, scale=case.scale,
                                           enable_gqa=True)[0, :, 0, :].numpy()
        np.testing.assert_allclose(got[b], o, rtol=1e-11, atol=1e-12)


def test_fp8kv_with_power_of_two_factors_is_the_bf16_decode():
    # codes times a power of two are exact in bf16: the fp8 decode must then be the bf16
    # decode of a cache holding those values
    case = inputs.make_fp8kv_case(3, 8, 2, 64, 16, [40, 17, 64], 71, poison=False)
    g = torch.Generator().manual_seed(72)
    for f in (case.k_scale, case.v_scale):
        f.copy_(torch.pow(2.0, torch.randint(-3, 4, f.shape, generator=g).float()).to(torch.bfloat16))
    kval = (case.k_codes.view(torch.float8_e4m3fn).float() * case.k_scale.float().permute(0, 2, 1)[..., None])
    vval = (case.v_codes.view(torch.float8_e4m3fn).float() * case.v_scale.float().permute(0, 2, 1)[..., None])
    assert torch.equal(kval.to(torch.bfloat16).float(), kval)
    bf = inputs.PagedCase(case.q, kval.to(torch.bfloat16), vval.to(torch.bfloat16), case.block_table,
                          case.seq_lens, case.page_size, case.scale)
    np.testing.assert_allclose(run_fp8kv(case), run_oracle(bf), rtol=1e-13, atol=1e-14)


def test_fp8kv_factors_scale_the_output_and_the_logits():
    case = inputs.make_fp8kv_case(2, 8, 2, 64, 16, [33, 50], 73, poison=False)
    base = run_fp8kv(case)
    doubled = inputs.Fp8KvCase(case.q, case.k_codes, case.v_codes, case.k_scale,
                               (case.v_scale.float() * 2).to(torch.bfloat16), case.block_table, case.seq_lens,
                               case.page_size, case.scale)
    np.testing.assert_allclose(run_fp8kv(doubled), 2 * base, rtol=1e-13, atol=1e-14)
    # every key factor times 4 is the softmax scale times 4
    k4 = inputs.Fp8KvCase(case.q, case.k_codes, case.v_codes, (case.k_scale.float() * 4).to(torch.bfloat16),
                          case.v_scale, case.block_table, case.seq_lens, case.page_size, case.scale)
    np.testing.assert_allclose(run_fp8kv(k4), run_fp8kv(case, scale=4 * case.scale), rtol=1e-12, atol=1e-13)


def test_fp8kv_page_permutation_and_empty_sequence():
    case = inputs.make_fp8kv_case(3, 8, 4, 64, 8, [0, 23, 64], 74, poison=False)
    got = run_fp8kv(case)
    assert np.all(got[0] == 0)
    P = case.k_codes.shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(75))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    moved = inputs.Fp8KvCase(case.q, case.k_codes[perm], case.v_codes[perm], case.k_scale[perm], case.v_scale[perm],
                             inv[case.block_table.long()].to(torch.int32), case.seq_lens, case.page_size, case.scale)
    np.testing.assert_array_equal(run_fp8kv(moved), got)


def test_kv_append_paged_fp8_places_and_quantises_rows():
    case = inputs.make_fp8kv_case(3, 8, 2, 64, 16, [16, 5, 31], 76, poison=False)
    g = torch.Generator().manual_seed(77)
    k_new = (inputs.randn_bf16((3, 2, 64), g, "cpu").float() * torch.tensor([1.0, 30.0, 0.01])[:, None, None])
    k_new = k_new.to(torch.bfloat16)
    v_new = inputs.randn_bf16((3, 2, 64), g, "cpu")
    kc, vc = case.k_codes.numpy().copy(), case.v_codes.numpy().copy()
    ks, vs = bits(case.k_scale).copy(), bits(case.v_scale).copy()
    pos = case.seq_lens.numpy().copy()
    assert oracle.kv_append_paged_fp8(bits(k_new), bits(v_new), kc, vc, ks, vs, case.block_table.numpy(), pos) == 0
    table = case.block_table.numpy()
    for b in range(3):
        page, slot = table[b, pos[b] // 16], pos[b] % 16
        for h in range(2):
            for new, codes, fac in ((k_new, kc, ks), (v_new, vc, vs)):
                x = new[b, h].float()
                amax = float(x.abs().max())
                s = torch.tensor([amax / 448.0], dtype=torch.float32).to(torch.bfloat16)
                assert fac[page, h, slot] == int(s.view(torch.int16)) & 0xFFFF
                want = (x / s.float()).to(torch.float8_e4m3fn).view(torch.uint8)
                assert np.array_equal(codes[page, slot, h], want.numpy())
    # every other slot is untouched
    changed = (kc != case.k_codes.numpy()).any(axis=(2, 3))
    assert changed.sum() <= 3
    # a position beyond the table is refused
    assert oracle.kv_append_paged_fp8(bits(k_new), bits(v_new), kc, vc, ks, vs, table,
                                      np.array([0, 10 ** 6, 1], np.int32)) == 2


# ---- masked decode ----------------------------------------------------------------------

def random_mask(B, width, seed, p_keep=0.6):
    g = torch.Generator().manual_seed(seed)
    return (torch.rand((B, width), generator=g) < p_keep).to(torch.uint8)


def run_masked(case, mask):
    return oracle.decode_paged_masked(bits(case.q), bits(case.k_cache), bits(case.v_cache), case.block_table.numpy(),
                                      case.seq_lens.numpy(), mask.numpy(), case.scale)


@pytest.mark.parametrize("shape", SHAPES[:4])
def test_masked_matches_torch_sdpa_with_bool_mask(shape):
    B, Hq, Hkv, D, ps, lens = shape
    case = inputs.make_paged_case(B, Hq, Hkv, D, ps, lens, 81 + D)
    mask = random_mask(B, max(lens) + 3, 82)
    mask[:, 0] = 1                       # keep one key per sequence so SDPA stays defined
    got = run_masked(case, mask)
    q = as_f64(case.q.float())
    ks, vs = gather_logical(case)
    for b in range(B):
        L = lens[b]
        kb = torch.from_numpy(ks[b]).permute(1, 0, 2)[None]
        vb = torch.from_numpy(vs[b]).permute(1, 0, 2)[None]
        am = mask[b, :L].bool()[None, None, None, :]
        o = F.scaled_dot_product_attention(torch.from_numpy(q[b])[None, :, None, :], kb, vb, attn_mask=am,
                                           scale=case.scale, enable_gqa=True)[0, :, 0, :].numpy()
        np.testing.assert_allclose(got[b], o, rtol=1e-11, atol=1e-12)


def test_masked_equals_decode_over_the_kept_keys_only():
    case = inputs.make_paged_case(3, 8, 2, 64, 16, [50, 9, 130], 83, poison=False)
    mask = random_mask(3, 130, 84, p_keep=0.3)
    got = run_masked(case, mask)
    ks, vs = gather_logical(case)
    for b in range(3):
        L = int(case.seq_lens[b])
        keep = mask[b, :L].numpy().astype(bool)
        n = int(keep.sum())
        # a contiguous cache holding only the kept keys, in order
        k = torch.from_numpy(ks[b][keep]).to(torch.bfloat16)[None]
        v = torch.from_numpy(vs[b][keep]).to(torch.bfloat16)[None]
        want = oracle.decode_contig(bits(case.q[b:b + 1]), bits(k), bits(v), np.array([n], np.int32), case.scale)
        np.testing.assert_allclose(got[b], want[0], rtol=1e-13, atol=1e-14)


def test_all_ones_and_all_zero_masks():
    case = inputs.make_paged_case(2, 8, 2, 64, 16, [40, 77], 85)
    ones = torch.ones((2, 80), dtype=torch.uint8)
    np.testing.assert_array_equal(run_masked(case, ones), run_oracle(case))
    zeros = torch.zeros((2, 80), dtype=torch.uint8)
    assert np.all(run_masked(case, zeros) == 0)


def test_multi_token_mask_joins_the_causal_rule():
    kv, qt, qi = multi_case([40, 90], [3, 5], 86)
    mask = random_mask(8, 96, 87)
    mask[:, 0] = 1
    got = oracle.decode_paged_multi(bits(qt), bits(kv.k_cache), bits(kv.v_cache), kv.block_table.numpy(),
                                    kv.seq_lens.numpy(), qi, kv.scale, mask=mask.numpy())
    ks, vs = gather_logical(kv)
    q = as_f64(qt.float())
    for b, (L, ql) in enumerate(zip([40, 90], [3, 5])):
        kb = torch.from_numpy(ks[b]).permute(1, 0, 2)[None]
        vb = torch.from_numpy(vs[b]).permute(1, 0, 2)[None]
        for i in range(ql):
            r = qi[b] + i
            pos = L - ql + i
            am = (torch.arange(L) <= pos) & mask[r, :L].bool()
            o = F.scaled_dot_product_attention(torch.from_numpy(q[r])[None, :, None, :], kb, vb,
                                               attn_mask=am[None, None, None, :], scale=kv.scale,
                                               enable_gqa=True)[0, :, 0, :].numpy()
            np.testing.assert_allclose(got[r], o, rtol=1e-11, atol=1e-12)
    ones = np.ones((8, 96), np.uint8)
    plain = oracle.decode_paged_multi(bits(qt), bits(kv.k_cache), bits(kv.v_cache), kv.block_table.numpy(),
                                      kv.seq_lens.numpy(), qi, kv.scale)
    np.testing.assert_array_equal(oracle.decode_paged_multi(bits(qt), bits(kv.k_cache), bits(kv.v_cache),
                                                            kv.block_table.numpy(), kv.seq_lens.numpy(), qi,
                                                            kv.scale, mask=ones), plain)
