"""Host-side checks of the C ABI that need no GPU: the library loads, exports every symbol
include/dap.h declares, plans splits sensibly, sizes workspaces, and rejects bad arguments
with the documented status before touching CUDA."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_298_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return binding.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dap.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"defined", "sizeof"})


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(binding.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(8):
        assert binding.status_string(s)
    assert binding.status_string(99) == "unknown status"
    assert lib.dap_version() >= 100


def test_chunk_tokens_cover_and_round_to_tiles():
    for L in [0, 1, 31, 32, 33, 100, 2048, 32768]:
        for S in [1, 2, 3, 8, 32, 128]:
            c = binding.chunk_tokens(L, S)
            assert c % 64 == 0 and c >= 64
            assert c * S >= L                       # S chunks cover the longest sequence
            assert c - 64 < max(1, -(-L // S))      # and no chunk is a whole tile too long


def test_plan_splits_properties():
    # one SM-wave worth of long sequences is still split; huge batches are not
    assert binding.plan_splits(152, 1, 64, 8, 128, 64, 32768, 32768) > 8
    assert binding.plan_splits(152, 4096, 32, 8, 128, 16, 512, 4096 * 512) == 1
    # never more splits than 64-token chunks of the longest sequence
    for L in [1, 31, 100, 1000]:
        assert binding.plan_splits(152, 1, 32, 1, 128, 16, L, L) <= -(-L // 64)
    # degenerate inputs give one split
    assert binding.plan_splits(0, 1, 32, 8, 128, 16, 100, 100) == 1
    assert binding.plan_splits(152, 0, 32, 8, 128, 16, 100, 100) == 1
    assert binding.plan_splits(152, 4, 32, 8, 128, 16, 0, 0) == 1
    # more total work -> chunks no smaller
    a = binding.chunk_tokens(4096, binding.plan_splits(152, 16, 32, 8, 128, 16, 4096, 16 * 4096))
    b = binding.chunk_tokens(4096, binding.plan_splits(152, 128, 32, 8, 128, 16, 4096, 128 * 4096))
    assert b >= a


def test_workspace_bytes():
    assert binding.workspace_bytes(16, 32, 8, 128, 1) == 0
    n = binding.workspace_bytes(16, 32, 8, 128, 8)
    assert n >= 16 * 8 * 32 * (128 + 2) * 4 and n % 256 == 0
    # balanced schedule: two partial slots per persistent CTA (up to 1024) + unit records
    bal = binding.workspace_bytes(128, 32, 8, 128, binding.SPLITS_BALANCED)
    assert bal >= 2 * 1024 * 4 * (128 + 2) * 4 + 128 * 8 * 8
    assert bal < 8 << 20
    assert binding.workspace_bytes(5000, 32, 8, 128, binding.SPLITS_BALANCED) == 0  # one CTA per unit
    assert binding.workspace_bytes(16, 32, 8, 128, 0) == 0       # 0 is not a split count
    assert binding.workspace_bytes(16, 32, 8, 128, -2) == 0


def test_resolve_splits_is_the_planner_for_zero_and_clamps_explicit_counts():
    """num_splits = 0 means the planner's S on every decode entry point; explicit counts are
    kept unless more chunks than the longest sequence can fill; -1 selects the balanced
    schedule (one CTA per unit past 4096 sequences); anything below is invalid."""
    cases = [(152, 1, 64, 8, 128, 64, 32768, 32768), (152, 4, 64, 8, 128, 64, 32768, 4 * 32768),
             (152, 16, 32, 8, 128, 16, 2048, 16 * 2048), (152, 128, 32, 8, 128, 16, 4096, 278000),
             (152, 3, 8, 2, 64, 16, 100, 0), (152, 2048, 8, 2, 64, 16, 40, 0), (132, 7, 16, 4, 256, 8, 999, 0)]
    def clamp(S, L):   # splits beyond the chunks the longest sequence fills are dropped
        chunk = binding.chunk_tokens(L, S)
        return max(1, min(S, -(-L // chunk) if L > 0 else 1))

    for sms, B, Hq, Hkv, D, ps, L, tot in cases:
        plan = binding.plan_splits(sms, B, Hq, Hkv, D, ps, L, tot)
        assert binding.resolve_splits(0, sms, B, Hq, Hkv, D, ps, L, tot) == clamp(plan, L)
        for S in (1, 2, 7, 64, 1000):
            r = binding.resolve_splits(S, sms, B, Hq, Hkv, D, ps, L, tot)
            assert r == clamp(S, L)
            assert 1 <= r <= S and (r == S or r * binding.chunk_tokens(L, S) >= L)
    # long context B=1: the planner's 38 splits of 896-token chunks leave the 38th empty
    assert binding.plan_splits(152, 1, 64, 8, 128, 64, 32768, 32768) == 38
    assert binding.resolve_splits(0, 152, 1, 64, 8, 128, 64, 32768, 32768) == 37
    for sms, B, Hq, Hkv, D, ps, L, tot in cases:
        assert binding.resolve_splits(-1, sms, B, Hq, Hkv, D, ps, L, tot) == binding.SPLITS_BALANCED
    assert binding.resolve_splits(-1, 152, 5000, 32, 8, 128, 16, 100, 0) == 1
    assert binding.resolve_splits(-2, 152, 4, 32, 8, 128, 16, 100, 0) == 0
    assert binding.resolve_splits(3, 152, 4, 32, 8, 128, 16, 0, 0) == 1     # nothing to split


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails validation first


def paged_call(lib, **kw):
    args = dict(q=FAKE, qsb=32 * 128, qsh=128, k=FAKE, v=FAKE, P=64, ps=16, table=FAKE, maxp=8,
                lens=FAKE, maxlen=100, B=2, Hq=32, Hkv=8, D=128, scale=0.088, S=1, ws=None, wsb=0,
                out=FAKE, osb=32 * 128, osh=128)
    args.update(kw)
    return lib.decode_attn_paged(args["q"], args["qsb"], args["qsh"], args["k"], args["v"], args["P"],
                                 args["ps"], args["table"], args["maxp"], args["lens"], args["maxlen"],
                                 args["B"], args["Hq"], args["Hkv"], args["D"], args["scale"], args["S"],
                                 args["ws"], args["wsb"], args["out"], args["osb"], args["osh"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=-1), 2), (dict(Hq=30), 2), (dict(Hkv=0), 2), (dict(maxlen=-1), 2),
    (dict(maxlen=8 * 16 + 1), 2), (dict(ps=0), 2), (dict(P=0), 2), (dict(S=-2), 2),
    (dict(scale=float("nan")), 2), (dict(qsh=-8), 2),
    (dict(q=None), 1), (dict(out=None), 1), (dict(k=None), 1), (dict(table=None), 1),
    (dict(lens=None), 1),
    (dict(D=96), 3), (dict(Hq=48, Hkv=3), 3), (dict(Hq=64, Hkv=4), 3),
    (dict(q=ctypes.c_void_p((1 << 20) + 8)), 5), (dict(qsh=130), 5), (dict(osb=4100), 5),
    (dict(k=ctypes.c_void_p((1 << 20) + 4)), 5),
    (dict(S=4), 4), (dict(S=4, ws=FAKE, wsb=16), 4), (dict(S=-1), 4), (dict(S=-1, ws=FAKE, wsb=4096), 4),
    (dict(qsh=0), 2), (dict(osb=0), 2),
])
def test_paged_validation(lib, kw, status):
    assert paged_call(lib, **kw) == status


def test_empty_batch_is_a_no_op(lib):
    assert paged_call(lib, B=0, q=None, out=None, lens=None, k=None, v=None, table=None) == 0


def test_contig_validation(lib):
    f = lib.decode_attn_contig
    assert f(FAKE, 4096, 128, FAKE, FAKE, 100, FAKE, 101, 2, 32, 8, 128, 0.1, 1, None, 0, FAKE, 4096, 128,
             None) == 2   # max_kv_len > max_len
    assert f(FAKE, 4096, 128, None, FAKE, 100, FAKE, 50, 2, 32, 8, 128, 0.1, 1, None, 0, FAKE, 4096, 128,
             None) == 1


def test_fp8_validation(lib):
    f = lib.decode_attn_paged_fp8
    ok = dict(T=4, NH=128, HD=512, W=128, NB=64, bs=256)

    def call(**kw):
        a = dict(ok, **kw)
        return f(FAKE, FAKE, FAKE, FAKE, FAKE, a["T"], a["NH"], a["HD"], a["W"], a["NB"], a["bs"], 0.04,
                 FAKE, None)
    assert call(T=-1) == 2 and call(W=0) == 2 and call(bs=0) == 2
    assert call(HD=256) == 3 and call(NH=64) == 3 and call(W=129) == 3
    assert call(T=0) == 0
    assert f(None, FAKE, FAKE, FAKE, FAKE, 4, 128, 512, 128, 64, 256, 0.04, FAKE, None) == 1


def test_append_validation(lib):
    f = lib.kv_append_paged
    assert f(FAKE, FAKE, FAKE, FAKE, 8, 16, FAKE, 4, FAKE, -1, 2, 64, None) == 2
    assert f(FAKE, FAKE, FAKE, FAKE, 8, 16, FAKE, 4, FAKE, 2, 2, 60, None) == 3
    assert f(None, FAKE, FAKE, FAKE, 8, 16, FAKE, 4, FAKE, 2, 2, 64, None) == 1
    assert f(None, None, None, None, 8, 16, None, 4, None, 0, 2, 64, None) == 0
    assert f(ctypes.c_void_p((1 << 20) + 2), FAKE, FAKE, FAKE, 8, 16, FAKE, 4, FAKE, 2, 2, 64, None) == 5
    g = lib.kv_append_fp8
    assert g(FAKE, FAKE, FAKE, FAKE, 4, 384, 2, 16, None) == 3
    assert g(FAKE, FAKE, FAKE, FAKE, -1, 512, 2, 16, None) == 2
    assert g(FAKE, None, FAKE, FAKE, 4, 512, 2, 16, None) == 1


# ---- multi-token decode: host work map and validation -------------------------------------

def test_multi_tokens_per_tile(lib):
    # 16 query columns while the longest new-token run fits them, else 32 (one K/V stream
    # for up to 32 / G tokens of a sequence)
    assert [binding.multi_tokens_per_tile(8 * g, 8) for g in (1, 2, 4, 8)] == [16, 8, 4, 2]
    assert [binding.multi_tokens_per_tile(8 * g, 8, 4) for g in (1, 2, 4, 8)] == [16, 8, 4, 4]
    assert [binding.multi_tokens_per_tile(8 * g, 8, 17) for g in (1, 2, 4, 8)] == [32, 16, 8, 4]
    assert binding.multi_tokens_per_tile(64, 8, 2) == 2 and binding.multi_tokens_per_tile(64, 8, 3) == 4
    assert binding.multi_tokens_per_tile(30, 8) == 0 and binding.multi_tokens_per_tile(8, 0) == 0
    # with the head dim: 128-row tiles (128 / G tokens) past 16 / G tokens at D 64, 128, 256
    assert [binding.multi_tokens_per_tile(8 * g, 8, 4, 128) for g in (1, 2, 4, 8)] == [16, 8, 4, 16]
    assert [binding.multi_tokens_per_tile(8 * g, 8, 17, 64) for g in (1, 2, 4, 8)] == [128, 64, 32, 16]
    assert [binding.multi_tokens_per_tile(64, 8, 3, d) for d in (32, 64, 128, 256)] == [4, 16, 16, 16]
    assert binding.multi_tokens_per_tile(64, 8, 2, 128) == 2 and binding.multi_tokens_per_tile(64, 8, 3, -1) == 0


def test_q_tile_map_matches_the_pages_worked_example():
    import json
    with open(os.path.join(ROOT, "tests", "golden", "q_tile_map_astrai.json")) as f:
        g = json.load(f)
    qi, tb, ti = binding.q_tile_map(g["q_lens"], g["tokens_per_tile"])
    assert qi.tolist() == g["qo_indptr"]
    assert tb.tolist() == g["q_tile_to_batch"] and ti.tolist() == g["q_tile_to_index"]


def test_q_tile_map_matches_the_oracle_on_random_counts():
    import numpy as np
    import oracle
    rng = np.random.default_rng(5)
    for tpt in (2, 4, 8, 16):
        lens = rng.integers(0, 40, size=23)
        lens[[0, 7]] = 0
        qi, tb, ti = binding.q_tile_map(lens, tpt)
        oqi, otb, oti = oracle.q_tile_map(lens, tpt)
        assert qi.tolist() == oqi.tolist() and tb.tolist() == otb.tolist() and ti.tolist() == oti.tolist()


def test_q_tile_map_rejects_bad_input(lib):
    lens = (ctypes.c_int32 * 3)(4, -1, 2)
    qi = (ctypes.c_int32 * 4)()
    tb = (ctypes.c_int32 * 8)()
    ti = (ctypes.c_int32 * 8)()
    assert lib.dap_q_tile_map(lens, 3, 4, qi, tb, ti, 8) == -1            # negative count
    lens = (ctypes.c_int32 * 3)(4, 9, 2)
    assert lib.dap_q_tile_map(lens, 3, 4, qi, tb, ti, 4) == -1            # needs 5 tiles
    assert lib.dap_q_tile_map(lens, 3, 0, qi, tb, ti, 8) == -1            # zero tile size
    assert lib.dap_q_tile_map(lens, 3, 4, qi, tb, ti, 5) == 5


def test_workspace_bytes_multi():
    assert binding.workspace_bytes_multi(64, 32, 128, 1) == 0
    n = binding.workspace_bytes_multi(64, 32, 128, 5)
    assert n >= 64 * 5 * 32 * (128 + 2) * 4 and n % 256 == 0


def multi_call(lib, **kw):
    a = dict(q=FAKE, qst=32 * 128, qsh=128, k=FAKE, v=FAKE, P=64, ps=16, table=FAKE, maxp=8, lens=FAKE,
             qi=FAKE, tb=FAKE, ti=FAKE, ntiles=2, tpt=4, totq=8, maxlen=100, B=2, Hq=32, Hkv=8, D=128, scale=0.088,
             S=1, ws=None, wsb=0, out=FAKE, ost=32 * 128, osh=128)
    a.update(kw)
    return lib.decode_attn_paged_multi(a["q"], a["qst"], a["qsh"], a["k"], a["v"], a["P"], a["ps"], a["table"],
                                       a["maxp"], a["lens"], a["qi"], a["tb"], a["ti"], a["ntiles"], a["tpt"], a["totq"],
                                       a.get("mask"), a.get("mst", 0), a["maxlen"], a["B"], a["Hq"], a["Hkv"],
                                       a["D"], a["scale"], a["S"], a["ws"], a["wsb"], a["out"], a["ost"], a["osh"],
                                       None)


@pytest.mark.parametrize("kw,status", [
    (dict(totq=-1), 2), (dict(ntiles=0), 2), (dict(totq=0), 2), (dict(ntiles=9), 2), (dict(B=0), 2),
    (dict(Hq=30), 2), (dict(maxlen=8 * 16 + 1), 2), (dict(S=-2), 2), (dict(S=-1), 3), (dict(qsh=0), 2),
    (dict(q=None), 1), (dict(qi=None), 1), (dict(tb=None), 1), (dict(ti=None), 1), (dict(table=None), 1),
    (dict(D=96), 3), (dict(Hq=64, Hkv=4), 3),
    (dict(qi=ctypes.c_void_p((1 << 20) + 2)), 5), (dict(qst=4100), 5),
    (dict(S=4), 4), (dict(S=4, ws=FAKE, wsb=16), 4),
    (dict(mask=FAKE, mst=96), 2), (dict(mask=FAKE, mst=120), 5), (dict(mask=ctypes.c_void_p((1 << 20) + 4), mst=128), 5),
    (dict(tpt=3), 2), (dict(tpt=16), 2), (dict(tpt=0), 2), (dict(tpt=8, mask=FAKE, mst=128), 3),
    # 128-row tiles (tokens_per_tile = 128 / G): D 64, 128 and 256 only
    (dict(tpt=32, D=32), 3), (dict(tpt=32, mask=FAKE, mst=128, D=32), 3), (dict(tpt=64), 2),
])
def test_multi_validation(lib, kw, status):
    assert multi_call(lib, **kw) == status


def test_multi_empty_is_a_no_op(lib):
    assert multi_call(lib, totq=0, ntiles=0, q=None, out=None, k=None, qi=None, tb=None, ti=None) == 0


# ---- fp8 (e4m3) GQA cache: validation --------------------------------------------------

def fp8kv_call(lib, **kw):
    a = dict(q=FAKE, qsb=32 * 128, qsh=128, kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE, P=64, ps=16, table=FAKE, maxp=8,
             lens=FAKE, maxlen=100, B=2, Hq=32, Hkv=8, D=128, scale=0.088, S=1, ws=None, wsb=0, out=FAKE,
             osb=32 * 128, osh=128)
    a.update(kw)
    return lib.decode_attn_paged_fp8kv(a["q"], a["qsb"], a["qsh"], a["kc"], a["vc"], a["ks"], a["vs"], a["P"],
                                       a["ps"], a["table"], a["maxp"], a["lens"], a["maxlen"], a["B"], a["Hq"],
                                       a["Hkv"], a["D"], a["scale"], a["S"], a["ws"], a["wsb"], a["out"], a["osb"],
                                       a["osh"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=-1), 2), (dict(Hq=30), 2), (dict(maxlen=8 * 16 + 1), 2), (dict(S=-2), 2), (dict(S=-1), 3),
    (dict(P=0), 2),
    (dict(kc=None), 1), (dict(ks=None), 1), (dict(vs=None), 1), (dict(table=None), 1), (dict(q=None), 1),
    (dict(D=32, qsb=32 * 32, qsh=32, osb=32 * 32, osh=32), 3), (dict(Hq=64, Hkv=4), 3),
    (dict(ks=ctypes.c_void_p((1 << 20) + 8)), 5), (dict(kc=ctypes.c_void_p((1 << 20) + 4)), 5),
    (dict(S=4), 4), (dict(S=4, ws=FAKE, wsb=64), 4),
])
def test_fp8kv_validation(lib, kw, status):
    assert fp8kv_call(lib, **kw) == status


def test_fp8kv_empty_batch_is_a_no_op(lib):
    assert fp8kv_call(lib, B=0, q=None, out=None, kc=None, vc=None, ks=None, vs=None, lens=None, table=None) == 0


def test_append_paged_fp8_validation(lib):
    f = lib.kv_append_paged_fp8
    ok = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, 16, FAKE, 4, FAKE, 2, 2, 128, None]
    def call(i=None, v=None):
        a = list(ok)
        if i is not None:
            a[i] = v
        return f(*a)
    assert call(11, -1) == 2 and call(6, 0) == 2
    assert call(13, 96) == 3
    assert call(0, None) == 1 and call(4, None) == 1
    assert call(11, 0) == 0
    assert call(2, ctypes.c_void_p((1 << 20) + 4)) == 5 and call(4, ctypes.c_void_p((1 << 20) + 1)) == 5


def masked_call(lib, **kw):
    a = dict(q=FAKE, qsb=32 * 128, qsh=128, k=FAKE, v=FAKE, P=64, ps=16, table=FAKE, maxp=8, lens=FAKE, mask=FAKE,
             mst=128, maxlen=100, B=2, Hq=32, Hkv=8, D=128, scale=0.088, S=1, ws=None, wsb=0, out=FAKE,
             osb=32 * 128, osh=128)
    a.update(kw)
    return lib.decode_attn_paged_masked(a["q"], a["qsb"], a["qsh"], a["k"], a["v"], a["P"], a["ps"], a["table"],
                                        a["maxp"], a["lens"], a["mask"], a["mst"], a["maxlen"], a["B"], a["Hq"],
                                        a["Hkv"], a["D"], a["scale"], a["S"], a["ws"], a["wsb"], a["out"], a["osb"],
                                        a["osh"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=-1), 2), (dict(maxlen=8 * 16 + 1), 2), (dict(mst=96), 2), (dict(S=-2), 2), (dict(S=-1), 3),
    (dict(mask=None), 1), (dict(q=None), 1), (dict(table=None), 1),
    (dict(D=96), 3), (dict(D=48, qsb=32 * 48, qsh=48, osb=32 * 48, osh=48), 3),
    (dict(mst=120), 5), (dict(mask=ctypes.c_void_p((1 << 20) + 8)), 5),
    (dict(S=4), 4),
])
def test_masked_validation(lib, kw, status):
    assert masked_call(lib, **kw) == status


def test_masked_empty_batch_is_a_no_op(lib):
    assert masked_call(lib, B=0, q=None, out=None, lens=None, mask=None, k=None, table=None) == 0


# ---- the binding refuses tensors the kernels could not use ---------------------------------

def test_binding_refuses_cpu_tensors_before_any_launch():
    """A CPU tensor would reach the kernels as a host address; the binding raises DapError
    (status None) before the library is called."""
    import torch
    from paged_kv_cache_298_gb300 import inputs
    case = inputs.tiny_paged()                      # every tensor on the CPU
    kw = dict(max_kv_len=case.max_kv_len, num_splits=1)
    with pytest.raises(binding.DapError) as e:
        binding.decode_attn_paged(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens, **kw)
    assert e.value.status is None and "CUDA" in str(e.value)
    with pytest.raises(binding.DapError):
        binding.decode_attn_paged_noalloc(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                          max_kv_len=case.max_kv_len)
    f = inputs.make_fp8_case(1, 128, 512, 2, 16, 8, 5)
    with pytest.raises(binding.DapError):
        binding.decode_attn_paged_fp8(f.q, f.kv_cache, f.inv_scale, f.indices, f.lens)
    with pytest.raises(binding.DapError):
        binding.kv_append_paged(case.q[:, :2], case.q[:, :2], case.k_cache, case.v_cache, case.block_table,
                                case.seq_lens)
    del torch


class _Fake:
    """Stands in for a tensor or stream on a given device (only what the binding's device
    rule reads), so the rule can be checked without a GPU."""

    def __init__(self, kind, index=None):
        import torch
        self.is_cuda = kind == "cuda"
        self.device = torch.device(kind, index) if index is not None else torch.device(kind)


def test_binding_refuses_tensors_and_streams_on_another_device():
    import torch
    dev = binding._device_of("call", _Fake("cuda", 0), k=_Fake("cuda", 0), workspace=None)
    assert dev == torch.device("cuda", 0)
    with pytest.raises(binding.DapError) as e:
        binding._device_of("call", _Fake("cuda", 0), k=_Fake("cuda", 0), v=_Fake("cuda", 1))
    assert e.value.status is None and "v is on cuda:1" in str(e.value)
    with pytest.raises(binding.DapError) as e:
        binding._device_of("call", _Fake("cuda", 0), out=_Fake("cpu"))
    assert "out is not a CUDA tensor" in str(e.value)
    with pytest.raises(binding.DapError):
        binding._stream(_Fake("cuda", 1), torch.device("cuda", 0))
