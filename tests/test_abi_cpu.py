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
    bal = binding.workspace_bytes(128, 32, 8, 128, 0)
    assert bal >= 2 * 1024 * 4 * (128 + 2) * 4 + 128 * 8 * 8
    assert bal < 8 << 20
    assert binding.workspace_bytes(5000, 32, 8, 128, 0) == 0      # huge batches run one CTA per unit
    assert binding.workspace_bytes(16, 32, 8, 128, -1) == 0


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
    (dict(maxlen=8 * 16 + 1), 2), (dict(ps=0), 2), (dict(P=0), 2), (dict(S=-1), 2),
    (dict(scale=float("nan")), 2), (dict(qsh=-8), 2),
    (dict(q=None), 1), (dict(out=None), 1), (dict(k=None), 1), (dict(table=None), 1),
    (dict(lens=None), 1),
    (dict(D=96), 3), (dict(Hq=48, Hkv=3), 3), (dict(Hq=64, Hkv=4), 3),
    (dict(q=ctypes.c_void_p((1 << 20) + 8)), 5), (dict(qsh=130), 5), (dict(osb=4100), 5),
    (dict(k=ctypes.c_void_p((1 << 20) + 4)), 5),
    (dict(S=4), 4), (dict(S=4, ws=FAKE, wsb=16), 4), (dict(S=0), 4),
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
