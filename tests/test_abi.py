"""The C-ABI library on a machine without a GPU: it builds, loads, exports every
symbol the public header declares, validates arguments before touching CUDA,
and its host-side task order is dependency-safe."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from transformer_ffn_gb300 import build
    build.build()
    import transformer_ffn_gb300 as tffn
    return tffn.load()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "tffn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("ffn_forward", "moe_ffn_forward", "tffn_workspace_bytes", "tffn_set_workspace",
              "tffn_check", "tffn_status_string", "tffn_set_option"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), f"missing export {n}"


def test_status_strings(lib):
    for code in range(-6, 1):
        s = lib.tffn_status_string(code)
        assert s and s != b"unknown status"
    assert lib.tffn_status_string(-99) == b"unknown status"


def _ffn(lib, X=16, W1=16, W2=16, Y=16, M=64, N=256, O=1024, P=256, act1=2, act2=0, b1=None, b2=None):
    return lib.ffn_forward(X, W1, b1, W2, b2, act1, act2, M, N, O, P, Y, None)


def test_ffn_validation_without_gpu(lib):
    bad = -1
    assert _ffn(lib, X=None) == bad
    assert _ffn(lib, W1=None) == bad
    assert _ffn(lib, W2=None) == bad
    assert _ffn(lib, Y=None) == bad
    assert _ffn(lib, N=12) == bad          # not a multiple of 8
    assert _ffn(lib, O=0) == bad
    assert _ffn(lib, P=4) == bad
    assert _ffn(lib, M=-1) == bad
    assert _ffn(lib, act1=7) == bad
    assert _ffn(lib, act2=-1) == bad
    assert _ffn(lib, X=24) == bad          # 8-byte aligned only
    assert _ffn(lib, b1=40) == bad
    assert _ffn(lib, M=0) == 0             # empty call: nothing to do, no launch
    assert _ffn(lib, M=0, X=None, Y=None) == 0
    assert lib.tffn_last_launch_count() == 0


def test_moe_validation_without_gpu(lib):
    E = 4
    arr = (ctypes.c_void_p * E)(*([16] * E))
    p = ctypes.cast(arr, ctypes.c_void_p)

    def call(top_k=2, E=E, T=32, N=64, w1=p, X=16, logits=16):
        return lib.moe_ffn_forward(X, logits, top_k, w1, None, p, None, 16, T, N, 64, 64, E, 2, 0,
                                   None, None)
    assert call(top_k=0) == -1
    assert call(top_k=5) == -1
    assert call(E=0, top_k=1) == -1
    assert call(E=65, top_k=1) == -1
    assert call(N=20) == -1
    assert call(X=None) == -1
    assert call(logits=None) == -1
    zeros = (ctypes.c_void_p * E)(*([16, 0, 16, 16]))
    assert call(w1=ctypes.cast(zeros, ctypes.c_void_p)) == -1
    assert call(T=0) == 0
    assert call(T=0, X=None, logits=None) == 0


def test_workspace_bytes_holds_hidden_tensor(lib):
    import json
    with open(os.path.join(ROOT, "tests", "golden", "page1_llama3_70b_sizes.json")) as f:
        g = json.load(f)
    # one GPU's slice of the page's Llama 3 70B example: H^(g) is 56 MiB in bf16
    tokens, cols = g["tokens"], g["hidden_cols_per_gpu"]
    assert tokens * cols * 2 == g["hidden_slice_mib"] * 2**20
    ws = lib.tffn_workspace_bytes(tokens, g["N"], cols, g["P"], 0, 0)
    assert ws >= g["hidden_slice_mib"] * 2**20
    assert ws < (g["hidden_slice_mib"] + 16) * 2**20
    # invalid shapes report 0
    assert lib.tffn_workspace_bytes(tokens, 12, cols, 8, 0, 0) == 0


def test_engine_task_order_is_dependency_safe(lib):
    import transformer_ffn_gb300 as tffn
    for (mb, n1, n2, gm) in [(1, 4, 1, 8), (3, 5, 2, 1), (9, 7, 3, 4), (17, 3, 5, 8), (32, 64, 16, 8),
                             (5, 1, 1, 16), (40, 2, 9, 3)]:
        total, _ = tffn.debug_engine_task(mb, n1, n2, gm, 0)
        assert total == mb * (n1 + n2)
        seen = set()
        done_l1 = {}
        for t in range(total):
            tot_t, (layer, band, tile) = tffn.debug_engine_task(mb, n1, n2, gm, t)
            assert tot_t == total     # -1: the kernel's 32-bit mapping disagrees
            assert layer in (0, 1)
            assert 0 <= band < mb
            assert (layer, band, tile) not in seen
            seen.add((layer, band, tile))
            if layer == 0:
                assert 0 <= tile < n1
                done_l1[band] = done_l1.get(band, 0) + 1
            else:
                assert 0 <= tile < n2
                # every layer-1 tile of this band has a smaller ticket
                assert done_l1.get(band, 0) == n1
        assert len(seen) == total
        tot_t, (layer, _, _) = tffn.debug_engine_task(mb, n1, n2, gm, total)
        assert tot_t == total and layer == -1


def test_engine_task_32bit_form_at_scale(lib):
    """The kernel's 32-bit ticket arithmetic against the 64-bit form on
    launches with hundreds of thousands of tickets (sampled tickets, every
    segment boundary of the first and last groups)."""
    import random
    import transformer_ffn_gb300 as tffn
    rnd = random.Random(3)
    for (mb, n1, n2, gm) in [(4096, 112, 32, 8), (8191, 64, 16, 4), (2000, 7, 300, 3), (65536, 4, 1, 16)]:
        total, _ = tffn.debug_engine_task(mb, n1, n2, gm, 0)
        assert total == mb * (n1 + n2)
        first = min(gm, mb)
        picks = set(rnd.randrange(total) for _ in range(2000))
        picks |= {0, first * n1 - 1, first * n1, total - 1, total - first * n2, max(total - first * n2 - 1, 0)}
        for t in sorted(picks):
            tot_t, (layer, band, tile) = tffn.debug_engine_task(mb, n1, n2, gm, t)
            assert tot_t == total, (mb, n1, n2, gm, t)
            assert layer in (0, 1) and 0 <= band < mb
            assert 0 <= tile < (n1 if layer == 0 else n2)


def test_debug_tiles(lib):
    import transformer_ffn_gb300 as tffn
    t = tffn.debug_tiles()
    assert t["BM"] in (128, 256) and t["BN"] % 64 == 0 and t["BK"] == 64
    assert t["decode_slice"] == t["decode_kc"]


def test_ops_fail_loudly_without_library(monkeypatch, tmp_path):
    import transformer_ffn_gb300 as tffn
    monkeypatch.setattr(tffn, "_lib", None)
    monkeypatch.setattr(tffn, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        tffn.load()


def _owned_blocks(nblk, grid):
    return [(c * nblk // grid, (c + 1) * nblk // grid) for c in range(grid)]


def _check_stream_k(U, G, kch, maxp):
    # contiguous ranges of U units over G CTAs: a partition, sizes within one,
    # every CTA with at least one unit, no slice split over more than maxp CTAs
    starts = [c * U // G for c in range(G + 1)]
    assert starts[0] == 0 and starts[-1] == U
    sizes = [b - a for a, b in zip(starts, starts[1:])]
    assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    owners = {}
    for c in range(G):
        for s in range(starts[c] // kch, (starts[c + 1] - 1) // kch + 1):
            owners.setdefault(s, set()).add(c)
    assert max(len(v) for v in owners.values()) <= maxp


@pytest.mark.parametrize("path,M,N,O,P,glu", [
    (2, 16, 8192, 28672, 8192, False), (2, 16, 4096, 14336, 4096, True), (2, 32, 4096, 14336, 4096, True),
    (2, 8, 512, 20480, 256, True), (2, 1, 256, 384, 136, True), (2, 64, 1024, 2048, 512, True),
    (6, 128, 4096, 14336, 4096, False), (6, 128, 4096, 14336, 4096, True), (6, 256, 4096, 14336, 4096, False),
    (6, 128, 8192, 28672, 8192, False), (6, 64, 256, 40960, 264, False), (6, 100, 256, 20480, 264, True),
    (6, 65, 136, 520, 264, False), (6, 1, 256, 264, 72, False),
])
@pytest.mark.parametrize("sms", [152, 148, 132])
def test_stream_plans(lib, path, M, N, O, P, glu, sms):
    import transformer_ffn_gb300 as tffn
    pl = tffn.debug_stream_plan(path, M, N, O, P, sms, glu)
    G, win, nblk = pl["grid"], pl["win"], pl["nblk"]
    assert 1 <= G <= sms
    assert nblk == (O + 63) // 64
    # layer 2 is always Stream-K over its slices
    cols2 = 128 if path == 2 else 256
    kc2 = 128 if path == 2 else 64
    assert pl["slices1"] == (P + cols2 - 1) // cols2 and pl["kch1"] == (O + kc2 - 1) // kc2
    assert pl["units1"] == pl["slices1"] * pl["kch1"] and G <= pl["units1"]
    _check_stream_k(pl["units1"], G, pl["kch1"], pl["maxp1"])
    # the window layer 1: when it is used and how much each CTA owns
    if path == 2:
        expect = 1 if (glu and M <= 32 and nblk <= 2 * G) else 0
    else:
        expect = 1 if nblk <= 2 * G else (2 if (not glu and nblk <= 4 * G) else 0)
    assert win == expect
    if win:
        owned = _owned_blocks(nblk, G)
        assert max(b - a for a, b in owned) <= 2 * win
        assert owned[0][0] == 0 and owned[-1][1] == nblk
        assert all(owned[i][1] == owned[i + 1][0] for i in range(G - 1))
        assert pl["maxp0"] == 1   # the window is never split, on either stream
    else:
        assert pl["units0"] == pl["slices0"] * pl["kch0"] and G <= pl["units0"]
        _check_stream_k(pl["units0"], G, pl["kch0"], pl["maxp0"])
    # the split-K partial area holds every split slice's parts
    rows = (32 if M <= 32 else 64) if path == 2 else (32 if M <= 32 else 64 if M <= 64 else 128 if M <= 128 else 256)
    part = rows * (128 if path == 2 else 256) * 4
    need = 0
    for l in (0, 1):
        if l == 0 and win:
            continue
        if pl[f"maxp{l}"] > 1:
            need += pl[f"slices{l}"] * pl[f"maxp{l}"] * part
    assert pl["partial_bytes"] >= need


def test_stream_plan_validation(lib):
    import transformer_ffn_gb300 as tffn
    with pytest.raises(tffn.TffnError):
        tffn.debug_stream_plan(6, 257, 64, 64, 64, 152)
    with pytest.raises(tffn.TffnError):
        tffn.debug_stream_plan(3, 16, 64, 64, 64, 152)


def test_timing_sample_and_options_without_gpu(lib):
    # the sampling interval of the dominant-kernel timing is validated on the
    # host; the MoE combine option round-trips like the others
    lib.tffn_timing_sample.argtypes = [ctypes.c_int]
    lib.tffn_timing_sample.restype = ctypes.c_int
    assert lib.tffn_timing_sample(0) == -1
    assert lib.tffn_timing_sample(-3) == -1
    assert lib.tffn_timing_sample(4) == 0
    assert lib.tffn_timing_sample(1) == 0
    lib.tffn_set_option.argtypes = [ctypes.c_int, ctypes.c_int64]
    lib.tffn_set_option.restype = ctypes.c_int64
    prev = lib.tffn_set_option(6, 0)          # TFFN_OPT_MOE_COMBINE
    assert prev == 1                          # fused by default
    assert lib.tffn_set_option(6, prev) == 0
    prev = lib.tffn_set_option(4, 0)          # TFFN_OPT_GROUP_M: 0 = chosen by shape
    assert lib.tffn_set_option(4, prev) == 0


def test_noalloc_validation_without_gpu(lib):
    # argument errors come back before any CUDA call; the error query fails
    # cleanly (TFFN_ERR_CUDA) when there is no device to synchronise
    fn = lib.ffn_forward_decode_noalloc
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i64, i64, i64, i64, vp, vp]
    fn.restype = i32
    p = ctypes.c_void_p(1 << 20)
    assert fn(p, p, None, p, None, 1, 0, 33, 64, 64, 64, p, None) == -1     # more than 32 rows
    assert fn(p, p, None, p, None, 1, 0, 16, 60, 64, 64, p, None) == -1     # N not a multiple of 8
    assert fn(p, p, None, p, None, 9, 0, 16, 64, 64, 64, p, None) == -1     # unknown activation
    assert fn(None, None, None, None, None, 1, 0, 0, 64, 64, 64, None, None) == 0   # empty call
    chk = lib.tffn_check_noalloc
    chk.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    chk.restype = i32
    import torch
    if not torch.cuda.is_available():
        detail = (ctypes.c_int32 * 4)(7, 7, 7, 7)
        assert chk(None, detail) == -3
        assert list(detail) == [0, 0, 0, 0]
