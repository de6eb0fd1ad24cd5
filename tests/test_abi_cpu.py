"""The C-ABI library loads and exports every declared symbol; host-side logic (no GPU)."""
import ctypes
import os
import re

import numpy as np
import pytest

import nvfp4_grouped_gemm_gb300 as moe
from nvfp4_grouped_gemm_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_native.lib_path()):
        import nvfp4_grouped_gemm_gb300.build as b
        b.build()
    return _native.load()


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    bound = {s[0] for s in _native.SIGNATURES}
    assert set(names) <= bound | set(), set(names) - bound


def test_status_strings(lib):
    for code, name in _native.STATUS.items():
        assert lib.moe_status_string(code).decode() == name
    assert lib.moe_status_string(99).decode() == "MOE_ERR_UNKNOWN"


def test_workspace_layout_host_logic(lib):
    H, F, E, k = 2560, 640, 512, 10
    for T in (1, 8, 128):
        L = moe.workspace_layout(T, H, F, E, k, moe.PATH_DECODE)
        P = T * k
        assert L["error_word"] == 0 and L["pair_pos"] == 256
        assert L["h"] >= L["pair_pos"] + 4 * P
        assert L["partial"] >= L["h"] + 4 * P * F
        assert L["total"] == moe.workspace_bytes(T, H, F, E, k, moe.PATH_DECODE)
        for v in L.values():
            assert v % 256 == 0
    Lp = moe.workspace_layout(4096, 4096, 640, 288, 8, moe.PATH_PREFILL)
    assert Lp["qx_codes"] > 0 and Lp["qh_codes"] > 0
    assert moe.workspace_bytes(0, H, F, E, k) == 0
    assert moe.workspace_bytes(4, 100, F, E, k) == 0        # H % 256 != 0 unsupported
    assert moe.workspace_bytes(4, 8192, F, E, k) == 0       # H > 4096 unsupported
    assert moe.workspace_bytes(4, H, F, 8, 10) == 0         # k > E
    # per-path F limits: decode up to 1408, prefill up to 4096
    assert moe.workspace_bytes(4, H, 1408, E, k, moe.PATH_DECODE) > 0
    assert moe.workspace_bytes(4, H, 1472, E, k, moe.PATH_DECODE) == 0
    assert moe.workspace_bytes(4, H, 1472, E, k, moe.PATH_PREFILL) > 0
    assert moe.workspace_bytes(4, H, 4160, E, k, moe.PATH_PREFILL) == 0
    # the tensor-core decode form (from 256 pairs) cannot stage F = 1088, 1216, 1344
    for f in range(64, 1409, 64):
        small = moe.workspace_bytes(4, H, f, E, k, moe.PATH_DECODE)
        wide = moe.workspace_bytes(64, H, f, E, k, moe.PATH_DECODE)
        assert small > 0
        assert (wide == 0) == (f in (1088, 1216, 1344)), f


def test_path_resolution(lib):
    th = moe.prefill_min_pairs()
    assert moe.resolve_path(1, 10) == moe.PATH_DECODE
    assert moe.resolve_path(th, 1) == moe.PATH_PREFILL
    assert moe.resolve_path(th - 1, 1) == moe.PATH_DECODE
    assert moe.resolve_path(4096, 8, moe.PATH_DECODE) == moe.PATH_DECODE


def test_host_validation_rejects_before_launch(lib):
    """Null pointers and bad sizes are rejected on the host (no CUDA call is made)."""
    assert lib.moe_route_topk(None, 4, 16, 2, None, None, None) == 1
    assert lib.moe_route_topk(8, 4, 16, 20, 8, 8, None) == 1            # k > E
    assert lib.moe_route_topk(8, 4, 16, 64, 8, 8, None) == 1
    assert lib.moe_route_topk(16, 4, 64, 40, 16, 16, None) == 2         # k > 32
    csr = _native.CSR(None, None, None, None)
    assert lib.moe_build_expert_csr(16, 4, 2, 16, csr, 256, 1 << 20, None) == 1
    good = _native.CSR(16, 16, 16, 16)
    assert lib.moe_build_expert_csr(16, 4, 2, 2048, good, 256, 1 << 20, None) == 2   # E > 1024
    assert lib.moe_build_expert_csr(16, 4, 2, 16, good, None, 0, None) == 3
    assert lib.moe_build_expert_csr(16, 4, 2, 16, good, 258, 1 << 20, None) == 3     # misaligned
    bank = _native.Bank(16, 16, 16, 128, 256)
    # x misaligned
    assert lib.moe_grouped_gate_up_silu_nvfp4(8, 4, 256, 64, 2, ctypes.byref(bank), good, 0,
                                              256, 1 << 20, None) == 1
    # rows mismatch (2F = 128 expected, bank says 128 ok; give F=96 -> unsupported F%64)
    assert lib.moe_grouped_gate_up_silu_nvfp4(16, 4, 256, 96, 2, ctypes.byref(bank), good, 0,
                                              256, 1 << 20, None) == 2
    # workspace too small
    assert lib.moe_grouped_gate_up_silu_nvfp4(16, 4, 256, 64, 2, ctypes.byref(bank), good, 0,
                                              256, 16, None) == 3
    # F beyond the decode path's limit
    wide = _native.Bank(16, 16, 16, 2 * 2048, 256)
    assert lib.moe_grouped_gate_up_silu_nvfp4(16, 4, 256, 2048, 2, ctypes.byref(wide), good, 1,
                                              256, 1 << 30, None) == 2
    # interleaved import: null, in_f not a multiple of 64, misaligned codes
    assert lib.moe_nvfp4_from_interleaved(None, 4, 128, 16, 16, None) == 1
    assert lib.moe_nvfp4_from_interleaved(16, 4, 96, 16, 16, None) == 1
    assert lib.moe_nvfp4_from_interleaved(16, 4, 128, 24, 16, None) == 1
    assert lib.moe_nvfp4_from_interleaved(16, 0, 128, 16, 16, None) == 1
    dbank = _native.Bank(16, 16, 16, 256, 64)
    assert lib.moe_grouped_down_combine_nvfp4(ctypes.byref(dbank), good, 16, 4, 256, 64, 2, 0,
                                              None, 256, 1 << 20, None) == 1


def test_prepack_sizes_and_validation(lib):
    """The prepacked scale plane is as large as the planar one; sizes it cannot tile, null
    or misaligned pointers, a short buffer, an unknown order, and a bank whose plane was
    written in the other call's row order are rejected on the host (no CUDA call)."""
    assert lib.moe_nvfp4_sf_atoms_bytes(512, 1280, 2560) == 512 * 1280 * 2560 // 16
    assert lib.moe_nvfp4_sf_atoms_bytes(288, 4096, 640) == 288 * 4096 * 640 // 16
    assert lib.moe_nvfp4_sf_atoms_bytes(4, 192, 256) == 0          # rows % 128
    assert lib.moe_nvfp4_sf_atoms_bytes(4, 256, 96) == 0           # in_f % 64
    assert lib.moe_nvfp4_sf_atoms_bytes(0, 256, 256) == 0
    n = 4 * 256 * 256 // 16
    GU, ROWS = moe.SF_ATOMS_GATE_UP, moe.SF_ATOMS_ROWS
    assert lib.moe_nvfp4_prepack_sf(None, 4, 256, 256, GU, 256, n, None) == 1
    assert lib.moe_nvfp4_prepack_sf(256, 4, 256, 256, GU, None, n, None) == 1
    assert lib.moe_nvfp4_prepack_sf(256, 4, 256, 256, GU, 256, n - 16, None) == 1
    assert lib.moe_nvfp4_prepack_sf(256, 4, 256, 256, 3, 256, n, None) == 1
    assert lib.moe_nvfp4_prepack_sf(256, 4, 256, 256, ROWS, 264, n, None) == 1
    assert lib.moe_nvfp4_prepack_sf(256, 4, 192, 256, ROWS, 256, n, None) == 1
    good = _native.CSR(16, 16, 16, 16)
    # a gate/up bank (rows = 2F = 128, in_f = H = 256) carrying a down-order plane, and a
    # misaligned plane
    wrong = _native.Bank(16, 16, 16, 128, 256, None, 256, ROWS)
    assert lib.moe_grouped_gate_up_silu_nvfp4(16, 4, 256, 64, 2, ctypes.byref(wrong), good, 0,
                                              256, 1 << 30, None) == 1
    odd = _native.Bank(16, 16, 16, 128, 256, None, 264, GU)
    assert lib.moe_grouped_gate_up_silu_nvfp4(16, 4, 256, 64, 2, ctypes.byref(odd), good, 0,
                                              256, 1 << 30, None) == 1
    dwrong = _native.Bank(16, 16, 16, 256, 64, None, 256, GU)
    assert lib.moe_grouped_down_combine_nvfp4(ctypes.byref(dwrong), good, 16, 4, 256, 64, 2, 0,
                                              256, 256, 1 << 30, None) == 1


def test_kernel_launch_count_host_logic(lib):
    """The per-layer kernel count the library reports follows its own launch plan: decode
    below 256 pairs runs x-gather, gate/up, h-prep, down and combine after the CSR; from 256
    pairs it runs x slices, the gate/up GEMM, h slices, the down GEMM and the combine;
    prefill runs Q(x), the gate/up GEMM, Q(h), the down GEMM and the combine (the CSR call
    writes the tile lists of both tensor-core forms); the CSR is one kernel below 4096 pairs
    and three from there on."""
    assert moe.kernel_launches(8, 2560, 640, 512, 10) == 1 + 5
    assert moe.decode_tensor_core_min_pairs() == 256
    assert moe.kernel_launches(25, 2560, 640, 256, 10) == 1 + 5
    assert moe.kernel_launches(26, 2560, 640, 256, 10) == 1 + 5
    assert moe.kernel_launches(128, 2560, 640, 256, 10) == 1 + 5
    assert moe.kernel_launches(4096, 4096, 640, 288, 8) == 3 + 5
    assert moe.kernel_launches(4, 256, 64, 16, 2, moe.PATH_PREFILL) == 1 + 5
    assert moe.kernel_launches(0, 256, 64, 16, 2) == 0


@pytest.mark.parametrize("path,rpp,tile_rows,region_name",
                         [(moe.PATH_PREFILL, 1, 128, "tiles"), (moe.PATH_DECODE, 4, 32, "slice_tiles")])
def test_tile_list_always_fits_its_workspace_region(lib, path, rpp, tile_rows, region_name):
    """Each tile list (a count, then one 16-byte record per tile) never outgrows the
    workspace region the layout gives it: an expert with m pairs needs ceil(m*rpp/tile_rows)
    tiles, at most m*rpp/tile_rows + 1, and at most min(E, P) experts are active.  Both
    regions sit before h at offsets that depend only on P and E (the CSR call writes them
    without knowing H, F or the path)."""
    rng = np.random.default_rng(23)
    H, F = 256, 64
    for _ in range(200):
        E = int(rng.integers(1, 1025))
        k = int(rng.integers(1, min(E, 32) + 1))
        T = int(rng.integers(1, 600))
        if path == moe.PATH_DECODE and T * k < moe.decode_tensor_core_min_pairs():
            T = (moe.decode_tensor_core_min_pairs() + k - 1) // k
        P = T * k
        L = moe.workspace_layout(T, H, F, E, k, path)
        L2 = moe.workspace_layout(T, 4096, 640, E, k, moe.PATH_PREFILL if path == moe.PATH_DECODE
                                  else moe.PATH_DECODE)
        for n in ("error_word", "pair_pos", "tiles", "slice_tiles", "h"):
            assert L[n] == L2[n]
        start = L[region_name]
        ends = sorted(v for n, v in L.items() if n != "total" and v > start) + [L["total"]]
        region = ends[0] - start
        skew = rng.uniform(0.5, 3.0)
        ids = np.minimum((rng.uniform(size=P) ** skew * E).astype(np.int64), E - 1)
        counts = np.bincount(ids, minlength=E)
        tiles = int(np.sum((counts * rpp + tile_rows - 1) // tile_rows))
        assert 16 + 16 * tiles <= region, (T, k, E, tiles, region)


@pytest.mark.parametrize("gate_up", [True, False])
def test_prepack_layout_restatement_against_the_definition(gate_up):
    """The numpy restatement the GPU prepack tests compare with, against a plain loop over
    the layout's definition in include/moe.h (every byte of a small bank, both orders)."""
    from prepack_layout import expected_atoms
    rng = np.random.default_rng(7)
    E, R, K = 2, 256, 192
    S = K // 16
    scales = rng.integers(0, 127, size=(E, R, S), dtype=np.uint8)
    got = expected_atoms(scales, gate_up)
    tiles, kst = R // 128, K // 64
    want = np.zeros(E * tiles * kst * 512, np.uint8)
    for e in range(E):
        for t in range(tiles):
            for j in range(kst):
                a = (e * tiles + t) * kst + j
                for r in range(32):
                    for x in range(4):
                        m = 32 * x + r
                        if gate_up:
                            row = (R // 2 if m % 2 else 0) + 64 * t + m // 2
                        else:
                            row = 128 * t + m
                        for b in range(4):
                            want[a * 512 + 16 * r + 4 * x + b] = scales[e, row, 4 * j + b]
    assert np.array_equal(got, want)
