"""Host logic of the one-kernel decode layer: which sizes it takes, its workspace words and
its argument checks (no GPU needed: nothing is launched for a refused call)."""
import pytest

import nvfp4_grouped_gemm_gb300 as moe
from nvfp4_grouped_gemm_gb300 import _native


def test_supported_sizes():
    H, F, E, k = 2560, 640, 512, 10
    for T in (1, 2, 4, 8, 16, 25):
        assert moe.decode_layer_supported(T, H, F, E, k), T
    assert not moe.decode_layer_supported(26, H, F, E, k)        # 260 pairs: tensor-core form
    assert not moe.decode_layer_supported(33, H, F, E, 1)        # more tokens than routed per CTA
    assert moe.decode_layer_supported(32, H, F, E, 1)
    assert not moe.decode_layer_supported(4, H, 704, E, k)       # F > 640
    assert not moe.decode_layer_supported(4, H, 576, E, k)       # F % 128 != 0
    assert moe.decode_layer_supported(4, H, 128, E, k)
    assert moe.decode_layer_supported(4, 4096, 256, 1024, 32)
    assert not moe.decode_layer_supported(4, 100, F, E, k)       # H % 256 != 0
    assert not moe.decode_layer_supported(0, H, F, E, k)
    assert not moe.decode_layer_supported(4, H, F, 8, k)         # k > E


def test_sync_words_in_the_decode_layout():
    """The barrier words sit after every other decode region, so no offset the CSR call
    relies on moves; other paths have none."""
    L = moe.workspace_layout(8, 2560, 640, 512, 10, moe.PATH_DECODE)
    others = [v for n, v in L.items() if n not in ("total", "sync")]
    assert L["sync"] > max(others) and L["sync"] + 48 <= L["total"]
    assert L["pair_pos"] == 256
    Lp = moe.workspace_layout(4096, 4096, 640, 288, 8, moe.PATH_PREFILL)
    assert Lp["sync"] == 0


def test_refused_arguments_launch_nothing():
    lib = _native.load()
    bank = _native.Bank(None, None, 512, 1280, 2560, None)
    st = lib.moe_decode_layer_nvfp4(None, None, None, None, 8, 2560, 640, 10, bank, bank, None,
                                    None, 0, None)
    assert _native.STATUS[st] == "MOE_ERR_INVALID_ARG"
