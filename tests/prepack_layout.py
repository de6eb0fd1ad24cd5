"""The prepacked scale-factor layout of moe_nvfp4_prepack_sf, restated with numpy for the
tests: byte 16r + 4x + b of atom (e, t, j) is scale byte 4j + b of tile row 32x + r, where
tile t's row m is bank row 128t + m, or for a gate/up bank gate row 64t + m/2 (even m) and
up row F + 64t + m/2 (odd m)."""
import numpy as np


def expected_atoms(scales: np.ndarray, gate_up: bool) -> np.ndarray:
    """The atoms of a planar scale plane [E, rows, in_f/16], as one flat u8 array."""
    E, R, S = scales.shape
    tiles, kst = R // 128, S // 4
    m = np.arange(128)
    if gate_up:
        F = R // 2
        rows = 64 * np.arange(tiles)[:, None] + (np.where(m % 2 == 1, F, 0) + m // 2)[None, :]
    else:
        rows = 128 * np.arange(tiles)[:, None] + m[None, :]
    w = scales[:, rows, :].reshape(E, tiles, 4, 32, kst, 4)      # [e, t, x, r, j, b]
    return np.ascontiguousarray(w.transpose(0, 1, 4, 3, 2, 5)).reshape(-1)
