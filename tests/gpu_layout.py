"""Test-side conversion of the library's device layouts (include/fsa.h) into the
oracle's logical layouts (one code byte per element, one scale byte per block).
Pure re-indexing: no arithmetic of the method."""
import numpy as np


def _unpack6(groups):
    """[..., 16] bytes (12 packed + 4 pad) -> [..., 16] 6-bit codes, LSB first."""
    b = groups[..., :12].astype(np.uint32)
    out = np.empty(groups.shape[:-1] + (16,), np.uint8)
    for t in range(4):                       # 4 triplets of 3 bytes = 4 codes each
        w = b[..., 3 * t] | (b[..., 3 * t + 1] << 8) | (b[..., 3 * t + 2] << 16)
        for e in range(4):
            out[..., 4 * t + e] = (w >> (6 * e)) & 0x3F
    return out


def unpack_codes(raw, fmt, n_elems):
    """raw: [..., row_bytes] -> [..., n_elems] logical codes."""
    if fmt == 0:
        return raw[..., :n_elems].copy()
    if fmt in (1, 4):
        g = raw.reshape(raw.shape[:-1] + (raw.shape[-1] // 16, 16))
        assert not g[..., 12:].any(), "6-bit group padding bytes must be zero"
        return _unpack6(g).reshape(raw.shape[:-1] + (-1,))[..., :n_elems]
    lo, hi = raw & 0x0F, raw >> 4
    return np.stack([lo, hi], axis=-1).reshape(raw.shape[:-1] + (-1,))[..., :n_elems]


def unpack_rows(codes, scales, fmt, B, H, S, D):
    """FSA_MX_ROWS device buffers -> (codes [B,H,S,D], scales [B,H,S,D/32]); checks padding slots.
    fmt 5 (NVFP4): scales [B,H,S,D/16] from D/64 atoms per tile (rows past S: 0x38)."""
    if fmt == 5:
        return _unpack_rows_nvfp4(codes, scales, B, H, S, D)
    rb = D if fmt in (0, 1, 4) else D // 2
    c = unpack_codes(np.asarray(codes).reshape(B, H, S, rb), fmt, D)
    nt = (S + 127) // 128
    flat = np.asarray(scales).reshape(-1)
    assert flat.size == B * H * nt * 512
    s_idx = np.arange(S)
    off = (s_idx // 128) * 512 + (s_idx % 32) * 16 + ((s_idx % 128) // 32) * 4                 # [S]
    idx = (np.arange(B * H) * nt * 512)[:, None, None] + off[None, :, None] + np.arange(D // 32)[None, None, :]
    sc = flat[idx].reshape(B, H, S, D // 32)
    used = np.zeros(flat.size, bool)
    used[idx.reshape(-1)] = True
    assert np.all(flat[~used] == 0x7F), "unused scale slots must be 0x7F"
    return c, sc


def _unpack_rows_nvfp4(codes, scales, B, H, S, D):
    c = unpack_codes(np.asarray(codes).reshape(B, H, S, D // 2), 2, D)
    nt, na = (S + 127) // 128, D // 64
    flat = np.asarray(scales).reshape(-1)
    assert flat.size == B * H * nt * na * 512
    s_idx = np.arange(S)
    blk = np.arange(D // 16)
    off = ((s_idx // 128) * na * 512 + (s_idx % 32) * 16 + ((s_idx % 128) // 32) * 4)[:, None] + \
          (blk // 4 * 512 + blk % 4)[None, :]                                                   # [S, D/16]
    idx = (np.arange(B * H) * nt * na * 512)[:, None, None] + off[None]
    sc = flat[idx].reshape(B, H, S, D // 16)
    used = np.zeros(flat.size, bool)
    used[idx.reshape(-1)] = True
    assert np.all(flat[~used] == 0x38), "scale slots of rows past S must be 0x38"
    return c, sc


def unpack_cols(codes, scales, fmt, B, H, S, D):
    """FSA_MX_COLS_T device buffers -> (codes [B,H,D,S32], scales [B,H,D,S32/32]), S32 = S rounded up to 32."""
    Sp = (S + 127) // 128 * 128
    S32 = (S + 31) // 32 * 32
    rb = Sp if fmt in (0, 1, 4) else Sp // 2
    c = unpack_codes(np.asarray(codes).reshape(B, H, D, rb), fmt, Sp)
    assert not c[..., S:].any(), "codes past the sequence end must be zero"
    nt = Sp // 128
    flat = np.asarray(scales).reshape(-1)
    assert flat.size == B * H * nt * 512
    d = np.arange(D)
    blk = np.arange(Sp // 32)
    off = (blk // 4 * 512 + blk % 4)[None, :] + ((d % 32) * 16 + (d // 32) * 4)[:, None]         # [D, nblk]
    idx = (np.arange(B * H) * nt * 512)[:, None, None] + off[None]
    sc = flat[idx].reshape(B, H, D, Sp // 32)
    assert np.all(sc[..., S32 // 32:] == 0x7F), "blocks past the sequence end hold 0x7F"
    used = np.zeros(flat.size, bool)
    used[idx.reshape(-1)] = True
    assert np.all(flat[~used] == 0x7F), "unused scale slots must be 0x7F"
    return c[..., :S32], sc[..., :S32 // 32]
