"""Helpers shared by the GPU tests: moving seeded numpy inputs to the device
and reading results back (plumbing only)."""
import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in BF16 ulps between two BF16 bit arrays (sign-magnitude order)."""
    def key(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    return np.abs(key(a_bits) - key(b_bits))


def unpack_weights(packed: np.ndarray, N: int, K: int) -> np.ndarray:
    """Row-major [N][K] INT8 codes from the packed layout documented in
    include/quasar.h (128 x 128 blocks, tile-major, 16-byte chunks of row r
    stored at chunk position c ^ (r % 8), bytes holding code + 128)."""
    KB = (K + 127) // 128
    TN = (N + 127) // 128
    a = (np.asarray(packed).view(np.uint8)[: TN * KB * 16384] ^ 0x80).view(np.int8).reshape(TN, KB, 128, 8, 16)
    r = np.arange(128)[:, None]
    phys = np.arange(8)[None, :] ^ (r & 7)              # logical chunk c lives at phys[r, c]
    logical = a[:, :, r, phys, :]                        # [TN][KB][128][8][16]
    return logical.transpose(0, 2, 1, 3, 4).reshape(TN * 128, KB * 128)[:N, :K]


def unpack_weights_w4(packed: np.ndarray, N: int, K: int) -> np.ndarray:
    """Row-major [N][K] 4-bit codes from the packed layout documented in
    include/quasar.h (128 x 128 blocks of 8 KB, row r at 64 r, 16-byte chunk
    c at position c ^ ((r >> 1) & 3), byte j = 4 w + b holding code(32 c +
    4 w + b) + 8 in its low nibble and code(32 c + 16 + 4 w + b) + 8 in its
    high nibble)."""
    KB = (K + 127) // 128
    TN = (N + 127) // 128
    a = np.asarray(packed).view(np.uint8)[: TN * KB * 8192].reshape(TN, KB, 128, 4, 16)
    r = np.arange(128)[:, None]
    phys = np.arange(4)[None, :] ^ ((r >> 1) & 3)
    ch = a[:, :, r, phys, :].astype(np.int16)          # [TN][KB][128][4 logical chunks][16 bytes]
    lo = (ch & 0xF) - 8                                 # K offsets 0..15 of the chunk
    hi = (ch >> 4) - 8                                  # K offsets 16..31
    codes = np.concatenate([lo, hi], axis=-1)           # [.., 4, 32]
    return codes.transpose(0, 2, 1, 3, 4).reshape(TN * 128, KB * 128)[:N, :K].astype(np.int8)
