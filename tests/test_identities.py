"""Integer identities the CUDA kernels rely on, checked exhaustively on the CPU.

The row GEMV turns a packed word of eight int4 codes (element 2j in the low nibble of byte j,
2j+1 in the high nibble; value u - 8, "colibri 开发演进实录" §2.1 int4-gs64) into two words of
signed bytes holding 16 (u - 8) with three bit operations, so that signed dp4a against the
int8 activation codes gives 16 times the group's dot(u - 8, q) with no zero-point term
("colibri 开发演进实录" §2.2 K1).  These tests pin that transform against the definition.
"""
import numpy as np

U32 = np.uint32


def _lo(w):
    return ((w << U32(4)) & U32(0xF0F0F0F0)) ^ U32(0x80808080)


def _hi(w):
    return (w & U32(0xF0F0F0F0)) ^ U32(0x80808080)


def _signed_bytes(w):
    return w.astype("<u4").view(np.int8).reshape(-1, 4).astype(np.int64)


def test_every_byte_value():
    # each byte of the result depends only on the same byte of the input
    b = np.arange(256, dtype=U32)
    for shift in range(4):
        w = b << U32(8 * shift)
        lo = _signed_bytes(_lo(w))[:, shift]
        hi = _signed_bytes(_hi(w))[:, shift]
        assert np.array_equal(lo, 16 * ((b & 15).astype(np.int64) - 8))
        assert np.array_equal(hi, 16 * ((b >> 4).astype(np.int64) - 8))


def test_random_words_and_chunk_dot():
    rng = np.random.default_rng(7)
    w = rng.integers(0, 2 ** 32, size=(4096, 4), dtype=np.uint64).astype(U32)   # 16-byte chunks
    q = rng.integers(-127, 128, size=(4096, 32), dtype=np.int64)                # int8 codes
    # element n of a chunk: word n // 8, nibble n % 8
    n = np.arange(32)
    u = (w[:, n // 8] >> U32(4) * (n % 8).astype(U32)) & U32(15)
    ref = ((u.astype(np.int64) - 8) * q).sum(axis=1)
    # the kernel's form: word k's low nibbles meet the even codes of run k, high nibbles the
    # odd ones (codes stored per run of 8 as [e0 e2 e4 e6 | e1 e3 e5 e7])
    lo = _signed_bytes(_lo(w).ravel()).reshape(4096, 4, 4)
    hi = _signed_bytes(_hi(w).ravel()).reshape(4096, 4, 4)
    runs = q.reshape(4096, 4, 8)
    got = (lo * runs[:, :, 0::2]).sum(axis=(1, 2)) + (hi * runs[:, :, 1::2]).sum(axis=(1, 2))
    assert np.array_equal(got, 16 * ref)
    # the partial sums stay far inside int32 (a chunk's |16 dot| <= 16 * 8 * 127 * 32)
    assert np.abs(got).max() <= 16 * 8 * 127 * 32 < 2 ** 31
