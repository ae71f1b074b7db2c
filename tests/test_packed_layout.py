"""Host check of the packed weight layout helper used by the GPU tests: a
direct transcription of the layout rule in include/quasar.h (one byte at a
time) must round-trip through tests.gpu_util.unpack_weights."""
import numpy as np
import pytest

from tests.gpu_util import unpack_weights


def pack_by_rule(wq):
    N, K = wq.shape
    KB, TN = (K + 127) // 128, (N + 127) // 128
    out = np.full(TN * KB * 16384, -128, np.int8)   # code 0 is stored as byte 0x80
    for n in range(N):
        tn, r = divmod(n, 128)
        for k in range(K):
            kb, kk = divmod(k, 128)
            c, e = divmod(kk, 16)
            out[(tn * KB + kb) * 16384 + r * 128 + ((c ^ (r % 8)) * 16) + e] = np.int8(int(wq[n, k]) ^ -128)
    return out


@pytest.mark.parametrize("N,K", [(8, 16), (136, 144), (130, 272)])
def test_unpack_inverts_documented_layout(N, K):
    rng = np.random.default_rng(N * 1000 + K)
    wq = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    packed = pack_by_rule(wq)
    assert np.array_equal(unpack_weights(packed, N, K), wq)
