"""The streaming-read probe (pkv_hbm_read_probe) reads every byte exactly once: its XOR fold of
the buffer's 32-bit words equals numpy's, bit for bit, at sizes from one 16-byte word to buffers
with ragged ends against the grid's stride."""
import ctypes

import numpy as np
import pytest

from paged_kv_cache_258_gb300 import pkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_words", [4, 8, 1000, 4 * 150_001, 4 * (1 << 20) + 4 * 37])
def test_fold_matches_numpy(n_words):
    import torch
    rng = np.random.default_rng(n_words)
    host = rng.integers(0, 2 ** 32, size=n_words, dtype=np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).cuda()
    fold = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_hbm_read_probe(buf, fold)
    got = int(fold.cpu().numpy().view(np.uint32)[0])
    assert got == int(np.bitwise_xor.reduce(host))


def test_probe_rejects_bad_sizes_and_alignment():
    import torch
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    fold = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = pkv.lib()
    vp = ctypes.c_void_p
    assert L.pkv_hbm_read_probe(vp(buf.data_ptr()), 20, vp(fold.data_ptr()), vp(0)) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_hbm_read_probe(vp(buf.data_ptr() + 4), 32, vp(fold.data_ptr()), vp(0)) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_hbm_read_probe(vp(buf.data_ptr()), 0, vp(fold.data_ptr()), vp(0)) == pkv.PKV_OK
    torch.cuda.synchronize()
    assert int(fold.item()) == 0
