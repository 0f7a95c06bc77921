"""pkv_upload_metadata: a step's metadata image, pinned host -> device, through a kernel.

Bit-exact for every size (16-byte words and a 4-byte tail), refusals for memory the kernel cannot
read, and the property the engine relies on: the upload does not wait behind a bulk host-to-device
copy that another stream has in flight.
"""
import ctypes

import pytest

from paged_kv_cache_258_gb300 import pkv

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("words", [1, 3, 4, 5, 25, 1024, 6147, 300_001])
def test_upload_is_bit_exact(words):
    g = torch.Generator().manual_seed(words)
    src = torch.randint(-2**31, 2**31 - 1, (words,), dtype=torch.int32, generator=g).pin_memory()
    dst = torch.full((words + 8,), -7, dtype=torch.int32, device="cuda")
    pkv.pkv_upload_metadata(dst[:words], src)
    torch.cuda.synchronize()
    assert torch.equal(dst[:words].cpu(), src)
    assert bool((dst[words:] == -7).all())  # nothing written past the end


def test_upload_refuses_memory_the_kernel_cannot_read():
    L = pkv.lib()
    dst = torch.zeros(64, dtype=torch.int32, device="cuda")
    pageable = torch.arange(64, dtype=torch.int32)
    pinned = pageable.pin_memory()
    on_device = pageable.cuda()
    host_dst = torch.zeros(64, dtype=torch.int32).pin_memory()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(d, x, n=256):
        return L.pkv_upload_metadata(ctypes.c_void_p(d.data_ptr()), ctypes.c_void_p(x.data_ptr()), n, s)

    assert call(dst, pageable) == pkv.PKV_ERR_INVALID_ARG
    assert call(dst, on_device) == pkv.PKV_ERR_INVALID_ARG
    assert call(host_dst, pinned) == pkv.PKV_ERR_INVALID_ARG   # dst must be device memory
    assert call(dst[1:], pinned, 192) == pkv.PKV_ERR_INVALID_ARG  # 16-byte alignment of dst
    assert call(dst, pinned[1:], 192) == pkv.PKV_ERR_INVALID_ARG  # and of src
    assert call(dst, pinned) == pkv.PKV_OK
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), pageable)
    assert pkv.pkv_get_device_status() == 0


def test_upload_does_not_wait_behind_another_streams_bulk_copy():
    """A 2 GiB pinned host -> device copy on one stream (about 10 ms on the host link) is in
    flight when the metadata upload is issued on another: the upload is done while the bulk copy
    still runs."""
    n = (2 << 30) // 4
    big_h = torch.empty(n, dtype=torch.int32).pin_memory()
    big_d = torch.empty(n, dtype=torch.int32, device="cuda")
    meta_h = torch.arange(4096, dtype=torch.int32).pin_memory()
    meta_d = torch.zeros(4096, dtype=torch.int32, device="cuda")
    bulk, side = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(2):  # the first round warms up the kernel and the copy path
        torch.cuda.synchronize()
        with torch.cuda.stream(bulk):
            big_d.copy_(big_h, non_blocking=True)
            bulk_done = torch.cuda.Event()
            bulk_done.record(bulk)
        pkv.pkv_upload_metadata(meta_d, meta_h, stream=side)
        meta_done = torch.cuda.Event()
        meta_done.record(side)
        meta_done.synchronize()
        still_copying = not bulk_done.query()
        torch.cuda.synchronize()
    assert torch.equal(meta_d.cpu(), meta_h)
    assert still_copying
