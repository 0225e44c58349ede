"""The HBM bandwidth probes (read-only XOR fold and copy) through the C ABI."""
import numpy as np
import pytest
import torch

import split_kv_paged_gqa_gb300 as fd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("nbytes", [16, 4096 + 48, (3 << 20) + 16 * 7, 256 << 20])
def test_read_probe_folds_every_word(nbytes):
    g = torch.Generator(device="cuda").manual_seed(nbytes)
    src = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda").random_(generator=g)
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    fd.fd_probe_hbm_read(src, sink)
    torch.cuda.synchronize()
    want = np.bitwise_xor.reduce(src.cpu().numpy().view(np.uint32).reshape(-1, 4), axis=0)
    assert np.array_equal(sink.cpu().numpy().view(np.uint32), want)
    fd.fd_probe_hbm_read(src, sink)          # sink ^= the same fold -> 0
    torch.cuda.synchronize()
    assert not sink.any().item()


@pytest.mark.parametrize("nbytes", [16, 4096 + 48, (3 << 20) + 16 * 7, 256 << 20])
def test_copy_probe_copies_every_byte(nbytes):
    g = torch.Generator(device="cuda").manual_seed(nbytes + 1)
    src = torch.empty(nbytes, dtype=torch.uint8, device="cuda").random_(generator=g)
    dst = torch.zeros_like(src)
    fd.fd_probe_hbm_copy(src, dst)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)


def test_probes_reject_bad_sizes_and_overlap():
    src = torch.zeros(64, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(fd.FdError) as e:
        fd.fd_probe_hbm_read(src[:40], sink)      # not a multiple of 16 bytes
    assert e.value.status == fd.FD_ERR_UNSUPPORTED
    lib = fd.load_library()
    s = lib.fd_probe_hbm_copy(src.data_ptr(), src.data_ptr() + 16, 32, None)
    assert s == fd.FD_ERR_INVALID_ARG                 # overlapping ranges
    s = lib.fd_probe_hbm_copy(src.data_ptr() + 8, src.data_ptr() + 48, 16, None)
    assert s == fd.FD_ERR_UNSUPPORTED                 # misaligned source
