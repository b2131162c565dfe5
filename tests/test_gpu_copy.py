"""scan_copy, the bandwidth-reference copies: both modes copy every byte,
write nothing past the destination, and handle sizes that leave a partial
last trip (vector copy) or a partial last tile (tensor copies)."""

import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
PAD = 4096  # bytes of sentinel on each side


@pytest.mark.parametrize("mode", ["vec", "tma"])
@pytest.mark.parametrize("nbytes", [128, 4096, 32768, 32768 * 3 + 128 * 7, 1 << 24,
                                    (1 << 26) + 128 * 5])
def test_copy_every_byte_and_nothing_more(lib, mode, nbytes):
    m = lib.SCAN_COPY_VEC if mode == "vec" else lib.SCAN_COPY_TMA
    g = torch.Generator(device="cpu").manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).to(DEV)
    buf = torch.full((nbytes + 2 * PAD,), 0xA5, dtype=torch.uint8, device=DEV)
    dst = buf[PAD:PAD + nbytes]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.scan_copy(src, dst, m, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == lib.SCAN_OK
    assert torch.equal(dst, src)
    assert bool((buf[:PAD] == 0xA5).all()) and bool((buf[PAD + nbytes:] == 0xA5).all())


def test_copy_rejects_sizes_its_mode_cannot_move(lib):
    src = torch.zeros(100, dtype=torch.uint8, device=DEV)
    dst = torch.zeros(100, dtype=torch.uint8, device=DEV)
    with pytest.raises(lib.ScanError) as e:
        lib.scan_copy(src, dst, lib.SCAN_COPY_TMA)
    assert e.value.status == lib.SCAN_ERR_INVALID_ARG
    with pytest.raises(lib.ScanError) as e:
        lib.scan_copy(src[:90], dst[:90], lib.SCAN_COPY_VEC)
    assert e.value.status == lib.SCAN_ERR_INVALID_ARG
