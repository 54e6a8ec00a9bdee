"""pkv_stage_copy: kernel copies between device memory and pinned host memory
are byte-exact in every direction and for byte counts that are not a multiple
of 16; pageable host memory is refused without a launch."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [1, 15, 16, 17, 4096 + 5, 1638144, (3 << 20) + 9])
def test_stage_copy_round_trip(pkv_lib, nbytes):
    g = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes + 32,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.full((nbytes + 32,), 7, dtype=torch.uint8, device="cuda")
    back = torch.zeros(nbytes + 32, dtype=torch.uint8).pin_memory()
    dev2 = torch.zeros(nbytes + 32, dtype=torch.uint8, device="cuda")
    assert pkv_lib.pkv_stage_copy(dev, src, nbytes) == 0          # host -> device
    assert pkv_lib.pkv_stage_copy(dev2, dev, nbytes) == 0         # device -> device
    assert pkv_lib.pkv_stage_copy(back, dev2, nbytes) == 0        # device -> host
    torch.cuda.synchronize()
    assert torch.equal(dev[:nbytes].cpu(), src[:nbytes])
    assert (dev[nbytes:].cpu() == 7).all()                       # nothing past the end
    assert torch.equal(back[:nbytes], src[:nbytes])
    assert not back[nbytes:].any()


def test_stage_copy_refuses_pageable_memory(pkv_lib):
    pageable = torch.ones(4096, dtype=torch.uint8)
    dev = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert pkv_lib.pkv_stage_copy(dev, pageable) == pkv_lib.PKV_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert not dev.any()
