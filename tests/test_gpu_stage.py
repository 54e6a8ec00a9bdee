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


def test_device_address(pkv_lib):
    dev = torch.zeros(64, dtype=torch.uint8, device="cuda")
    pinned = torch.zeros(64, dtype=torch.uint8).pin_memory()
    assert pkv_lib.pkv_device_address(dev) == dev.data_ptr()
    assert pkv_lib.pkv_device_address(pinned) is not None
    assert pkv_lib.pkv_device_address(torch.zeros(64, dtype=torch.uint8)) is None


@pytest.mark.parametrize("fused", [False, True])
def test_decode_into_pinned_host_output(pkv_lib, fused):
    """The decode kernels write a pinned host `out` directly (and, fused, read the
    queries and new rows from pinned memory): the same bits as device tensors,
    for single-split and split sequences alike."""
    from paged_kv_cache_24_gb300.workloads import config_spec, make_workload
    spec = config_spec(0, dtype=torch.bfloat16, num_seqs=6, num_q_heads=8, num_kv_heads=2,
                       head_dim=128, block_size=16, lens=[1, 30, 500, 2100, 4000, 0],
                       explicit_pool=None, lens_are_pre_append=False)
    outs = []
    for host in (False, True):
        w = make_workload(spec, device="cuda")
        lens = w.lens_steps[0].contiguous()
        out = (torch.full_like(w.q_steps[0], float("nan"), device="cpu").pin_memory() if host
               else torch.full_like(w.q_steps[0], float("nan")))
        if fused:
            # with host output, the queries and new rows come from pinned memory too
            q, kn, vn = ((t.cpu().pin_memory() for t in (w.q_steps[0], w.k_steps[0],
                                                          w.v_steps[0]))
                         if host else (w.q_steps[0], w.k_steps[0], w.v_steps[0]))
            pkv_lib.pkv_append_decode(q, kn, vn, w.k_cache, w.v_cache, w.block_tables, lens, 0,
                                      w.scale, out=out, tokens_per_split=512)
        else:
            slots = pkv_lib.pkv_slot_mapping(w.block_tables, w.pos_steps[0].contiguous(),
                                             spec.block_size)
            pkv_lib.pkv_append(w.k_steps[0], w.v_steps[0], slots, w.k_cache, w.v_cache)
            pkv_lib.pkv_decode(w.q_steps[0], w.k_cache, w.v_cache, w.block_tables, lens, 0,
                               w.scale, out=out, tokens_per_split=512)
        torch.cuda.synchronize()
        outs.append(out.cpu())
    assert not torch.isnan(outs[1].float()).any()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    with pytest.raises(ValueError):
        pkv_lib.pkv_decode(w.q_steps[0], w.k_cache, w.v_cache, w.block_tables, lens, 0, w.scale,
                           out=torch.empty(w.q_steps[0].shape, dtype=torch.bfloat16))
