"""DecodeStep (CUDA-graph step fed from pinned host memory) against the eager
calls and the oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_24_gb300.workloads import config_spec, make_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("direct_in", [True, False])
@pytest.mark.parametrize("direct_out", [False, True])
@pytest.mark.parametrize("fused", [True, False])
def test_decode_step_graph_matches_eager_and_oracle(pkv_lib, oracle_lib, fused, direct_out,
                                                    direct_in):
    pkv = pkv_lib
    spec = config_spec(4, num_seqs=24, num_q_heads=16, num_kv_heads=4, steps=3, seed=9)
    w = make_workload(spec, device="cuda")
    kc_e, vc_e = w.k_cache.clone(), w.v_cache.clone()
    kc_h, vc_h = w.k_cache.cpu(), w.v_cache.cpu()
    bt_h = w.block_tables.cpu().numpy()
    step = pkv.DecodeStep(w.k_cache, w.v_cache, spec.num_seqs, spec.num_q_heads, w.max_blocks,
                          spec.window, w.scale, num_buffers=spec.steps, fused=fused,
                          direct_out=direct_out, direct_in=direct_in)
    assert step.direct_out == direct_out
    assert step.direct_in == direct_in
    for s in range(spec.steps):
        h = step.host[s]
        h["q"].copy_(w.q_steps[s]); h["k"].copy_(w.k_steps[s]); h["v"].copy_(w.v_steps[s])
        h["positions"].copy_(w.pos_steps[s]); h["context_lens"].copy_(w.lens_steps[s])
        h["block_tables"].copy_(w.block_tables)
    for s in range(spec.steps):
        got = step.run(s).clone()
        # eager path on a copy of the pools
        slots = pkv.pkv_slot_mapping(w.block_tables, w.pos_steps[s].contiguous(), 16)
        pkv.pkv_append(w.k_steps[s], w.v_steps[s], slots, kc_e, vc_e)
        ref = pkv.pkv_decode(w.q_steps[s], kc_e, vc_e, w.block_tables,
                             w.lens_steps[s].contiguous(), spec.window, w.scale)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.cpu().view(torch.int16))
        # oracle
        o_slots = oracle.slot_mapping(bt_h, w.pos_steps[s].cpu().numpy(), 16)
        oracle.append(w.k_steps[s].cpu(), w.v_steps[s].cpu(), o_slots, kc_h, vc_h)
        exp = oracle.decode(w.q_steps[s].cpu(), kc_h, vc_h, bt_h, w.lens_steps[s].cpu().numpy(),
                            spec.window, w.scale)
        err = np.abs(got.double().numpy() - exp)
        assert (err <= 2e-3 + 0.5 * torch.finfo(torch.float16).eps * np.abs(exp)).all()
    assert torch.equal(w.k_cache.view(torch.int16), kc_e.view(torch.int16))
    assert torch.equal(w.v_cache.cpu().view(torch.int16), vc_h.view(torch.int16))
