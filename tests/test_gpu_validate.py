"""pkv_validate_indices: the debug check of block tables, context lengths and
slots finds the first out-of-range index, in its stated order, and accepts
every index the kernels would use as given."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _case(device="cuda"):
    # 4 sequences, pages of 16 tokens, 6 table entries each, a pool of 40 blocks
    torch.manual_seed(0)
    nb, bs, mb = 40, 16, 6
    tables = torch.randperm(nb)[:24].reshape(4, mb).to(torch.int32)
    lens = torch.tensor([0, 17, 96, 50], dtype=torch.int32)
    # entries past a context's last page are never read: leave garbage there
    tables[0, :] = -7
    tables[1, 2:] = 10 ** 6
    tables[3, 4:] = -1
    slots = torch.tensor([-1, 3, 100, nb * bs - 1, -5], dtype=torch.int64)
    return [t.to(device) for t in (tables, lens, slots)] + [nb, bs]


@pytest.mark.parametrize("device", ["cuda", "cpu"])
def test_valid_indices_pass(pkv_lib, device):
    tables, lens, slots, nb, bs = _case(device)
    assert pkv_lib.pkv_validate_indices(tables, lens, nb, bs) is None
    assert pkv_lib.pkv_validate_indices(tables, lens, nb, bs, slot_mapping=slots) is None


def test_context_length_checks(pkv_lib):
    tables, lens, slots, nb, bs = _case()
    lens[2] = 6 * bs + 1                      # one past the table's reach
    tables[1, 0] = nb                         # also bad, but check 1 comes first
    assert pkv_lib.pkv_validate_indices(tables, lens, nb, bs) == \
        ("context_length", 2, 0, 6 * bs + 1)
    lens[2] = 6 * bs                          # exactly the reach: fine
    lens[0] = -1
    assert pkv_lib.pkv_validate_indices(tables, lens, nb, bs) == ("context_length", 0, 0, -1)


def test_block_table_checks(pkv_lib):
    tables, lens, slots, nb, bs = _case()
    tables[3, 3] = nb                         # used: 50 tokens need pages 0..3
    assert pkv_lib.pkv_validate_indices(tables, lens, nb, bs) == \
        ("block_table_entry", 3, 3, nb)
    tables[3, 3] = 0
    tables[2, 5] = -2                         # 96 tokens: page 5 is the last one used
    assert pkv_lib.pkv_validate_indices(tables, lens, nb, bs) == \
        ("block_table_entry", 2, 5, -2)


def test_slot_checks(pkv_lib):
    tables, lens, slots, nb, bs = _case()
    slots[2] = nb * bs                        # one past the pool
    assert pkv_lib.pkv_validate_indices(tables, lens, nb, bs, slot_mapping=slots) == \
        ("slot", 2, 0, nb * bs)
    slots = torch.tensor([7, 9, -1, 7, 9, -1, 9], dtype=torch.int64, device="cuda")
    # token 3 repeats token 0's slot and token 4 token 1's: the earliest repeat wins
    assert pkv_lib.pkv_validate_indices(tables, lens, nb, bs, slot_mapping=slots) == \
        ("duplicate_slot", 3, 0, 7)


def test_slots_from_the_library_are_valid(pkv_lib):
    """The slot mapping kernel's output passes the check (one token per sequence)."""
    from paged_kv_cache_24_gb300.workloads import CONFIGS, config_spec, make_workload
    w = make_workload(config_spec(CONFIGS["serving_fp16"]), device="cuda")
    slots = pkv_lib.pkv_slot_mapping(w.block_tables, w.pos_steps[0].contiguous(),
                                     w.spec.block_size)
    nb = w.k_cache.shape[0]
    assert pkv_lib.pkv_validate_indices(w.block_tables, w.lens_steps[0].contiguous(), nb,
                                        w.spec.block_size, slot_mapping=slots) is None


def test_flagged_indices_are_the_ones_decode_marks(pkv_lib):
    """Every sequence the check would flag comes back NaN from the decode, and
    only those: the check and the kernels agree on what a bad index is."""
    dt = torch.bfloat16
    q = torch.randn(4, 8, 128, device="cuda").to(dt)
    kc = torch.randn(6, 2, 16, 128, device="cuda").to(dt)
    vc = torch.randn_like(kc)
    bt = torch.tensor([[0, 1], [2, 99], [3, -5], [4, 5]], dtype=torch.int32, device="cuda")
    lens = torch.tensor([20, 20, 20, 33], dtype=torch.int32, device="cuda")
    out = pkv_lib.pkv_decode(q, kc, vc, bt, lens, 0, 0.1)
    torch.cuda.synchronize()
    flagged = []
    for b in range(4):
        one = pkv_lib.pkv_validate_indices(bt[b:b + 1].contiguous(), lens[b:b + 1].contiguous(),
                                           6, 16)
        flagged.append(one is not None)
        assert flagged[-1] == bool(torch.isnan(out[b].float()).any())
    assert flagged == [False, True, True, True]
    assert pkv_lib.pkv_validate_indices(bt, lens, 6, 16) == ("context_length", 3, 0, 33)
