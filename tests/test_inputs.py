"""CPU: the seeded input generators keep the page-table contract the library leaves to its
caller (dcp_inputs.check_page_table): CSR offsets from 0 to the table length, non-decreasing,
and no destination page value twice; and the check itself rejects each violation."""
import pytest
import torch

import dcp_inputs as di


@pytest.mark.parametrize("lens,n_dcp", [([1024], 4), ([64 * 9 + 5, 130, 1], 8), ([100_000] * 3, 8), ([64], 1)])
def test_generated_tables_keep_the_contract(lens, n_dcp):
    gen = torch.Generator().manual_seed(7)
    slots = sum((n + 63) // 64 for n in lens)  # room for every page on any rank
    for make in (di.page_table, di.token_page_table):
        ptr, vp = make(lens, n_dcp, slots, gen)
        di.check_page_table(ptr, vp)
        assert int(ptr[-1]) == vp.numel()


def test_check_rejects_duplicates_and_bad_offsets():
    ptr = torch.tensor([0, 2, 4], dtype=torch.int64)
    di.check_page_table(ptr, torch.tensor([3, 1, 7, 2], dtype=torch.int32))
    with pytest.raises(ValueError, match="more than once"):
        di.check_page_table(ptr, torch.tensor([3, 1, 7, 3], dtype=torch.int32))
    with pytest.raises(ValueError, match="non-decreasing"):
        di.check_page_table(torch.tensor([0, 3, 2, 4], dtype=torch.int64), torch.arange(4, dtype=torch.int32))
    with pytest.raises(ValueError, match="from 0"):
        di.check_page_table(torch.tensor([0, 2, 3], dtype=torch.int64), torch.arange(4, dtype=torch.int32))
