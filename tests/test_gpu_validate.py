"""kvc_validate: the opt-in deep check of block tables, context lengths and slot mappings.

Expected verdicts are written out from the checks' definitions (include/kvc.h): integer work,
so every answer is exact, including the smallest offending index.
"""
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def _setup():
    import pagedattention_kvc_store_gb300 as kvc
    from workloads import config_case
    from workloads.device import to_device

    case = config_case(1)
    d = to_device(case)
    slots = torch.empty(case.num_tokens, dtype=torch.int32, device="cuda")
    kvc.kvc_slot_mapping(slots, d.block_table, d.context_lens, None, case.page_size)
    return kvc, case, d, slots


def test_valid_step_passes():
    kvc, case, d, slots = _setup()
    pool = kvc.pool_desc(d.k_pool)
    assert kvc.kvc_validate(pool, d.block_table, d.context_lens, slots) == (-1, "")
    assert kvc.kvc_validate(pool, slot_mapping=slots) == (-1, "")
    assert kvc.kvc_validate(pool, d.block_table, d.context_lens) == (-1, "")


def test_padding_slots_pass():
    kvc, case, d, slots = _setup()
    slots[1] = -1
    slots[3] = -7
    assert kvc.kvc_validate(kvc.pool_desc(d.k_pool), slot_mapping=slots)[0] == -1


def test_page_id_outside_pool():
    kvc, case, d, slots = _setup()
    bt = d.block_table.clone()
    # sequence 2 (ctx 33, three pages) gets a page id past the pool in its last page
    bt[2, 2] = case.num_pages
    bad, why = kvc.kvc_validate(kvc.pool_desc(d.k_pool), bt, d.context_lens)
    assert bad == 2 and "page id" in why
    # an entry past a sequence's last page is never read: not an error
    bt = d.block_table.clone()
    bt[0, bt.shape[1] - 1] = -5
    assert kvc.kvc_validate(kvc.pool_desc(d.k_pool), bt, d.context_lens)[0] == -1


def test_context_longer_than_row():
    kvc, case, d, slots = _setup()
    ctx = d.context_lens.clone()
    ctx[3] = d.block_table.shape[1] * case.page_size + 1
    ctx[1] = -1
    bad, why = kvc.kvc_validate(kvc.pool_desc(d.k_pool), d.block_table, ctx)
    assert bad == 1 and "context_lens" in why


def test_slot_past_pool():
    kvc, case, d, slots = _setup()
    s = slots.clone()
    s[2] = case.num_pages * case.page_size
    bad, why = kvc.kvc_validate(kvc.pool_desc(d.k_pool), slot_mapping=s)
    assert bad == 2 and "past the pool" in why


def test_duplicate_slots_report_smallest_token():
    kvc, case, d, slots = _setup()
    # 400 distinct slots (3 is coprime with the 512 slots of the pool), then three collisions
    s = torch.arange(400, dtype=torch.int32, device="cuda") * 3 % (case.num_pages * case.page_size)
    s[350] = s[117]
    s[380] = s[117]
    s[300] = s[10]
    bad, why = kvc.kvc_validate(kvc.pool_desc(d.k_pool), slot_mapping=s)
    assert bad == 10 and "two tokens" in why
