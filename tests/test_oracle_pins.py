"""The fp64 oracle against its pins (CPU only), and the pins against planted
mistakes: each copy of the oracle compiled with one deliberate error must fail
at least one pin."""
import pytest

import oracle
import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(0)


def test_kv_len_below_rows_is_reported():
    from paged_split_kv_03_gb300.synth import make_workload
    wl = make_workload(batch=2, rows=[3, 1], kv_lens=[5, 9], num_qo_heads=2, num_kv_heads=1,
                       head_dim=8, page_size=4, seed=3)
    wl.kv_len[0] = 2  # fewer cached tokens than query rows
    out, lse, rc = oracle.attention_for(wl)
    assert rc == oracle.PDO_ERR_KVLEN


@pytest.mark.parametrize("mutation", sorted(pins.MUTATIONS), ids=lambda m: f"mut{m}")
def test_pins_catch_planted_mistake(mutation):
    oracle.build(mutation)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutation)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {mutation}: {pins.MUTATIONS[mutation]}"
