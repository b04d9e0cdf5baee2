"""The CPU oracle against the pages' values, closed forms, invariants and the
per-token brute force (no GPU)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("name", P.ALL)
def test_oracle_pin(oracle_lib, name):
    getattr(P, name)(oracle_lib)


def test_config0_payload(oracle_lib):
    """The tiny workload moves 884,736 MLA + 1,262,592 KDA bytes."""
    case = P.tiny_case(oracle_lib, 0)
    L, C = case["L"], case["C"]
    assert C == 128
    n_chunks = sum(int(x) // C for x in case["lengths"])
    assert n_chunks == 6
    kda_og = L.object_group[0]
    mla_og = L.object_group[3]
    assert n_chunks * L.object_bytes(C, mla_og) == 884_736
    assert n_chunks * L.object_bytes(C, kda_og) == 1_262_592
    assert case["arena_bytes"] == 2_147_328
