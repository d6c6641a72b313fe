"""The host-side grouping of a pass's products into phase launches
(mlq_q4k_phase / mlq_nbits_phase: products that read one input in one
launch), on the CPU.  Data flow: page "Legacy-ISA ML Inference Runtime --
Design Spec", Sec. 6 "Forward pass" (a product's output is a later
product's input)."""
import pytest

from block_quantized_decode_gb300 import inputs as I


@pytest.fixture(scope="module")
def group():
    torch = pytest.importorskip("torch")  # noqa: F841 (runner imports torch)
    from block_quantized_decode_gb300.runner import phase_groups
    return phase_groups


def check(groups, mats, max_products=4):
    names = [n for _, ns, _ in groups for n in ns]
    assert names == [m[0] for m in mats], "every product once, in pass order"
    by = {m[0]: m for m in mats}
    seen = set()
    for inp, ns, k in groups:
        assert 1 <= len(ns) <= max_products
        for n in ns:
            assert by[n][3] == inp and by[n][2] == k, "one input, one width per group"
        assert inp == "x" or inp in seen, "a group's input is produced by an earlier group"
        seen.update(ns)


@pytest.mark.parametrize("wl", [I.tinyllama_layer_q4k(), I.qwen_layer_int4_blk128(), I.qwen_layer_int8_sq8()],
                         ids=lambda w: w.name)
def test_layer_passes_group_into_four_phases(group, wl):
    g = group(wl.mats)
    check(g, wl.mats)
    assert [len(ns) for _, ns, _ in g] == [3, 1, 2, 1]   # q|k|v, o, gate|up, down


def test_grouping_limits_and_chains(group):
    mats = [(f"p{i}", 64, 512, "x") for i in range(6)]          # six products of one input
    g = group(mats)
    check(g, mats)
    assert [len(ns) for _, ns, _ in g] == [4, 2]
    chain = [("a", 512, 256, "x"), ("b", 256, 512, "a"), ("c", 64, 256, "b"), ("d", 32, 256, "b"),
             ("e", 16, 256, "x")]
    g = group(chain)
    check(g, chain)
    assert [ns for _, ns, _ in g] == [["a"], ["b"], ["c", "d"], ["e"]]
    assert group([]) == []
    g = group(mats, max_products=1)
    check(g, mats, 1)
    assert len(g) == 6
