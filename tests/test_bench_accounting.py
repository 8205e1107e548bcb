"""The benchmark's algorithmic byte count (the roofline numerator) against figures worked
out by hand from the configuration: what each step must move, per unit and per step —
summary rows of the scored candidates, the selected blocks' K and V, page-table
entries, indices, q and the outputs."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from workloads import make_workload  # noqa: E402


def _llama_32k_selection():
    # Streaming KV heads 0-3: sink 128 tokens = blocks 0-3, local 2048 tokens = blocks
    # 960-1023 (68 blocks). Retrieval heads 4-7: blocks 0 and 1023 forced, k = 51.
    streaming = list(range(4)) + list(range(960, 1024))
    retrieval = [0] + list(range(100, 151)) + [1023]
    return [streaming] * 4 + [retrieval] * 4


def test_llama_32k_layer_bytes():
    wl = make_workload(2)
    sel = _llama_32k_selection()
    assert [len(x) for x in sel] == [68] * 4 + [53] * 4
    got = bench.algorithmic_bytes(wl, sel, sel)
    # scores: 4 retrieval units x 1022 candidates x 4 sub-blocks x 128 dims x 4 B,
    # + q (4 heads x 128 x 2 B) + one fp32 score per candidate
    assert got["score"] == 4 * (1022 * 4 * 128 * 4 + 4 * 128 * 2 + 1022 * 4) == 8_392_672
    # attention: 484 full blocks of 32 tokens, K and V of 128 bf16 each; q; 2 pages per
    # block; one index per block; out (4 x 128 fp32) and lse (4 fp32) per unit
    kv = 484 * 32 * 128 * 2 * 2
    assert got["attn"] == kv + 8 * 4 * 128 * 2 + 968 * 4 + 484 * 4 + 8 * 4 * 129 * 4 == 7_960_368
    # selection: each retrieval unit reads its candidates' scores and writes its list
    assert got["select"] == 4 * (1022 * 4 + 53 * 4) == 17_200
    # set-difference: both lists read and the outputs written
    assert got["setdiff"] == (484 + 484) * 4 * 2 == 7_744
    # sub-block update: the 8 tokens of the appended token's sub-block, one fp32 row out
    assert got["summary_update"] == 8 * (8 * 128 * 2 + 128 * 4) == 20_480
    assert got["layer_step"] == 16_398_464


def test_ragged_tail_block_bytes():
    # T = 4133 = 129 * 32 + 5: the tail block holds 5 tokens in one page.
    wl = make_workload(2, T=4133)
    sel = [[] for _ in range(wl.U)]
    sel[5] = [0, 7, 129]
    got = bench.algorithmic_bytes(wl, sel, [[] for _ in range(wl.U)])
    constants = wl.U * (4 * 128 * 2 + 4 * 129 * 4)           # q, out and lse of every unit
    tokens, pages = 32 + 32 + 5, 2 + 2 + 1
    assert got["attn"] == constants + tokens * 128 * 2 * 2 + pages * 4 + 3 * 4
    # the appended token (position 4132) is the 5th of its sub-block of 8
    assert got["summary_update"] == wl.U * (5 * 128 * 2 + 128 * 4)
