"""The launch table (grid, ring stages, L2 prefetch window, shared memory, consumer) worked out on
the host for a GB300 (152 SMs, 232,448 bytes of opt-in shared memory per block), pinned to values
derived by hand from the shared-memory layout:

    [1024 B misc][reduction buffer, unless it fits the dead tail of the bf16 activation area]
    [activations: bf16 2 M K (fused entries) or int8 M x stride (stride K, K + 16 for the MMA
    consumer)][ring, from a 128-byte boundary: stages x 4 blocks of 8448 B (int4) / 12544 B (int6)]

with the reduction buffer 4 x M x 128 x 4 bytes, three stages (two rows, and five or more: four)
within the device limit, else the largest ring that fits; and against what ncu reported for the
same launches on a GB300 (gate_up at M = 1: 112,640 B)."""
import pytest

import weight_only_quantised_gb300 as woq

GB300 = dict(sms=152, smem_max=232448)


@pytest.fixture(autouse=True)
def table_defaults():
    woq.woq_tune_override(0, 0, -1)
    woq.woq_tune_path(0)
    yield
    woq.woq_tune_override(0, 0, -1)
    woq.woq_tune_path(0)


@pytest.mark.parametrize("bits,M,N,K,entry,want", [
    # qkv 5120 -> 7168, one row: ring at 1024 + 10240 = 11264; 3 x 33792 + 11264 = 112640
    # (4 stages: 146432 > 115712); 56 x 40 = 2240 blocks < 5000: one prefetch stage
    (4, 1, 7168, 5120, 1, dict(ctas=152, stages=3, prefetch_stages=1, smem_bytes=112640, consumer=0)),
    # gate_up 5120 -> 34816: same layout; 10880 blocks >= 5000 at one row: two prefetch stages
    (4, 1, 34816, 5120, 1, dict(ctas=152, stages=3, prefetch_stages=2, smem_bytes=112640, consumer=0)),
    # down 17408 -> 5120: ring at 1024 + 34816 = 35840; 3 x 33792 + 35840 = 137216
    (4, 1, 5120, 17408, 1, dict(ctas=152, stages=3, prefetch_stages=2, smem_bytes=137216, consumer=0)),
    # LM head at four rows: ring at 1024 + 40960 = 41984; 3 stages: 143360
    (4, 4, 152064, 5120, 1, dict(ctas=152, stages=3, prefetch_stages=1, smem_bytes=143360, consumer=0)),
    # two rows take four stages where they fit: 21504 + 4 x 33792 = 156672
    (4, 2, 7168, 5120, 1, dict(ctas=152, stages=4, prefetch_stages=1, smem_bytes=156672, consumer=0)),
    # five rows: MMA consumer, four stages: 52224 + 4 x 33792 = 187392
    (4, 5, 7168, 5120, 1, dict(ctas=152, stages=4, prefetch_stages=1, smem_bytes=187392, consumer=1)),
    # int8 entry: reduction buffer before 5120 B of q: ring at 3072 + 5120 = 8192; 3 stages: 109568
    (4, 1, 7168, 5120, 0, dict(ctas=152, stages=3, prefetch_stages=1, smem_bytes=109568, consumer=0)),
    # int6: stages of 50176 B: 11264 + 3 x 50176 = 161792
    (6, 1, 7168, 5120, 1, dict(ctas=152, stages=3, prefetch_stages=1, smem_bytes=161792, consumer=0)),

    # one block in all: one CTA; reduction buffer outside the 256-byte activation area:
    # ring at 3072 + 256 -> 3328; 3 stages: 104704
    (4, 1, 128, 128, 1, dict(ctas=1, stages=3, prefetch_stages=1, smem_bytes=104704, consumer=0)),
    # 5 blocks: two CTAs (at least one four-block stage each); int8 entry, ring at 3072 + 128 -> 3200,
    # 3 stages: 104576
    (4, 1, 640, 128, 0, dict(ctas=2, stages=3, prefetch_stages=1, smem_bytes=104576, consumer=0)),
])
def test_plan_for_a_gb300(bits, M, N, K, entry, want):
    assert woq.woq_plan_launch(bits, M, N, K, entry, **GB300) == want


def test_ring_budget_follows_the_device_limit():
    # with 120,000 bytes a five-row launch fits two stages: 52224 + 2 x 33792 = 119808
    assert woq.woq_plan_launch(4, 5, 7168, 5120, 1, sms=152, smem_max=120000)["stages"] == 2
    # and nothing fits 60,000 bytes for qkv at one row (11264 + 2 x 33792 = 78848)
    with pytest.raises(woq.WoqError) as e:
        woq.woq_plan_launch(4, 1, 7168, 5120, 1, sms=152, smem_max=60000)
    assert e.value.status == woq.WOQ_ERR_SHAPE
    # the grid follows the SM count
    assert woq.woq_plan_launch(4, 1, 7168, 5120, 1, sms=76, smem_max=232448)["ctas"] == 76


def test_overrides_and_the_swiglu_grid():
    woq.woq_tune_override(2, 0, -1)
    # two CTAs per SM where the blocks allow it (2240 blocks: 560 four-block stages)
    assert woq.woq_plan_launch(4, 1, 7168, 5120, 1, **GB300)["ctas"] == 304
    # the SwiGLU entry's grid-wide step needs every CTA resident: one per SM
    assert woq.woq_plan_launch(4, 1, 7168, 5120, 2, **GB300)["ctas"] == 152
    woq.woq_tune_override(1, 6, 0)
    p = woq.woq_plan_launch(4, 1, 7168, 5120, 1, **GB300)
    assert p["stages"] == 6 and p["prefetch_stages"] == 0 and p["smem_bytes"] == 11264 + 6 * 33792
    woq.woq_tune_override(0, 0, -1)
    woq.woq_tune_path(2)
    assert woq.woq_plan_launch(4, 1, 7168, 5120, 1, **GB300)["consumer"] == 1
    assert woq.woq_plan_launch(6, 1, 7168, 5120, 1, **GB300)["consumer"] == 0  # int6: dp4a only


@pytest.mark.parametrize("bits,M,N,K,entry", [
    (4, 1, 7168, 100, 1),   # K not a multiple of 128
    (4, 0, 7168, 5120, 1),  # no rows
    (4, 9, 7168, 5120, 1),  # more rows than int4 takes
    (6, 5, 7168, 5120, 1),  # more rows than int6 takes
    (4, 8, 7168, 17408, 1),  # M K above the activation tile
    (4, 1, 0, 5120, 1),     # no outputs
    (4, 1, 7168, 5120, 3),  # no such entry
    (5, 1, 7168, 5120, 1),  # no such width
])
def test_plan_rejects_bad_shapes(bits, M, N, K, entry):
    with pytest.raises(woq.WoqError) as e:
        woq.woq_plan_launch(bits, M, N, K, entry, **GB300)
    assert e.value.status == woq.WOQ_ERR_SHAPE


def test_plan_needs_out_and_a_device():
    assert woq.lib.woq_plan_launch(4, 1, 128, 128, 1, 152, 232448, None) == woq.WOQ_ERR_NULL
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU")
    with pytest.raises(woq.WoqError) as e:
        woq.woq_plan_launch(4, 1, 128, 128, 1)  # the current device's values: none here
    assert e.value.status == woq.WOQ_ERR_CUDA
